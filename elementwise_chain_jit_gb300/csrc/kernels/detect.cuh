// detect.cuh -- detection-head decode: sigmoid, box affine, channel->last
// transpose and the concat of all scales, one CTA per (scale, anchor, tile of
// TC cells).
//
// The generated source defines before including this file:
//   DT (input dtype), NA, NO, TC (cells per tile, a multiple of 8), BLOCK,
// and after it the dispatch kernels that call tile_work<> with each scale's
// baked H, W, stride, anchor and row offset.
//
// A tile reads NO channel planes x TC cells (contiguous runs of 8 cells per
// thread, coalesced along the cells), decodes each value in fp32 registers
// and writes it into shared memory laid out [cell][k] -- exactly the layout
// of the output rows -- so that the write-out is one contiguous run of
// TC*NO floats per CTA with 16-byte stores.
#pragma once
#include "fuse/common.cuh"

struct Feats {
  const void* p[8];
};

template <int W>
__device__ __forceinline__ float decode(int k, int cell, float v, float stride, float aw, float ah) {
  const float p = sigmoid(v);  // rcp_ge1 of 1 + exp(-v): within an ulp of the division
  if (k == 0) return (2.0f * p - 0.5f + static_cast<float>(cell % W)) * stride;
  if (k == 1) return (2.0f * p - 0.5f + static_cast<float>(cell / W)) * stride;
  if (k == 2) { const float t = 2.0f * p; return t * t * aw; }
  if (k == 3) { const float t = 2.0f * p; return t * t * ah; }
  return p;
}

// VEC: 16-byte input loads and output stores (pointers checked by the host)
template <bool VEC, int H, int W>
__device__ __forceinline__ void tile_work(const void* feat, float* out, int a, int c0, float stride,
                                          float aw, float ah, long long row_first, float* tile) {
  constexpr int HW = H * W;
  constexpr int G = TC / 8;
  const int ncell = HW - c0 < TC ? HW - c0 : TC;
  if constexpr (VEC && HW % 8 == 0) {
    // every (channel, 8-cell group) item of this thread: all loads first,
    // then the decodes, so the loads of a tile are in flight together
    constexpr int NWI = 8 * Dt<DT>::bytes / 4;
    constexpr int PER = (NO * G + BLOCK - 1) / BLOCK;
    u32 w[PER][NWI];
#pragma unroll
    for (int n = 0; n < PER; ++n) {
      const int it = threadIdx.x + n * BLOCK;
      const int k = it / G, g = it % G;
      if (it < NO * G && c0 + g * 8 < HW) {
        const long long off = static_cast<long long>(a * NO + k) * HW + c0 + g * 8;
        load_words(static_cast<const u32*>(feat) + off * Dt<DT>::bytes / 4, w[n]);
      }
    }
#pragma unroll
    for (int n = 0; n < PER; ++n) {
      const int it = threadIdx.x + n * BLOCK;
      const int k = it / G, g = it % G;
      const int cell = c0 + g * 8;
      if (it < NO * G && cell < HW) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          tile[(g * 8 + e) * NO + k] = decode<W>(k, cell + e, get_elem<DT>(w[n], e), stride, aw, ah);
      }
    }
  } else {
    for (int it = threadIdx.x; it < NO * TC; it += BLOCK) {
      const int k = it / TC, cl = it % TC;
      if (cl < ncell) {
        const long long off = static_cast<long long>(a * NO + k) * HW + c0 + cl;
        tile[cl * NO + k] = decode<W>(k, c0 + cl, load_elem<DT>(feat, off), stride, aw, ah);
      }
    }
  }
  __syncthreads();
  // rows [row_first, row_first + ncell) of the output are contiguous
  float* dst = out + row_first * NO;
  const int total = ncell * NO;
  if constexpr (VEC) {
    const int head = static_cast<int>((4 - (row_first * NO) % 4) % 4) < total
                         ? static_cast<int>((4 - (row_first * NO) % 4) % 4)
                         : total;
    const int body = (total - head) / 4;
    if (threadIdx.x < head) dst[threadIdx.x] = tile[threadIdx.x];
    if (head == 0) {
      // the tile is 16-byte aligned: one 16-byte shared load a store
      const float4* t4 = reinterpret_cast<const float4*>(tile);
      for (int i = threadIdx.x; i < body; i += BLOCK) {
        const float4 v = t4[i];
        const u32 w[4] = {__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                          __float_as_uint(v.w)};
        st_words16(reinterpret_cast<u32*>(dst) + 4 * i, w);
      }
    } else {
      for (int i = threadIdx.x; i < body; i += BLOCK) {
        u32 w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = __float_as_uint(tile[head + 4 * i + e]);
        st_words16(reinterpret_cast<u32*>(dst + head) + 4 * i, w);
      }
    }
    for (int i = head + 4 * body + threadIdx.x; i < total; i += BLOCK) dst[i] = tile[i];
  } else {
    for (int i = threadIdx.x; i < total; i += BLOCK) dst[i] = tile[i];
  }
}
