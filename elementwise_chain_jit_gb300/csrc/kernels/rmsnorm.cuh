// rmsnorm.cuh -- residual add + RMSNorm + cast, one CTA per row.
//
// The generated source defines before including this file:
//   DT      dtype code of x, residual, weight and both outputs
//   HIDDEN  row length
//   BLOCK   threads per CTA
//   VEC     elements per thread-vector in the vector kernel (VEC*bytes is
//           16 or 32), HIDDEN % VEC == 0
//   R       vectors per thread: ceil(HIDDEN / VEC / BLOCK)
//   FUSE_RMS_VEC  1 when a vector width fits the row (else only the
//           scalar kernel exists)
//
// Per row ("TeleTron", sections 3.3 and 4.2): h = x + residual in fp32,
// residual_out = dt(h), ms = sum(h^2)/HIDDEN accumulated in fp32 (per thread,
// then a warp shuffle tree, then across warps through shared memory),
// out = dt(h * (1/sqrt(ms + eps)) * w).
#pragma once
#include "fuse/common.cuh"

constexpr int NWARPS = BLOCK / 32;
constexpr int NVR = HIDDEN / VEC;                 // vectors per row
constexpr int NWV = VEC * Dt<DT>::bytes / 4;      // words per vector

__device__ __forceinline__ float block_sum(float v, float* part) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < NWARPS; ++i) t += part[i];
  return t;
}

#if FUSE_RMS_VEC
// vector kernel: h stays in registers between the reduction and the output
extern "C" __global__ void __launch_bounds__(BLOCK)
rmsnorm_vec(const void* x, const void* res, const void* w, void* out, void* res_out,
            long long rows, float eps) {
  pdl_enter();
  __shared__ float part[NWARPS];
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const u32* xr = static_cast<const u32*>(x) + row * (HIDDEN * Dt<DT>::bytes / 4);
    const u32* rr = static_cast<const u32*>(res) + row * (HIDDEN * Dt<DT>::bytes / 4);
    u32* orow = static_cast<u32*>(out) + row * (HIDDEN * Dt<DT>::bytes / 4);
    u32* rorow = static_cast<u32*>(res_out) + row * (HIDDEN * Dt<DT>::bytes / 4);
    u32 wx[R][NWV], wr[R][NWV], ww[R][NWV];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      if (NVR % BLOCK == 0 || v < NVR) {
        load_words(xr + v * NWV, wx[i]);
        load_words(rr + v * NWV, wr[i]);
        load_words_cached(static_cast<const u32*>(w) + v * NWV, ww[i]);
      }
    }
    float h[R][VEC];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      if (NVR % BLOCK == 0 || v < NVR) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          h[i][e] = get_elem<DT>(wx[i], e) + get_elem<DT>(wr[i], e);
          ss += h[i][e] * h[i][e];
        }
        u32 o[NWV];
        pack_vec<DT>(h[i], o);
        store_words(rorow + v * NWV, o);
      }
    }
    const float rstd = 1.0f / sqrtf(block_sum(ss, part) / HIDDEN + eps);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      if (NVR % BLOCK == 0 || v < NVR) {
        float y[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) y[e] = h[i][e] * rstd * get_elem<DT>(ww[i], e);
        u32 o[NWV];
        pack_vec<DT>(y, o);
        store_words(orow + v * NWV, o);
      }
    }
    __syncthreads();  // part[] is reused by the next row
  }
}
#endif

// scalar kernel (pointers not aligned to the vector width): two passes over
// the row, element by element
extern "C" __global__ void __launch_bounds__(BLOCK)
rmsnorm_scalar(const void* x, const void* res, const void* w, void* out, void* res_out,
               long long rows, float eps) {
  pdl_enter();
  __shared__ float part[NWARPS];
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const long long base = row * HIDDEN;
    float ss = 0.f;
    for (int i = threadIdx.x; i < HIDDEN; i += BLOCK) {
      const float hv = load_elem<DT>(x, base + i) + load_elem<DT>(res, base + i);
      ss += hv * hv;
    }
    const float rstd = 1.0f / sqrtf(block_sum(ss, part) / HIDDEN + eps);
    for (int i = threadIdx.x; i < HIDDEN; i += BLOCK) {
      const float hv = load_elem<DT>(x, base + i) + load_elem<DT>(res, base + i);
      store_elem<DT>(res_out, base + i, hv);
      store_elem<DT>(out, base + i, hv * rstd * load_elem<DT>(w, i));
    }
    __syncthreads();
  }
}
