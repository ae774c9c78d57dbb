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
//   ROW_PREFETCH  1: the vector kernel asks L2 for its first row before the
//           launch-order wait
//
// Per row ("TeleTron", sections 3.3 and 4.2): h = x + residual in fp32,
// residual_out = dt(h), ms = sum(h^2)/HIDDEN accumulated in fp32,
// out = dt(h * (1/sqrt(ms + eps)) * w).  The sum of squares is a balanced
// tree (per thread, then over lanes, then over warps; common.cuh), so each
// square is rounded at most ceil(log2 HIDDEN) + 3 times on its way into ms.
#pragma once
#include "fuse/common.cuh"

constexpr int NWARPS = BLOCK / 32;
constexpr int NVR = HIDDEN / VEC;                 // vectors per row
constexpr int NWV = VEC * Dt<DT>::bytes / 4;      // words per vector

#if FUSE_RMS_VEC
// vector kernel: h stays in registers between the reduction and the output
extern "C" __global__ void __launch_bounds__(BLOCK)
rmsnorm_vec(const void* x, const void* res, const void* w, void* out, void* res_out,
            long long rows, float eps) {
  // ask L2 for the CTA's first row before waiting for the previous kernel
  // (programmatic dependent launch; L2 is coherent, the loads come after)
  if constexpr (ROW_PREFETCH && (VEC * Dt<DT>::bytes) % 16 == 0) {
    if (threadIdx.x == 0 && blockIdx.x < rows) {
      constexpr unsigned RB = HIDDEN * Dt<DT>::bytes;
      prefetch_l2(static_cast<const char*>(x) + blockIdx.x * (long long)RB, RB);
      prefetch_l2(static_cast<const char*>(res) + blockIdx.x * (long long)RB, RB);
    }
  }
  pdl_enter();
  __shared__ float part[2][NWARPS];
  for (long long row = blockIdx.x, it = 0; row < rows; row += gridDim.x, ++it) {
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
    float ssv[R];  // per vector: its squares summed as a tree
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      ssv[i] = 0.f;
      if (NVR % BLOCK == 0 || v < NVR) {
        float sq[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          h[i][e] = get_elem<DT>(wx[i], e) + get_elem<DT>(wr[i], e);
          sq[e] = h[i][e] * h[i][e];
        }
        ssv[i] = tree_sum(sq);
        u32 o[NWV];
        pack_vec<DT>(h[i], o);
        store_words(rorow + v * NWV, o);
      }
    }
    // part[] alternates between rows, so one barrier per row suffices
    const float ss = cta_sum<NWARPS>(tree_sum(ssv), part[it & 1]);
    const float rstd = 1.0f / sqrtf(ss / HIDDEN + eps);
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
  }
}
#endif

// scalar kernel (pointers not aligned to the vector width): two passes over
// the row, element by element; each thread's squares are summed by a cascade
// (a balanced tree built as they arrive)
constexpr int SITER = (HIDDEN + BLOCK - 1) / BLOCK;  // elements per thread

extern "C" __global__ void __launch_bounds__(BLOCK)
rmsnorm_scalar(const void* x, const void* res, const void* w, void* out, void* res_out,
               long long rows, float eps) {
  pdl_enter();
  __shared__ float part[2][NWARPS];
  for (long long row = blockIdx.x, it = 0; row < rows; row += gridDim.x, ++it) {
    const long long base = row * HIDDEN;
    Cascade<SITER> acc;
#pragma unroll
    for (int k = 0; k < SITER; ++k) {
      const int i = threadIdx.x + k * BLOCK;
      float sq = 0.f;
      if (HIDDEN % BLOCK == 0 || i < HIDDEN) {
        const float hv = load_elem<DT>(x, base + i) + load_elem<DT>(res, base + i);
        sq = hv * hv;
      }
      acc.add(k, sq);
    }
    const float rstd = 1.0f / sqrtf(cta_sum<NWARPS>(acc.total(), part[it & 1]) / HIDDEN + eps);
    for (int i = threadIdx.x; i < HIDDEN; i += BLOCK) {
      const float hv = load_elem<DT>(x, base + i) + load_elem<DT>(res, base + i);
      store_elem<DT>(res_out, base + i, hv);
      store_elem<DT>(out, base + i, hv * rstd * load_elem<DT>(w, i));
    }
  }
}
