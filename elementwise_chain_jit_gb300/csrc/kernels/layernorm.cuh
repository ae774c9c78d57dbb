// layernorm.cuh -- residual add + LayerNorm + cast, one CTA per row.
//
// The generated source defines before including this file:
//   DT, HIDDEN, BLOCK, VEC, R   as for rmsnorm.cuh
//   HAS_RES, HAS_GAMMA, HAS_BETA  0/1: residual add, scale, shift present
//   FUSE_LN_VEC  1 when a vector width fits the row
//
// Per row ("DeepJIT ... 串行小核墙" section 4.3: one block per row, the
// statistics reduced in the block, then the normalisation in the same pass
// over the data):  h = x (+ residual) in fp32; residual_out = dt(h);
// mean = sum(h)/HIDDEN; var = sum((h - mean)^2)/HIDDEN -- the same quantity
// as the page's E[h^2] - mean^2, taken in two passes over the registers so
// that fp32 does not cancel; out = dt((h - mean) * (1/sqrt(var + eps)) *
// gamma + beta).  Reductions: per-thread sums, a warp shuffle tree, then the
// warps' partial sums through shared memory.
#pragma once
#include "fuse/common.cuh"

constexpr int NWARPS = BLOCK / 32;
constexpr int NVR = HIDDEN / VEC;
constexpr int NWV = VEC * Dt<DT>::bytes / 4;

__device__ __forceinline__ float ln_block_sum(float v, float* part) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < NWARPS; ++i) t += part[i];
  return t;
}

// Pairwise combination of (count, mean, sum of squared deviations) of two
// disjoint sets (Chan, Golub and LeVeque's parallel variance update):
// mean = mean_a + d*n_b/n, M2 = M2_a + M2_b + d^2*n_a*n_b/n with
// d = mean_b - mean_a.  Empty sets (n = 0) leave the other side unchanged.
__device__ __forceinline__ void chan_merge(float& n, float& mean, float& m2, float nb, float meanb,
                                           float m2b) {
  const float nt = n + nb;
  if (nt == 0.f) return;
  const float d = meanb - mean;
  const float f = nb / nt;
  mean += d * f;
  m2 += m2b + d * d * n * f;
  n = nt;
}

#ifndef LN_MAX_REGS
#define LN_MAX_REGS 255
#endif
#if FUSE_LN_VEC
extern "C" __global__ void __maxnreg__(LN_MAX_REGS)
layernorm_vec(const void* x, const void* res, const void* gamma, const void* beta, void* out,
              void* res_out, long long rows, float eps) {
  pdl_enter();
  __shared__ float pn[NWARPS], pmean[NWARPS], pm2[NWARPS];
  constexpr long long ROW_W = (long long)HIDDEN * Dt<DT>::bytes / 4;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const u32* xr = static_cast<const u32*>(x) + row * ROW_W;
    u32 wx[R][NWV], wr[R][NWV];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      if (NVR % BLOCK == 0 || v < NVR) {
        load_words(xr + v * NWV, wx[i]);
        if constexpr (HAS_RES) load_words(static_cast<const u32*>(res) + row * ROW_W + v * NWV, wr[i]);
      }
    }
    float h[R][VEC];
    float s1 = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      if (NVR % BLOCK == 0 || v < NVR) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          h[i][e] = get_elem<DT>(wx[i], e);
          if constexpr (HAS_RES) h[i][e] += get_elem<DT>(wr[i], e);
          s1 += h[i][e];
        }
        if constexpr (HAS_RES) {
          u32 o[NWV];
          pack_vec<DT>(h[i], o);
          store_words(static_cast<u32*>(res_out) + row * ROW_W + v * NWV, o);
        }
      }
    }
    // this thread's (count, mean, M2) over its registers, then one merge tree:
    // warp lanes into lane 0, then every thread merges the warps' partials in
    // the same order (one barrier per row, identical statistics everywhere)
    float cnt = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (NVR % BLOCK == 0 || static_cast<int>(threadIdx.x) + i * BLOCK < NVR) cnt += VEC;
    float mean = cnt > 0.f ? s1 / cnt : 0.f, m2 = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      if (NVR % BLOCK == 0 || v < NVR) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float d = h[i][e] - mean;
          m2 += d * d;
        }
      }
    }
    if constexpr (NVR % BLOCK == 0 && (NWARPS & (NWARPS - 1)) == 0) {
      // every thread holds R*VEC values: each merge joins two equal sets, so
      // mean = (a + b) / 2 and M2 = M2a + M2b + d^2 * n / 2 (n per side)
      float half_n = 0.5f * cnt;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float mb = __shfl_down_sync(0xffffffffu, mean, o);
        const float qb = __shfl_down_sync(0xffffffffu, m2, o);
        const float d = mb - mean;
        mean = 0.5f * (mean + mb);
        m2 += qb + d * d * half_n;
        half_n *= 2.f;
      }
      if ((threadIdx.x & 31) == 0) {
        pmean[threadIdx.x >> 5] = mean;
        pm2[threadIdx.x >> 5] = m2;
      }
      __syncthreads();
      // the warps' partials merged by a butterfly over lanes (lane % NWARPS
      // holds warp lane % NWARPS); both partners of a step compute
      // mean = (a + b) / 2 and M2 = (M2a + M2b) + d^2 * n / 2, which do not
      // depend on the operand order, so every lane ends with the same bits
      mean = pmean[(threadIdx.x & 31) % NWARPS];
      m2 = pm2[(threadIdx.x & 31) % NWARPS];
#pragma unroll
      for (int step = 1; step < NWARPS; step *= 2) {
        const float mb = __shfl_xor_sync(0xffffffffu, mean, step);
        const float qb = __shfl_xor_sync(0xffffffffu, m2, step);
        const float d = mb - mean;
        mean = 0.5f * (mean + mb);
        m2 = (m2 + qb) + d * d * half_n;
        half_n *= 2.f;
      }
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float nb = __shfl_down_sync(0xffffffffu, cnt, o);
        const float mb = __shfl_down_sync(0xffffffffu, mean, o);
        const float qb = __shfl_down_sync(0xffffffffu, m2, o);
        chan_merge(cnt, mean, m2, nb, mb, qb);
      }
      if ((threadIdx.x & 31) == 0) {
        pn[threadIdx.x >> 5] = cnt;
        pmean[threadIdx.x >> 5] = mean;
        pm2[threadIdx.x >> 5] = m2;
      }
      __syncthreads();
      cnt = pn[0];
      mean = pmean[0];
      m2 = pm2[0];
#pragma unroll
      for (int w = 1; w < NWARPS; ++w) chan_merge(cnt, mean, m2, pn[w], pmean[w], pm2[w]);
    }
    const float rstd = 1.0f / sqrtf(m2 / HIDDEN + eps);
    // gamma and beta (the same for every row, cache-resident) are read only
    // now: the pointers pass through an empty asm that takes rstd, so the
    // compiler cannot hoist their loads above the reductions, where they would
    // hold registers
    const u32* gp = static_cast<const u32*>(gamma);
    const u32* bp = static_cast<const u32*>(beta);
    asm volatile("" : "+l"(gp), "+l"(bp) : "f"(rstd));
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int v = threadIdx.x + i * BLOCK;
      if (NVR % BLOCK == 0 || v < NVR) {
        u32 wg[NWV], wb[NWV];
        if constexpr (HAS_GAMMA) load_words_cached(gp + v * NWV, wg);
        if constexpr (HAS_BETA) load_words_cached(bp + v * NWV, wb);
        float y[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          float t = (h[i][e] - mean) * rstd;
          if constexpr (HAS_GAMMA) t *= get_elem<DT>(wg, e);
          if constexpr (HAS_BETA) t += get_elem<DT>(wb, e);
          y[e] = t;
        }
        u32 o[NWV];
        pack_vec<DT>(y, o);
        store_words(static_cast<u32*>(out) + row * ROW_W + v * NWV, o);
      }
    }
    __syncthreads();  // pn/pmean/pm2 are reused by the next row
  }
}
#endif

// any alignment: three passes over the row, element by element
extern "C" __global__ void __launch_bounds__(BLOCK)
layernorm_scalar(const void* x, const void* res, const void* gamma, const void* beta, void* out,
                 void* res_out, long long rows, float eps) {
  pdl_enter();
  __shared__ float part1[NWARPS], part2[NWARPS];
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const long long base = row * HIDDEN;
    float s1 = 0.f;
    for (int i = threadIdx.x; i < HIDDEN; i += BLOCK) {
      float hv = load_elem<DT>(x, base + i);
      if constexpr (HAS_RES) hv += load_elem<DT>(res, base + i);
      s1 += hv;
    }
    const float mean = ln_block_sum(s1, part1) / HIDDEN;
    float s2 = 0.f;
    for (int i = threadIdx.x; i < HIDDEN; i += BLOCK) {
      float hv = load_elem<DT>(x, base + i);
      if constexpr (HAS_RES) hv += load_elem<DT>(res, base + i);
      s2 += (hv - mean) * (hv - mean);
    }
    const float rstd = 1.0f / sqrtf(ln_block_sum(s2, part2) / HIDDEN + eps);
    for (int i = threadIdx.x; i < HIDDEN; i += BLOCK) {
      float hv = load_elem<DT>(x, base + i);
      if constexpr (HAS_RES) {
        hv += load_elem<DT>(res, base + i);
        store_elem<DT>(res_out, base + i, hv);
      }
      float t = (hv - mean) * rstd;
      if constexpr (HAS_GAMMA) t *= load_elem<DT>(gamma, i);
      if constexpr (HAS_BETA) t += load_elem<DT>(beta, i);
      store_elem<DT>(out, base + i, t);
    }
    __syncthreads();
  }
}
