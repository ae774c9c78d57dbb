// rms_linear.cuh -- RMSNorm -> Linear -> scale on the 5th-generation tensor
// cores (tcgen05), one 128 x 256 output tile per CTA.
//
// "TeleTron" section 4.2 fuses RMSNorm into the linear layer: the row's RMS
// factor is computed in the block and used directly in the accumulation, so
// no normalised tensor is written.  Here
//   out[m, n] = scale * (s_m * sum_k (x[m,k] * gamma[k]) * w[n,k] + bias[n]),
//   s_m = 1 / sqrt(sum_k x[m,k]^2 / K + eps),
// with x [M, K], w [N, K] (K-major, as the MMA wants both operands), gamma
// [K], bias [N], out [M, N], all f16 or all bf16, fp32 accumulation in TMEM.
//
// Roles (6 warps):
//   warp 0     TMA producer: x tile 128 x 64 and w tile 256 x 64 per stage
//              (128-byte swizzle), STAGES-deep ring, mbarrier complete_tx.
//   warps 2-5  one tile row per thread: sum of squares of the row's x, then
//              x * gamma written back in place (the MMA's A operand); a
//              proxy fence, then "ready".  After the main loop the same
//              threads run the epilogue for their row: TMEM -> registers ->
//              s_m * acc + bias, * scale -> global.
//   warp 1     allocates 256 TMEM columns; one thread issues tcgen05.mma
//              (M 128, N 256, K 16; four per stage) and commits each stage to
//              its "empty" barrier, and the tile to "accum".
// Every mbarrier wait is bounded; a wait that runs out sets *err and the
// kernel winds down (it waits, again bounded, for its own TMA copies and
// frees its TMEM) instead of hanging.
//
// The generated source defines: DT (1 f16, 2 bf16), KDIM, NDIM, STAGES,
// HAS_BIAS, APPLY_GAMMA.  With APPLY_GAMMA false, gamma has already been
// folded into w (rms_linear_fold below): the row warps only read the x tile
// for the sum of squares, and the MMA consumes the TMA tiles as they land.
#pragma once
#include "fuse/common.cuh"

// w'[n, k] = dt(w[n, k] * gamma[k]): gamma folded into the weight once, so
// that the tile loop needs no transform of the A operand.
extern "C" __global__ void rms_linear_fold(const u16* __restrict__ w, const u16* __restrict__ gamma,
                                           u16* __restrict__ wout, long long total) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x)
    store_elem<DT>(wout, i, load_elem<DT>(w, i) * load_elem<DT>(gamma, i % KDIM));
}

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int KT = KDIM / BK;
constexpr u32 TMEM_COLS = 256;
constexpr u32 kMaxSpins = 1u << 22;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 8 * (3 * STAGES + 1) + 16;

struct __align__(64) TensorMap {
  unsigned long long v[16];
};

__device__ __forceinline__ u32 smem_u32(const void* p) {
  u32 r;
  asm("{ .reg .u64 t; cvta.to.shared.u64 t, %1; cvt.u32.u64 %0, t; }" : "=r"(r) : "l"(p));
  return r;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(u32 bar, u32 count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(u32 bar, u32 bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(u32 bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(u32 bar, u32 parity) {
  u32 ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded: false when the phase did not complete within kMaxSpins tries
__device__ __forceinline__ bool mbar_wait(u32 bar, u32 parity) {
  for (u32 i = 0; i < kMaxSpins; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(u32 dst, const TensorMap* map, u32 bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<unsigned long long>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(u32 slot, u32 ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(u32 taddr, u32 ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma(u32 d_tmem, unsigned long long a, unsigned long long b,
                                     u32 idesc, u32 accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, "
      "p; }" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(u32 bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_ld32(u32 taddr, u32 (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
//   bits  0-13 start address >> 4      bits 16-29 leading offset (unused here)
//   bits 32-45 stride offset >> 4      bits 46-48 0b001 (tcgen05 descriptor)
//   bits 61-63 swizzle mode (2 = 128-byte)
__device__ __forceinline__ unsigned long long sw128_desc(u32 addr) {
  unsigned long long d = (addr & 0x3FFFFu) >> 4;
  d |= 1ull << 16;
  d |= (unsigned long long)(1024 >> 4) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B f16 (0)
// or bf16 (1) in bits 7-9 / 10-12, both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
constexpr u32 kIdesc = (1u << 4) | ((DT == 2 ? 1u : 0u) << 7) | ((DT == 2 ? 1u : 0u) << 10) |
                            ((u32)(BN >> 3) << 17) | ((u32)(BM >> 4) << 24);

extern "C" __global__ void __launch_bounds__(192, 1)
rms_linear_kernel(const __grid_constant__ TensorMap tmap_x, const __grid_constant__ TensorMap tmap_w,
                  const u16* __restrict__ gamma, const u16* __restrict__ bias, u16* __restrict__ out,
                  float eps, float scale, int* err) {
  extern __shared__ unsigned char smem_raw[];
  const u32 raw = smem_u32(smem_raw);
  const u32 base = (raw + 1023u) & ~1023u;  // tiles 1024-aligned for the swizzle
  unsigned char* const base_ptr = smem_raw + (base - raw);
  const u32 bars = base + STAGES * STAGE_BYTES;
  auto stage_a = [&](int s) { return base + s * STAGE_BYTES; };
  auto stage_b = [&](int s) { return base + s * STAGE_BYTES + A_BYTES; };
  auto full = [&](int s) { return bars + 8u * s; };
  auto ready = [&](int s) { return bars + 8u * (STAGES + s); };
  auto empty = [&](int s) { return bars + 8u * (2 * STAGES + s); };
  const u32 accum = bars + 8u * (3 * STAGES);
  const u32 tmem_slot = accum + 8u;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(ready(s), 128);
      // with gamma applied in place the MMA's commit frees a stage (the row
      // warps finished before "ready"); with gamma folded into w the four
      // row warps, which only read the stage, arrive as well
      mbar_init(empty(s), APPLY_GAMMA ? 1 : 5);
    }
    mbar_init(accum, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const u32 tmem = *reinterpret_cast<volatile u32*>(base_ptr + (tmem_slot - base));

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      int issued = -1;
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % STAGES;
        const u32 ph = (kt / STAGES) & 1;
        if (!mbar_wait(empty(s), ph ^ 1)) { ok = false; break; }
        mbar_expect_tx(full(s), STAGE_BYTES);
        tma_load_2d(stage_a(s), &tmap_x, full(s), kt * BK, m0);
        tma_load_2d(stage_b(s), &tmap_w, full(s), kt * BK, n0);
        issued = kt;
      }
      if (!ok)  // let the copies already in flight land before the CTA exits
        for (int kt = issued - STAGES + 1 < 0 ? 0 : issued - STAGES + 1; kt <= issued; ++kt)
          mbar_wait(full(kt % STAGES), (kt / STAGES) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % STAGES;
        if (!mbar_wait(APPLY_GAMMA ? ready(s) : full(s), (kt / STAGES) & 1)) { ok = false; break; }
        tc_fence_after();
        const unsigned long long a = sw128_desc(stage_a(s)), b = sw128_desc(stage_b(s));
#pragma unroll
        for (int j = 0; j < BK / 16; ++j)  // K 16 = 32 bytes further along the swizzled rows
          umma(tmem, a + 2ull * j, b + 2ull * j, kIdesc, (kt | j) != 0);
        umma_commit(empty(s));
      }
      umma_commit(accum);
    }
  } else {
    const int q = warp & 3;       // the TMEM lane quarter this warp may read
    const int r = q * 32 + lane;  // this thread's row of the tile
    float ss = 0.f;
    for (int kt = 0; kt < KT; ++kt) {
      const int s = kt % STAGES;
      if (!mbar_wait(full(s), (kt / STAGES) & 1)) { ok = false; break; }
      // the row's 128 bytes hold its 64 values in 16-byte chunks, logical
      // chunk c at position c ^ (r % 8) (the 128-byte swizzle); step p visits
      // logical chunk p, so the 8 rows of a swizzle group hit 8 different
      // bank groups
      uint4* row = reinterpret_cast<uint4*>(base_ptr + (stage_a(s) - base) + r * 128);
      if constexpr (APPLY_GAMMA) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const uint4 g4 = __ldg(reinterpret_cast<const uint4*>(gamma + kt * BK + p * 8));
          uint4& slot = row[p ^ (r & 7)];
          uint4 v4 = slot;
          u32 wv[4] = {v4.x, v4.y, v4.z, v4.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w};
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float xv = get_elem<DT>(wv, e);
            ss += xv * xv;
            y[e] = xv * get_elem<DT>(gw, e);
          }
          pack_vec<DT>(y, wv);
          slot = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(ready(s));
      } else {
        // gamma is folded into w: only the sum of squares, read-only
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const uint4 v4 = row[p ^ (r & 7)];
          const u32 wv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float xv = get_elem<DT>(wv, e);
            ss += xv * xv;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
      }
    }
    const float rs = 1.0f / sqrtf(ss / KDIM + eps);
    if (!mbar_wait(accum, 0)) ok = false;
    tc_fence_after();
    u16* orow = out + (long long)(m0 + r) * NDIM + n0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      u32 acc[32];
      tmem_ld32(tmem + ((u32)(q * 32) << 16) + c * 32, acc);
      float y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float t = __uint_as_float(acc[i]) * rs;
        if constexpr (HAS_BIAS) t += load_elem<DT>(bias, n0 + c * 32 + i);
        y[i] = t * scale;
      }
      u32 o[16];
      pack_vec<DT>(y, o);
#pragma unroll
      for (int i = 0; i < 4; ++i) st_words16(reinterpret_cast<u32*>(orow + c * 32) + 4 * i, o + 4 * i);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (!ok) atomicExch(err, 1);
}
