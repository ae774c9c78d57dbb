// sync.cuh -- shared-memory addresses and mbarrier waits with a bound.
//
// Every wait in the library's kernels goes through mbar_wait: it tries the
// phase at most kMaxSpins times (each try may suspend the thread for a
// while) and then returns false, so that the caller records an error code
// and winds down instead of hanging.
#pragma once
#include "fuse/common.cuh"

// each try that finds the phase still open may suspend the thread for a few
// microseconds (measured on GB300: 2^22 tries took 15.7 s), so 2^18 tries
// give up after about a second -- 50,000 times the longest legitimate wait
// in these kernels (one block's main loop, ~21 us)
constexpr u32 kMaxSpins = 1u << 18;

__device__ __forceinline__ u32 dynamic_smem_bytes() {
  u32 r;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}

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
// bounded: false when the phase did not complete within `spins` tries
__device__ __forceinline__ bool mbar_wait(u32 bar, u32 parity, u32 spins = kMaxSpins) {
  for (u32 i = 0; i < spins; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// the same wait in all 32 lanes with one outcome for the warp: a lane that
// gave up makes the whole warp give up, so the .aligned tcgen05 loads after
// it are always executed by the full warp
__device__ __forceinline__ bool mbar_wait_warp(u32 bar, u32 parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}
