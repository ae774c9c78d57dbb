// common.cuh -- device helpers included by every generated kernel.
//
// Embedded into the library at build time and handed to NVRTC as the header
// "fuse/common.cuh".  No CUDA headers are needed: dtype conversions use the
// PTX cvt instructions (IEEE round-to-nearest-even), memory accesses use
// explicit 128-bit and 256-bit vector instructions.
#pragma once

typedef unsigned short u16;
typedef unsigned int u32;
typedef unsigned long long u64;

// ---------------------------------------------------------------- dtypes
// dtype codes match fuse_dtype: 0 = f32, 1 = f16, 2 = bf16

__device__ __forceinline__ float f16_to_f32(u16 h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}
__device__ __forceinline__ u16 f32_to_f16(float f) {
  u16 h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}
__device__ __forceinline__ float bf16_to_f32(u16 h) { return __uint_as_float(static_cast<u32>(h) << 16); }
__device__ __forceinline__ u16 f32_to_bf16(float f) {
  u16 h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}
// two floats -> one 32-bit word, element `lo` in the low half
__device__ __forceinline__ u32 pack2_f16(float lo, float hi) {
  u32 r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ u32 pack2_bf16(float lo, float hi) {
  u32 r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// 1/d for d >= 1: the hardware reciprocal approximation, documented (PTX ISA,
// rcp.approx.f32) to at most 1 ulp from 1/d over the whole range.  From
// d >= 2^126 on the true value is below the normal range and is flushed to 0;
// 1/inf = 0; NaN stays NaN.
__device__ __forceinline__ float rcp_ge1(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}
// logistic sigmoid 1 / (1 + exp(-x)), exp from CUDA's expf (no fast-math)
__device__ __forceinline__ float sigmoid(float x) { return rcp_ge1(1.0f + expf(-x)); }

// The opt-in approximations ("exp:fast", "sigmoid:fast" in a chain spec):
// exp(x) = 2^(x * L), L the fp32 nearest log2(e), by the hardware's ex2.approx
// with flush to zero.  Error: the product x * L is off by up to |x| (2^-24 for
// its rounding + 0.22 * 2^-24 for L's) in the exponent, which is a relative
// error of up to 1.25 * |x| * 2^-24 in the result; ex2.approx itself is within
// 2.45 * 2^-24 over every fp32 input with a normal result (measured on GB300
// over all of them; 3 * 2^-24 is used); results below 2^-126 flush to zero.
// inf, -inf and NaN give inf, 0 and NaN.
__device__ __forceinline__ float exp_fast(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x * 1.44269502162933349609375f));
  return r;
}
__device__ __forceinline__ float sigmoid_fast(float x) { return rcp_ge1(1.0f + exp_fast(-x)); }

// Packed fp32 pairs (sm_100 and later): one instruction adds or multiplies two
// lanes, each rounded to nearest even without flushing, the same bits as two
// scalar operations.  Inline asm, so the compiler does not contract them into
// fused multiply-adds.
__device__ __forceinline__ void add2(float& a, float& b, float c, float d) {
  unsigned long long x, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(c), "f"(d));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}
__device__ __forceinline__ void mul2(float& a, float& b, float c, float d) {
  unsigned long long x, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(c), "f"(d));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}

// exp_fast and sigmoid_fast on a pair, their adds and multiplies packed:
// each lane gets the bits of the scalar function
__device__ __forceinline__ float ex2_ftz(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}
__device__ __forceinline__ void exp_fast2(float& a, float& b) {
  mul2(a, b, 1.44269502162933349609375f, 1.44269502162933349609375f);
  a = ex2_ftz(a);
  b = ex2_ftz(b);
}
__device__ __forceinline__ void sigmoid_fast2(float& a, float& b) {
  mul2(a, b, -1.44269502162933349609375f, -1.44269502162933349609375f);
  float ea = ex2_ftz(a), eb = ex2_ftz(b);
  add2(ea, eb, 1.0f, 1.0f);
  a = rcp_ge1(ea);
  b = rcp_ge1(eb);
}

__device__ __forceinline__ float round_f16(float x) { return f16_to_f32(f32_to_f16(x)); }
__device__ __forceinline__ float round_bf16(float x) { return bf16_to_f32(f32_to_bf16(x)); }

template <int DT>
struct Dt;
template <>
struct Dt<0> {
  static constexpr int bytes = 4;
  typedef float storage;
};
template <>
struct Dt<1> {
  static constexpr int bytes = 2;
  typedef u16 storage;
};
template <>
struct Dt<2> {
  static constexpr int bytes = 2;
  typedef u16 storage;
};

// element e of a register vector of words holding dtype DT
template <int DT, int NW>
__device__ __forceinline__ float get_elem(const u32 (&w)[NW], int e) {
  if constexpr (DT == 0) {
    return __uint_as_float(w[e]);
  } else {
    const u32 x = w[e >> 1];
    const u16 h = (e & 1) ? static_cast<u16>(x >> 16) : static_cast<u16>(x & 0xffffu);
    if constexpr (DT == 1) return f16_to_f32(h);
    else return bf16_to_f32(h);
  }
}

// VEC floats -> words of dtype DT
template <int DT, int VEC, int NW>
__device__ __forceinline__ void pack_vec(const float (&y)[VEC], u32 (&w)[NW]) {
  if constexpr (DT == 0) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) w[i] = __float_as_uint(y[i]);
  } else {
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i)
      w[i] = DT == 1 ? pack2_f16(y[2 * i], y[2 * i + 1]) : pack2_bf16(y[2 * i], y[2 * i + 1]);
  }
}

// scalar element access (fallback kernels)
template <int DT>
__device__ __forceinline__ float load_elem(const void* p, long long i) {
  if constexpr (DT == 0) return static_cast<const float*>(p)[i];
  else if constexpr (DT == 1) return f16_to_f32(static_cast<const u16*>(p)[i]);
  else return bf16_to_f32(static_cast<const u16*>(p)[i]);
}
template <int DT>
__device__ __forceinline__ void store_elem(void* p, long long i, float v) {
  if constexpr (DT == 0) static_cast<float*>(p)[i] = v;
  else if constexpr (DT == 1) static_cast<u16*>(p)[i] = f32_to_f16(v);
  else static_cast<u16*>(p)[i] = f32_to_bf16(v);
}

// ---------------------------------------------------------------- memory
// Streaming loads of data read once: non-coherent path, no L1 allocation.
// The caller guarantees alignment to the access width.

__device__ __forceinline__ void ld_words32(const u32* p, u32* w) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}
__device__ __forceinline__ void ld_words16(const u32* p, u32* w) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p));
}
__device__ __forceinline__ void ld_words8(const u32* p, u32* w) {
  asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
}
__device__ __forceinline__ void st_words32(u32* p, const u32* w) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void st_words16(u32* p, const u32* w) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3])
               : "memory");
}
__device__ __forceinline__ void st_words8(u32* p, const u32* w) {
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(w[0]), "r"(w[1]) : "memory");
}

// NW consecutive words from p (p aligned to min(4*NW, 32) bytes), widest first
template <int NW>
__device__ __forceinline__ void load_words(const u32* p, u32 (&w)[NW]) {
  if constexpr (NW % 8 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 8) ld_words32(p + i, w + i);
  } else if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 4) ld_words16(p + i, w + i);
  } else if constexpr (NW % 2 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 2) ld_words8(p + i, w + i);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __ldg(p + i);
  }
}
template <int NW>
__device__ __forceinline__ void store_words(u32* p, const u32 (&w)[NW]) {
  if constexpr (NW % 8 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 8) st_words32(p + i, w + i);
  } else if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 4) st_words16(p + i, w + i);
  } else if constexpr (NW % 2 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 2) st_words8(p + i, w + i);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) p[i] = w[i];
  }
}

// Bulk prefetch of [p, p + bytes) into L2 (one thread issues it; p 16-byte
// aligned, bytes a multiple of 16).  A hint: it reads nothing into registers.
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- launch order
// Programmatic dependent launch (sm_90 and later).  A kernel launched with the
// programmatic-serialization attribute may have its CTAs scheduled before the
// previous kernel on the stream has finished; griddepcontrol.wait holds them
// until that kernel has completed and its writes are visible, so the stream
// order is kept.  launch_dependents then lets the next launch schedule its own
// CTAs early.  Both are no-ops for a launch without the attribute.  Every
// kernel of the library calls this first, before touching memory.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- reductions
// Every sum below is a balanced binary tree: a term passes through at most
// ceil(log2(number of nonzero terms)) fp32 additions at each stage (adding an
// exact zero does not round).  A row of n terms reduced per thread, across
// the lanes of a warp and across warps is therefore rounded at most
// ceil(log2 n) + 3 times on any path, which is what the error bounds of the
// row reductions are derived from.

// butterfly over the 32 lanes: every lane ends with the same bits (fp32
// addition is commutative, so both partners of a step compute the same sum)
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// a[0] + ... + a[N-1] as a balanced tree, in registers (N is a constant)
template <int N>
__device__ __forceinline__ float tree_sum(float (&a)[N]) {
#pragma unroll
  for (int w = 1; w < N; w *= 2) {
#pragma unroll
    for (int i = 0; i + w < N; i += 2 * w) a[i] += a[i + w];
  }
  return a[0];
}

__host__ __device__ constexpr int floor_log2(int n) { return n < 2 ? 0 : 1 + floor_log2(n / 2); }

// Cascade (pairwise) summation of N terms that arrive one at a time, in a
// loop the compiler unrolls: lvl[j] holds the sum of a complete tree of 2^j
// terms, like the bits of a binary counter, so the result is a balanced tree
// of depth ceil(log2 N) with only floor(log2 N) + 1 partial sums live.
template <int N>
struct Cascade {
  static constexpr int L = floor_log2(N) + 1;
  float lvl[L];
  // the k-th term (k counts from 0; k must fold to a constant)
  __device__ __forceinline__ void add(int k, float v) {
#pragma unroll
    for (int j = 0; j < L; ++j) {
      if ((k >> j) & 1) {
        v = lvl[j] + v;
      } else {
        lvl[j] = v;
        return;
      }
    }
  }
  // the partial trees of N's set bits, smallest first
  __device__ __forceinline__ float total() const {
    float acc = 0.f;
    bool first = true;
#pragma unroll
    for (int j = 0; j < L; ++j) {
      if ((N >> j) & 1) {
        acc = first ? lvl[j] : lvl[j] + acc;
        first = false;
      }
    }
    return acc;
  }
};

// Sum over a CTA of NWARPS_ warps: a butterfly within each warp, the warps'
// sums through shared memory `part`, then a second butterfly over them (lanes
// past NWARPS_ add zeros).  Every thread gets the same bits.  One barrier;
// the caller separates two uses of the same `part` by another barrier.
template <int NWARPS_>
__device__ __forceinline__ float cta_sum(float v, float* part) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  return warp_sum(lane < NWARPS_ ? part[lane] : 0.f);
}

// Loads of data many CTAs reuse (weights, tables): read-only path, cached.
__device__ __forceinline__ void ld_words32_cached(const u32* p, u32* w) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}
__device__ __forceinline__ void ld_words16_cached(const u32* p, u32* w) {
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p));
}
template <int NW>
__device__ __forceinline__ void load_words_cached(const u32* p, u32 (&w)[NW]) {
  if constexpr (NW % 8 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 8) ld_words32_cached(p + i, w + i);
  } else if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW; i += 4) ld_words16_cached(p + i, w + i);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __ldg(p + i);
  }
}
