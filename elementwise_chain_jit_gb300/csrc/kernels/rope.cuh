// rope.cuh -- QKV split + transpose + rotate-half RoPE, one CTA per token.
//
// The generated source defines before including this file:
//   DT      dtype code of qkv, q, k, v
//   HEADS   heads;  HD  head_dim (even);  HALF = HD / 2
//   BLOCK   threads per CTA
//   VEC     elements of each half a q/k item covers (HALF % VEC == 0)
//   VV      elements a v item copies (HD % VV == 0)
//   FUSE_ROPE_VEC  1 when vector widths fit (else only the scalar kernel)
//   ROW_PREFETCH  1: the vector kernel asks L2 for its token's row before
//           the launch-order wait
//
// qkv is [tokens, 3, HEADS, HD]; q, k, v are [HEADS, tokens, HD], with the
// token count a launch argument (one CTA per token), so one compiled kernel
// serves every token count.  Token t is at position pos0 + t; table[pos][0][i] = cos(theta), table[pos][1][i] =
// sin(theta), theta = pos * base^(-2i/HD), built on the device in fp64 and
// stored as fp32.  A q/k item rotates VEC pairs (i, i + HALF):
//   o[i] = x[i] cos - x[i + HALF] sin,  o[i + HALF] = x[i + HALF] cos + x[i] sin
// A v item copies VV elements bit for bit.  Each (token, head) row is
// contiguous on both sides, so every access is a 16/32-byte vector.
#pragma once
#include "fuse/common.cuh"

constexpr int BYTES = Dt<DT>::bytes;
constexpr int QK_PER_ROW = HALF / VEC;
constexpr int QK_ITEMS = 2 * HEADS * QK_PER_ROW;
constexpr int V_PER_ROW = HD / VV;
constexpr int V_ITEMS = HEADS * V_PER_ROW;
constexpr int NQK = (QK_ITEMS + BLOCK - 1) / BLOCK;  // q/k items per thread
constexpr int NV = (V_ITEMS + BLOCK - 1) / BLOCK;    // v items per thread
constexpr int NW = VEC * BYTES / 4;                  // words per half-vector
constexpr int NWV = VV * BYTES / 4;                  // words per v-vector
constexpr long long TOKEN_WORDS = 3LL * HEADS * HD * BYTES / 4;
constexpr int HD_WORDS = HD * BYTES / 4;
#if FUSE_ROPE_VEC
__host__ __device__ constexpr int cmin(int x, int y) { return x < y ? x : y; }
__host__ __device__ constexpr int cmax(int x, int y) { return x > y ? x : y; }
// Items a thread holds in registers at once: up to about 48 words of q/k
// operands (two half-vectors, their cosines and sines an item) and 16 words
// of v.  Rows wider than one round's items per thread take several rounds
// (a run-time loop), so neither registers nor the unrolled code grow with
// the head count.
constexpr int QB = cmin(NQK, cmax(1, 48 / (2 * NW + 2 * VEC)));
constexpr int VB = cmin(NV, cmax(1, 16 / NWV));
constexpr int ROUNDS = cmax((NQK + QB - 1) / QB, (NV + VB - 1) / VB);

// Round rd of a thread's work on token t: its v loads first, then the q/k
// loads, the rotation and the q/k stores, then the v stores.  In the common
// one-round case rd is the constant 0 and every bound check below whose
// items divide evenly over the block folds away.
__device__ __forceinline__ void rope_round(int rd, const u32* src, const float* tab, void* q, void* k,
                                           void* v, long long t, long long tokens) {
  constexpr bool V_EVEN = ROUNDS == 1 && V_ITEMS % BLOCK == 0;
  constexpr bool QK_EVEN = ROUNDS == 1 && QK_ITEMS % BLOCK == 0;
  u32 vw[VB][NWV];
#pragma unroll
  for (int n = 0; n < VB; ++n) {
    const int it = threadIdx.x + (rd * VB + n) * BLOCK;
    if (V_EVEN || it < V_ITEMS) {
      const int h = it / V_PER_ROW, j = it % V_PER_ROW;
      load_words(src + (2 * HEADS + h) * HD_WORDS + j * (NWV), vw[n]);
    }
  }
  u32 a[QB][NW], b[QB][NW], cw[QB][VEC], sw[QB][VEC];
#pragma unroll
  for (int n = 0; n < QB; ++n) {
    const int it = threadIdx.x + (rd * QB + n) * BLOCK;
    if (QK_EVEN || it < QK_ITEMS) {
      const int row = it / QK_PER_ROW;  // which * HEADS + h
      const int i0 = (it % QK_PER_ROW) * VEC;
      const u32* r = src + row * HD_WORDS;
      load_words(r + i0 * BYTES / 4, a[n]);
      load_words(r + (HALF + i0) * BYTES / 4, b[n]);
      load_words_cached(reinterpret_cast<const u32*>(tab + i0), cw[n]);
      load_words_cached(reinterpret_cast<const u32*>(tab + HALF + i0), sw[n]);
    }
  }
#pragma unroll
  for (int n = 0; n < QB; ++n) {
    const int it = threadIdx.x + (rd * QB + n) * BLOCK;
    if (QK_EVEN || it < QK_ITEMS) {
      const int row = it / QK_PER_ROW;
      const int which = row / HEADS, h = row % HEADS;
      const int i0 = (it % QK_PER_ROW) * VEC;
      float o1[VEC], o2[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float x1 = get_elem<DT>(a[n], e), x2 = get_elem<DT>(b[n], e);
        const float c = __uint_as_float(cw[n][e]), s = __uint_as_float(sw[n][e]);
        o1[e] = x1 * c - x2 * s;
        o2[e] = x2 * c + x1 * s;
      }
      u32* dst = static_cast<u32*>(which == 0 ? q : k) + (h * tokens + t) * HD_WORDS;
      u32 p1[NW], p2[NW];
      pack_vec<DT>(o1, p1);
      pack_vec<DT>(o2, p2);
      store_words(dst + i0 * BYTES / 4, p1);
      store_words(dst + (HALF + i0) * BYTES / 4, p2);
    }
  }
#pragma unroll
  for (int n = 0; n < VB; ++n) {
    const int it = threadIdx.x + (rd * VB + n) * BLOCK;
    if (V_EVEN || it < V_ITEMS) {
      const int h = it / V_PER_ROW, j = it % V_PER_ROW;
      store_words(static_cast<u32*>(v) + (h * tokens + t) * HD_WORDS + j * NWV, vw[n]);
    }
  }
}

extern "C" __global__ void __launch_bounds__(BLOCK)
rope_vec(const void* qkv, void* q, void* k, void* v, const float* table, long long pos0,
         long long tokens) {
  // ask L2 for (the first 64 KB of) the token's qkv row before waiting for the
  // previous kernel (programmatic dependent launch; L2 is coherent, the loads
  // come after)
  if constexpr (ROW_PREFETCH && (VEC * BYTES) % 16 == 0 && (VV * BYTES) % 16 == 0) {
    if (threadIdx.x == 0)
      prefetch_l2(static_cast<const u32*>(qkv) + blockIdx.x * TOKEN_WORDS,
                  static_cast<unsigned>(TOKEN_WORDS * 4 < 65536 ? TOKEN_WORDS * 4 : 65536));
  }
  pdl_enter();
  const long long t = blockIdx.x;
  const u32* src = static_cast<const u32*>(qkv) + t * TOKEN_WORDS;
  const float* tab = table + (pos0 + t) * (2 * HALF);
  if constexpr (ROUNDS == 1) {
    rope_round(0, src, tab, q, k, v, t, tokens);
  } else {
#pragma unroll 1
    for (int rd = 0; rd < ROUNDS; ++rd) rope_round(rd, src, tab, q, k, v, t, tokens);
  }
}

#endif

// any alignment: one element (or pair) per thread step
extern "C" __global__ void __launch_bounds__(BLOCK)
rope_scalar(const void* qkv, void* q, void* k, void* v, const float* table, long long pos0,
            long long tokens) {
  pdl_enter();
  const long long t = blockIdx.x;
  const long long src = t * 3LL * HEADS * HD;
  const float* tab = table + (pos0 + t) * (2 * HALF);
  for (int it = threadIdx.x; it < 2 * HEADS * HALF; it += BLOCK) {
    const int row = it / HALF, i = it % HALF;
    const int which = row / HEADS, h = row % HEADS;
    const float x1 = load_elem<DT>(qkv, src + row * HD + i);
    const float x2 = load_elem<DT>(qkv, src + row * HD + HALF + i);
    const float c = tab[i], s = tab[HALF + i];
    void* dst = which == 0 ? q : k;
    const long long o = (h * tokens + t) * HD;
    store_elem<DT>(dst, o + i, x1 * c - x2 * s);
    store_elem<DT>(dst, o + HALF + i, x2 * c + x1 * s);
  }
  for (int it = threadIdx.x; it < HEADS * HD; it += BLOCK) {
    const int h = it / HD, d = it % HD;
    typedef typename Dt<DT>::storage S;
    static_cast<S*>(v)[(h * tokens + t) * HD + d] =
        static_cast<const S*>(qkv)[src + (2 * HEADS + h) * HD + d];
  }
}
