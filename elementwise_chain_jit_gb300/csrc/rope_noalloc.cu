// rope_noalloc.cu -- rope_qkv_split_noalloc: QKV split + transpose + RoPE
// that allocates nothing.
//
// rope_qkv_split() keeps its cos/sin table in device memory it allocates
// itself (cuMemAlloc on first use and whenever the table must grow), and
// compiles its kernel with NVRTC on the first call for a shape.  Some callers
// cannot let a library do either: a serving process whose device memory has
// all been handed to its own caching allocator or arena, code that runs while
// a stream is being captured into a CUDA graph (where an allocation, or the
// synchronisation that may come with it, is an error), and latency-critical
// loops that forbid allocations after start-up.  This entry point serves them:
// its cos/sin rows live in a fixed array that is part of the library's own
// module (static device memory, reserved when the module is loaded on a
// device and held until the process exits), and its kernels are compiled
// ahead of time.
//
// Limits and sharing:
//  * tokens * head_dim <= kScratchFloats (2^20 fp32 values, 4 MB): one row of
//    head_dim/2 cosines and head_dim/2 sines per token of the call.  Larger
//    calls are rejected with FUSE_E_SHAPE.
//  * Every call on a device uses the same array, and each call rewrites the
//    rows it needs before reading them (nothing has to start at zero).  Two
//    calls whose work overlaps on the GPU -- on different streams, or from
//    different threads without ordering -- race on the array and may read each
//    other's rows.  Serialise them on one stream.
//  * Set-up, once per CUDA context: the array's device address is looked up
//    in the calling thread's current context (host code cannot use the
//    symbol itself: on the host it names a stand-in, not device memory), and
//    the file's seven kernels are loaded there.  CUDA loads modules and
//    kernels lazily by default (on first use), which allocates device memory
//    for their code and data, so the FIRST call in a context does that work,
//    whatever its dtype; make it before any stream capture begins and before
//    an arena takes the remaining device memory.  The result is kept per
//    context, under the driver's unique context id (never reused within a
//    process, so a context made after a device reset is set up afresh);
//    later calls allocate nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>

#include "internal.h"

// The shared cos/sin rows: row t (t < tokens of the call) holds cos(theta_i)
// for i < half, then sin(theta_i), for the token's position pos0 + t.
static constexpr long long kScratchFloats = 1LL << 20;
static __device__ __align__(256) float g_rope_rows[kScratchFloats];

namespace {

// sin and cos of a binary64 angle 0 <= theta < 2^22 (positions are below 2^22
// and the frequencies at most 1), to about binary64 accuracy.  Cody and
// Waite's reduction by pi/2, with pi/2 in three parts whose first two carry 30
// bits, so that k times each is exact for k < 2^22: r = theta - k pi/2 in
// [-pi/4, pi/4].  Then the Taylor series of sin to r^17 and of cos to r^18
// (remainders below 1e-19 there), and the quadrant k mod 4.
__device__ __forceinline__ void sincos_pos(double th, double* s, double* c) {
  const double k = rint(th * 0x1.45f306dc9c883p-1);  // theta * 2/pi
  double r = th - k * 0x1.921fb54000000p+0;
  r = r - k * 0x1.10b4611800000p-30;
  r = r - k * 0x1.313198a2e0370p-61;
  const double r2 = r * r;
  // 1/(2j+1)! and 1/(2j)!, alternating signs, j = 8 .. 0
  double ps = 0x1.952c77030ad4ap-49;
  ps = ps * r2 - 0x1.ae7f3e733b81fp-41;
  ps = ps * r2 + 0x1.6124613a86d09p-33;
  ps = ps * r2 - 0x1.ae64567f544e4p-26;
  ps = ps * r2 + 0x1.71de3a556c734p-19;
  ps = ps * r2 - 0x1.a01a01a01a01ap-13;
  ps = ps * r2 + 0x1.1111111111111p-7;
  ps = ps * r2 - 0x1.5555555555555p-3;
  const double sr = r + r * r2 * ps;
  double pc = -0x1.6827863b97d97p-53;
  pc = pc * r2 + 0x1.ae7f3e733b81fp-45;
  pc = pc * r2 - 0x1.93974a8c07c9dp-37;
  pc = pc * r2 + 0x1.1eed8eff8d898p-29;
  pc = pc * r2 - 0x1.27e4fb7789f5cp-22;
  pc = pc * r2 + 0x1.a01a01a01a01ap-16;
  pc = pc * r2 - 0x1.6c16c16c16c17p-10;
  pc = pc * r2 + 0x1.5555555555555p-5;
  pc = pc * r2 - 0.5;
  const double cr = 1.0 + r2 * pc;
  switch (static_cast<long long>(k) & 3) {
    case 0: *s = sr; *c = cr; break;
    case 1: *s = cr; *c = -sr; break;
    case 2: *s = -sr; *c = -cr; break;
    default: *s = -cr; *c = sr; break;
  }
}

// Row t of the shared array: cos(theta_i) for i < half, then sin(theta_i), with
// theta_i = (pos0 + t) * w_i and w_i = base^(-2i/hd).  Each CTA first takes
// w_i, cos w_i and sin w_i for every i of the head, in binary64; a thread then
// takes one i over a run of kRun consecutive tokens: sin and cos of the first
// angle directly (sincos_pos), and each next one by the angle-addition
// rotation by w_i, also in binary64.  The rotations add at most a few 1e-16 to
// the values over a run, far below an fp32 rounding, while the direct
// evaluations, the expensive part in binary64, drop to one in kRun.
constexpr int kRun = 16;

__global__ void rope_rows_build(float* rows, long long pos0, long long tokens, int hd,
                                double base) {
  __shared__ double w[512], cw[512], sw[512];
  const int half = hd / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    w[i] = pow(base, -2.0 * i / hd);
    sincos_pos(w[i], &sw[i], &cw[i]);
  }
  __syncthreads();
  const long long runs = (tokens + kRun - 1) / kRun;
  const long long total = runs * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long t0 = (idx / half) * kRun;
    const int i = static_cast<int>(idx % half);
    double sn, cs;
    sincos_pos(static_cast<double>(pos0 + t0) * w[i], &sn, &cs);
    const long long tn = tokens - t0 < kRun ? tokens - t0 : kRun;
    for (long long m = 0; m < tn; ++m) {
      rows[(t0 + m) * hd + i] = static_cast<float>(cs);
      rows[(t0 + m) * hd + half + i] = static_cast<float>(sn);
      const double c2 = cs * cw[i] - sn * sw[i];
      sn = sn * cw[i] + cs * sw[i];
      cs = c2;
    }
  }
}

template <int DT>
struct Elem;
template <>
struct Elem<FUSE_F32> {
  typedef float S;
  static __device__ float load(const S* p, long long i) { return p[i]; }
  static __device__ void store(S* p, long long i, float v) { p[i] = v; }
};
template <>
struct Elem<FUSE_F16> {
  typedef unsigned short S;
  static __device__ float load(const S* p, long long i) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(p[i]));
    return f;
  }
  static __device__ void store(S* p, long long i, float v) {
    unsigned short h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
    p[i] = h;
  }
};
template <>
struct Elem<FUSE_BF16> {
  typedef unsigned short S;
  static __device__ float load(const S* p, long long i) {
    return __uint_as_float(static_cast<unsigned>(p[i]) << 16);
  }
  static __device__ void store(S* p, long long i, float v) {
    unsigned short h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
    p[i] = h;
  }
};

// One CTA per token: the same split, transpose and rotation as the generated
// rope kernel, with the sizes as arguments and element-wise accesses.
template <int DT>
__global__ void rope_noalloc_kernel(const void* qkv, void* q, void* k, void* v, const float* rows,
                                    long long tokens, int heads, int hd) {
  typedef Elem<DT> E;
  typedef typename E::S S;
  const long long t = blockIdx.x;
  const int half = hd / 2;
  const S* src = static_cast<const S*>(qkv) + t * 3LL * heads * hd;
  const float* row = rows + t * hd;
  for (int it = threadIdx.x; it < 2 * heads * half; it += blockDim.x) {
    const int r = it / half, i = it % half;
    const int which = r / heads, h = r % heads;
    const float x1 = E::load(src, (long long)r * hd + i);
    const float x2 = E::load(src, (long long)r * hd + half + i);
    const float c = row[i], s = row[half + i];
    S* dst = static_cast<S*>(which == 0 ? q : k) + (h * tokens + t) * hd;
    E::store(dst, i, x1 * c - x2 * s);
    E::store(dst, half + i, x2 * c + x1 * s);
  }
  for (int it = threadIdx.x; it < heads * hd; it += blockDim.x) {
    const int h = it / hd, d = it % hd;
    static_cast<S*>(v)[(h * tokens + t) * hd + d] = src[(2LL * heads + h) * hd + d];
  }
}

// 16-byte vectors of NV elements (NV = 8 for f16/bf16, 4 for f32), unpacked to
// and packed from fp32 registers
template <int DT>
struct Vec16 {
  static constexpr int NV = DT == FUSE_F32 ? 4 : 8;
  static __device__ void unpack(const uint4& w, float (&x)[NV]) {
    const unsigned u[4] = {w.x, w.y, w.z, w.w};
    if constexpr (DT == FUSE_F32) {
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j] = __uint_as_float(u[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const unsigned short lo = static_cast<unsigned short>(u[j] & 0xffffu);
        const unsigned short hi = static_cast<unsigned short>(u[j] >> 16);
        if constexpr (DT == FUSE_BF16) {
          x[2 * j] = __uint_as_float(static_cast<unsigned>(lo) << 16);
          x[2 * j + 1] = __uint_as_float(static_cast<unsigned>(hi) << 16);
        } else {
          asm("cvt.f32.f16 %0, %1;" : "=f"(x[2 * j]) : "h"(lo));
          asm("cvt.f32.f16 %0, %1;" : "=f"(x[2 * j + 1]) : "h"(hi));
        }
      }
    }
  }
  static __device__ uint4 pack(const float (&y)[NV]) {
    unsigned u[4];
    if constexpr (DT == FUSE_F32) {
#pragma unroll
      for (int j = 0; j < 4; ++j) u[j] = __float_as_uint(y[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (DT == FUSE_BF16)
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(u[j]) : "f"(y[2 * j + 1]), "f"(y[2 * j]));
        else
          asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(u[j]) : "f"(y[2 * j + 1]), "f"(y[2 * j]));
      }
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
};

// The same kernel with 16-byte accesses: a q/k item rotates NV pairs (NV
// elements of each half row, with their NV cosines and sines), a v item copies
// NV elements.  The host takes it when head_dim / 2 is a multiple of NV and
// every tensor is 16-byte aligned (so every access is).
template <int DT>
__global__ void rope_noalloc_vec(const void* qkv, void* q, void* k, void* v, const float* rows,
                                 long long tokens, int heads, int hd) {
  typedef Vec16<DT> V;
  constexpr int NV = V::NV;
  typedef typename Elem<DT>::S S;
  const long long t = blockIdx.x;
  const int half = hd / 2, per_half = half / NV;
  const S* src = static_cast<const S*>(qkv) + t * 3LL * heads * hd;
  const float* row = rows + t * hd;
  for (int it = threadIdx.x; it < 2 * heads * per_half; it += blockDim.x) {
    const int r = it / per_half, i0 = (it % per_half) * NV;
    const int which = r / heads, h = r % heads;
    const uint4 wa = *reinterpret_cast<const uint4*>(src + static_cast<long long>(r) * hd + i0);
    const uint4 wb =
        *reinterpret_cast<const uint4*>(src + static_cast<long long>(r) * hd + half + i0);
    float x1[NV], x2[NV], c[NV], s[NV], o1[NV], o2[NV];
#pragma unroll
    for (int j = 0; j < NV; j += 4) {
      const float4 cj = *reinterpret_cast<const float4*>(row + i0 + j);
      const float4 sj = *reinterpret_cast<const float4*>(row + half + i0 + j);
      c[j] = cj.x; c[j + 1] = cj.y; c[j + 2] = cj.z; c[j + 3] = cj.w;
      s[j] = sj.x; s[j + 1] = sj.y; s[j + 2] = sj.z; s[j + 3] = sj.w;
    }
    V::unpack(wa, x1);
    V::unpack(wb, x2);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      o1[j] = x1[j] * c[j] - x2[j] * s[j];
      o2[j] = x2[j] * c[j] + x1[j] * s[j];
    }
    S* dst = static_cast<S*>(which == 0 ? q : k) + (h * tokens + t) * hd;
    *reinterpret_cast<uint4*>(dst + i0) = V::pack(o1);
    *reinterpret_cast<uint4*>(dst + half + i0) = V::pack(o2);
  }
  const int per_row = hd / NV;
  for (int it = threadIdx.x; it < heads * per_row; it += blockDim.x) {
    const int h = it / per_row, d0 = (it % per_row) * NV;
    *reinterpret_cast<uint4*>(static_cast<S*>(v) + (h * tokens + t) * hd + d0) =
        *reinterpret_cast<const uint4*>(src + (2LL * heads + h) * hd + d0);
  }
}

// The kernels of this file: loaded in the current context before the first
// launch, so that no launch (in particular none inside a stream capture)
// loads one lazily.
const void* const kKernels[] = {
    reinterpret_cast<const void*>(&rope_rows_build),
    reinterpret_cast<const void*>(&rope_noalloc_kernel<FUSE_F32>),
    reinterpret_cast<const void*>(&rope_noalloc_kernel<FUSE_F16>),
    reinterpret_cast<const void*>(&rope_noalloc_kernel<FUSE_BF16>),
    reinterpret_cast<const void*>(&rope_noalloc_vec<FUSE_F32>),
    reinterpret_cast<const void*>(&rope_noalloc_vec<FUSE_F16>),
    reinterpret_cast<const void*>(&rope_noalloc_vec<FUSE_BF16>),
};

int ensure_loaded(const void* kernel) {
  cudaFunction_t f = nullptr;
  cudaError_t e = cudaGetFuncBySymbol(&f, kernel);
  if (e != cudaSuccess)
    return fuse::fail(FUSE_E_CUDA, fuse::fmt("cudaGetFuncBySymbol: %s", cudaGetErrorString(e)));
  const fuse::DriverApi* api;
  if (int rc = fuse::driver(&api)) return rc;
  CUfunction cf = reinterpret_cast<CUfunction>(f);
  if (api->FuncIsLoaded && api->FuncLoad) {
    CUfunctionLoadingState st = CU_FUNCTION_LOADING_STATE_UNLOADED;
    CUresult r = api->FuncIsLoaded(&st, cf);
    if (r == CUDA_SUCCESS && st == CU_FUNCTION_LOADING_STATE_LOADED) return FUSE_OK;
    r = api->FuncLoad(cf);
    if (r != CUDA_SUCCESS) return fuse::cuda_fail(r, "cuFuncLoad (rope_qkv_split_noalloc)");
    return FUSE_OK;
  }
  // a driver without cuFuncLoad: reading the kernel's attributes loads it
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kernel);
  if (e != cudaSuccess)
    return fuse::fail(FUSE_E_CUDA, fuse::fmt("cudaFuncGetAttributes: %s", cudaGetErrorString(e)));
  return FUSE_OK;
}

// The array's device address in the current context, with every kernel of
// the file loaded there.
int setup_context(float** out) {
  float* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_rope_rows);
  if (e != cudaSuccess)
    return fuse::fail(FUSE_E_CUDA,
                      fuse::fmt("cudaGetSymbolAddress(rope rows): %s", cudaGetErrorString(e)));
  for (const void* k : kKernels)
    if (int rc = ensure_loaded(k)) return rc;
  *out = p;
  return FUSE_OK;
}

std::mutex g_ctx_mu;
std::map<unsigned long long, float*> g_ctx_rows;  // context id -> array address

// Set up the current context once; later calls find the address here.  A
// driver without context ids gets the set-up on every call (it allocates
// nothing once done, but needs the runtime's symbol lookup each time).
int rows_in_current_context(float** out) {
  const fuse::DriverApi* api;
  if (int rc = fuse::driver(&api)) return rc;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!api->CtxGetId || api->CtxGetCurrent(&ctx) != CUDA_SUCCESS || !ctx ||
      api->CtxGetId(ctx, &id) != CUDA_SUCCESS)
    return setup_context(out);
  std::lock_guard<std::mutex> lk(g_ctx_mu);
  if (auto it = g_ctx_rows.find(id); it != g_ctx_rows.end()) {
    *out = it->second;
    return FUSE_OK;
  }
  if (int rc = setup_context(out)) return rc;
  g_ctx_rows.emplace(id, *out);
  return FUSE_OK;
}

}  // namespace

extern "C" int rope_qkv_split_noalloc(const void* qkv, void* q, void* k, void* v, int64_t tokens,
                                      int heads, int head_dim, int64_t pos0, float base,
                                      fuse_dtype dt, void* stream) {
  fuse::NvtxRange nvtx_range("rope_qkv_split_noalloc");
  using namespace fuse;
  if (!valid_dtype(dt)) return fail(FUSE_E_DTYPE, fmt("invalid dtype %d", dt));
  if (tokens < 0 || heads < 1 || head_dim < 2 || head_dim > 1024 || head_dim % 2)
    return fail(FUSE_E_SHAPE, "need tokens >= 0, heads >= 1, head_dim even in 2..1024");
  if (heads > (1 << 20) / head_dim) return fail(FUSE_E_SHAPE, "heads * head_dim above 2^20");
  // (no product is formed before the operands are known to be small)
  if (tokens > kScratchFloats / head_dim)
    return fail(FUSE_E_SHAPE,
                fmt("tokens %lld * head_dim %d exceeds this entry point's fixed table of %lld "
                    "values; split the call or use rope_qkv_split",
                    (long long)tokens, head_dim, kScratchFloats));
  if (pos0 < 0 || pos0 > (int64_t(1) << 22) || tokens > (int64_t(1) << 22) - pos0)
    return fail(FUSE_E_SHAPE, "positions must lie in [0, 2^22)");
  if (!(base > 1.f) || !std::isfinite(base)) return fail(FUSE_E_ARG, "base must be finite and > 1");
  if (tokens == 0) return FUSE_OK;
  if (!qkv || !q || !k || !v) return fail(FUSE_E_NULL, "NULL tensor pointer");
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  float* rows = nullptr;
  if (int rc = rows_in_current_context(&rows)) return rc;
  // this library's runtime keeps its own last-error state; drop any error an
  // earlier call left there, so that only this call's launches are checked
  (void)cudaGetLastError();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one thread per (run of 16 tokens, pair index), at most two CTAs per SM
  // (each takes the head's frequencies once)
  const long long total = (tokens + 15) / 16 * (head_dim / 2);
  const unsigned grid = static_cast<unsigned>(std::min<long long>(d.sms * 2LL, (total + 255) / 256));
  rope_rows_build<<<grid, 256, 0, s>>>(rows, pos0, tokens, head_dim, static_cast<double>(base));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(FUSE_E_CUDA, fmt("rope_qkv_split_noalloc rows launch: %s", cudaGetErrorString(e)));
  stat_launch();
  const unsigned block = 256, ntok = static_cast<unsigned>(tokens);
  // 16-byte accesses when half a row is a whole number of vectors and every
  // tensor is 16-byte aligned; element-wise otherwise
  const int nv = dt == FUSE_F32 ? 4 : 8;
  bool vec = (head_dim / 2) % nv == 0;
  for (const void* p : {qkv, static_cast<const void*>(q), static_cast<const void*>(k),
                        static_cast<const void*>(v)})
    vec = vec && aligned16(p);
  if (dt == FUSE_F32) {
    if (vec) rope_noalloc_vec<FUSE_F32><<<ntok, block, 0, s>>>(qkv, q, k, v, rows, tokens, heads, head_dim);
    else rope_noalloc_kernel<FUSE_F32><<<ntok, block, 0, s>>>(qkv, q, k, v, rows, tokens, heads, head_dim);
  } else if (dt == FUSE_F16) {
    if (vec) rope_noalloc_vec<FUSE_F16><<<ntok, block, 0, s>>>(qkv, q, k, v, rows, tokens, heads, head_dim);
    else rope_noalloc_kernel<FUSE_F16><<<ntok, block, 0, s>>>(qkv, q, k, v, rows, tokens, heads, head_dim);
  } else {
    if (vec) rope_noalloc_vec<FUSE_BF16><<<ntok, block, 0, s>>>(qkv, q, k, v, rows, tokens, heads, head_dim);
    else rope_noalloc_kernel<FUSE_BF16><<<ntok, block, 0, s>>>(qkv, q, k, v, rows, tokens, heads, head_dim);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(FUSE_E_CUDA, fmt("rope_qkv_split_noalloc launch: %s", cudaGetErrorString(e)));
  stat_launch();
  return FUSE_OK;
}
