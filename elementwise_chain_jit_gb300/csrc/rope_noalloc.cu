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
// device and held until the process exits), and both kernels are compiled
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
//    the file's four kernels are loaded there.  CUDA loads modules and
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

__global__ void rope_rows_build(float* rows, long long pos0, long long tokens, int hd,
                                double base) {
  const int half = hd / 2;
  const long long total = tokens * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long t = idx / half;
    const int i = static_cast<int>(idx % half);
    const double theta = static_cast<double>(pos0 + t) * pow(base, -2.0 * i / hd);
    double s, c;
    sincos(theta, &s, &c);
    rows[t * hd + i] = static_cast<float>(c);
    rows[t * hd + half + i] = static_cast<float>(s);
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

// The kernels of this file: loaded in the current context before the first
// launch, so that no launch (in particular none inside a stream capture)
// loads one lazily.
const void* const kKernels[] = {
    reinterpret_cast<const void*>(&rope_rows_build),
    reinterpret_cast<const void*>(&rope_noalloc_kernel<FUSE_F32>),
    reinterpret_cast<const void*>(&rope_noalloc_kernel<FUSE_F16>),
    reinterpret_cast<const void*>(&rope_noalloc_kernel<FUSE_BF16>),
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
  const long long total = tokens * (head_dim / 2);
  const unsigned grid = static_cast<unsigned>(std::min<long long>(d.sms * 8LL, (total + 255) / 256));
  rope_rows_build<<<grid, 256, 0, s>>>(rows, pos0, tokens, head_dim, static_cast<double>(base));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(FUSE_E_CUDA, fmt("rope_qkv_split_noalloc rows launch: %s", cudaGetErrorString(e)));
  stat_launch();
  const unsigned block = 256;
  if (dt == FUSE_F32)
    rope_noalloc_kernel<FUSE_F32><<<static_cast<unsigned>(tokens), block, 0, s>>>(
        qkv, q, k, v, rows, tokens, heads, head_dim);
  else if (dt == FUSE_F16)
    rope_noalloc_kernel<FUSE_F16><<<static_cast<unsigned>(tokens), block, 0, s>>>(
        qkv, q, k, v, rows, tokens, heads, head_dim);
  else
    rope_noalloc_kernel<FUSE_BF16><<<static_cast<unsigned>(tokens), block, 0, s>>>(
        qkv, q, k, v, rows, tokens, heads, head_dim);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(FUSE_E_CUDA, fmt("rope_qkv_split_noalloc launch: %s", cudaGetErrorString(e)));
  stat_launch();
  return FUSE_OK;
}
