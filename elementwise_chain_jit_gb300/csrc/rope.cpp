// rope.cpp -- QKV split + transpose + rotate-half RoPE entry point.
//
// "TeleTron" section 3.1 names QKV projection -> head split -> RoPE -> scale
// as one multi-step fusion.  The projection is a GEMM and stays outside; the
// split, the [T,3,H,D] -> [H,T,D] transpose and the rotation are one kernel
// here: each token is one CTA, each (token, head) row is read and written as
// contiguous 16/32-byte vectors, and cos/sin come from a per-device table
// (fp64-built, fp32-stored) that stays resident in L2 across the 2*H q/k rows
// of a token.
#include <algorithm>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <map>
#include <tuple>

#include "internal.h"

namespace fuse {
namespace {

constexpr int64_t kMaxPositions = int64_t(1) << 22;

struct RopeKernel {
  std::shared_ptr<Module> mod;
  int block = 256;
  bool has_vec = false;
  int vec = 1, vv = 1;
};

struct Table {
  CUdeviceptr ptr = 0;
  int64_t cap = 0;  // positions
};

std::mutex g_mu;
std::map<std::tuple<int, int, int>, RopeKernel> g_kernels;  // (heads, head_dim, dtype)
std::map<std::tuple<int, uint32_t, int>, Table> g_tables;  // (device, base bits, head_dim)
std::vector<CUdeviceptr> g_retired;  // outgrown tables, kept: in-flight kernels may read them
std::shared_ptr<Module> g_table_mod;

int pick_vec(int n, int bytes) {
  int v = 32 / bytes;
  while (v > 1 && n % v) v /= 2;
  return v * bytes >= 4 ? v : 0;
}

// the token-row L2 prefetch before the launch-order wait
// (FUSE_ROW_PREFETCH=0 turns it off; read once)
int row_prefetch() {
  static const int on = [] {
    const char* e = getenv("FUSE_ROW_PREFETCH");
    return e && *e == '0' ? 0 : 1;
  }();
  return on;
}

// One kernel per (heads, head_dim, dtype): the token count and the start
// position come with the launch, so a serving loop whose batch changes every
// step compiles nothing after its first call.
int rope_kernel(int heads, int hd, fuse_dtype dt, RopeKernel* out) {
  auto key = std::make_tuple(heads, hd, static_cast<int>(dt));
  if (auto it = g_kernels.find(key); it != g_kernels.end()) {
    stat_hit();
    *out = it->second;
    return FUSE_OK;
  }
  RopeKernel k;
  const int bytes = dtype_bytes(dt);
  k.vec = pick_vec(hd / 2, bytes);
  k.vv = pick_vec(hd, bytes);
  k.has_vec = k.vec > 0 && k.vv > 0;
  if (!k.has_vec) k.vec = k.vv = 1;
  const int items = 2 * heads * (hd / 2 / k.vec);
  k.block = std::min(256, std::max(32, (items + 31) / 32 * 32));
  std::string src = fmt(
      "// QKV split + transpose + RoPE: heads %d, head_dim %d, %s\n"
      "constexpr int DT = %d;\nconstexpr int HEADS = %d;\nconstexpr int HD = %d;\n"
      "constexpr int HALF = %d;\nconstexpr int BLOCK = %d;\n"
      "constexpr int VEC = %d;\nconstexpr int VV = %d;\n#define FUSE_ROPE_VEC %d\n"
      "#define ROW_PREFETCH %d\n#include \"fuse/rope.cuh\"\n",
      heads, hd, dtype_name(dt), static_cast<int>(dt), heads, hd, hd / 2, k.block, k.vec, k.vv,
      k.has_vec ? 1 : 0, row_prefetch());
  if (int rc = jit_compile(src, "rope_qkv_split", &k.mod)) return rc;
  g_kernels.emplace(key, k);
  *out = k;
  return FUSE_OK;
}

// Table covering positions [0, need) on the current device; builds (or
// grows) it with a kernel on a private stream and waits for it once.
int rope_table(const DeviceInfo& d, float base, int hd, int64_t need, CUdeviceptr* out) {
  uint32_t bits;
  memcpy(&bits, &base, 4);
  Table& t = g_tables[std::make_tuple(d.ordinal, bits, hd)];
  if (t.cap >= need) {
    *out = t.ptr;
    return FUSE_OK;
  }
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  int64_t cap = std::max<int64_t>({need, 2 * t.cap, 4096});
  cap = std::min<int64_t>((cap + 4095) / 4096 * 4096, kMaxPositions);
  if (!g_table_mod) {
    if (int rc = jit_compile("#include \"fuse/rope_table.cuh\"\n", "rope_table", &g_table_mod))
      return rc;
  }
  CUfunction fn;
  if (int rc = jit_function(*g_table_mod, "rope_table_build", d, &fn)) return rc;
  CUdeviceptr p;
  CUresult r = api->MemAlloc(&p, static_cast<size_t>(cap) * hd * sizeof(float));
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuMemAlloc(rope table)");
  CUstream s;
  if ((r = api->StreamCreate(&s, CU_STREAM_NON_BLOCKING)) != CUDA_SUCCESS) {
    api->MemFree(p);
    return cuda_fail(r, "cuStreamCreate");
  }
  long long npos = cap;
  int hdi = hd;
  double b = base;
  void* args[] = {&p, &npos, &hdi, &b};
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(d.sms * 8, (cap * hd / 2 + 255) / 256));
  int rc = launch(fn, grid, 256, 0, s, args);
  if (rc == FUSE_OK && (r = api->StreamSynchronize(s)) != CUDA_SUCCESS)
    rc = cuda_fail(r, "building the RoPE table");
  api->StreamDestroy(s);
  if (rc != FUSE_OK) {
    api->MemFree(p);
    return rc;
  }
  if (t.ptr) g_retired.push_back(t.ptr);
  t.ptr = p;
  t.cap = cap;
  *out = p;
  return FUSE_OK;
}

}  // namespace
}  // namespace fuse

extern "C" int rope_qkv_split(const void* qkv, void* q, void* k, void* v, int64_t tokens,
                              int heads, int head_dim, int64_t pos0, float base, fuse_dtype dt,
                              void* stream) {
  fuse::NvtxRange nvtx_range("rope_qkv_split");
  using namespace fuse;
  if (!valid_dtype(dt)) return fail(FUSE_E_DTYPE, fmt("invalid dtype %d", dt));
  if (tokens < 0 || heads < 1 || head_dim < 2 || head_dim > 1024 || head_dim % 2)
    return fail(FUSE_E_SHAPE, "need tokens >= 0, heads >= 1, head_dim even in 2..1024");
  if (heads > (1 << 20) / head_dim) return fail(FUSE_E_SHAPE, "heads * head_dim above 2^20");
  if (tokens > 0x7fffffff) return fail(FUSE_E_SHAPE, "tokens above 2^31 - 1");
  if (pos0 < 0 || pos0 > kMaxPositions || tokens > kMaxPositions - pos0)
    return fail(FUSE_E_SHAPE, "positions must lie in [0, 2^22)");
  if (!(base > 1.f) || !std::isfinite(base)) return fail(FUSE_E_ARG, "base must be finite and > 1");
  if (tokens == 0) return FUSE_OK;
  if (!qkv || !q || !k || !v) return fail(FUSE_E_NULL, "NULL tensor pointer");
  RopeKernel kr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (int rc = rope_kernel(heads, head_dim, dt, &kr)) return rc;
  }
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  CUdeviceptr table;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (int rc = rope_table(d, base, head_dim, pos0 + tokens, &table)) return rc;
  }
  const int bytes = dtype_bytes(dt);
  bool vec = kr.has_vec;
  const uintptr_t need_qk = std::min(32, kr.vec * bytes), need_v = std::min(32, kr.vv * bytes);
  for (const void* p : {qkv, static_cast<const void*>(q), static_cast<const void*>(k),
                        static_cast<const void*>(v)})
    vec = vec && reinterpret_cast<uintptr_t>(p) % need_qk == 0 &&
          reinterpret_cast<uintptr_t>(p) % need_v == 0;
  CUfunction fn;
  if (int rc = jit_function(*kr.mod, vec ? "rope_vec" : "rope_scalar", d, &fn)) return rc;
  long long p0 = pos0, nt = tokens;
  void* args[] = {&qkv, &q, &k, &v, &table, &p0, &nt};
  return launch(fn, static_cast<unsigned>(tokens), static_cast<unsigned>(kr.block), 0, stream,
                args);
}
