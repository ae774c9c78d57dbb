// layernorm.cpp -- residual add + LayerNorm + cast entry point.
//
// The LayerNorm of "DeepJIT ... 串行小核墙" section 4.3 (one block per row,
// statistics reduced in the block, normalisation in the same pass), with the
// page's suggested upgrade (warp-shuffle reductions) and an optional fused
// residual add.  Row length, vector width, block size and the presence of
// residual / gamma / beta are baked into the generated source.
#include <algorithm>
#include <map>
#include <tuple>

#include <cstdlib>

#include "internal.h"

namespace fuse {
namespace {

struct LnKernel {
  std::shared_ptr<Module> mod;
  int block = 256, vec = 1;
  bool has_vec = false;
};

std::mutex g_mu;
std::map<std::tuple<int64_t, int, int>, LnKernel> g_kernels;

// Registers a thread may use.  With one vector a thread (rows up to 16384
// bf16 elements) the compiler left to itself takes 72 (3 CTAs of 256 threads
// per SM); capped at 48 (5 CTAs) it holds the row's values without spilling.
// Measured on GB300 at hidden 4096 bf16: 100.1 us with 72 registers, 93.0
// with 64, 90.9 with 48, 90.9 with 40 (spilling), 94.2 with 36.  Longer rows
// keep several vectors a thread in 1024-thread blocks and get the most those
// blocks allow (64).  FUSE_LN_MAX_REGS overrides.
int max_regs(int block, int64_t r) {
  const int limit = std::min(255, 65536 / block / 8 * 8);
  const char* e = getenv("FUSE_LN_MAX_REGS");
  const int want = e && *e ? atoi(e) : (r == 1 ? 48 : limit);
  return std::min(limit, std::max(24, want));
}

// the first-row L2 prefetch before the launch-order wait (FUSE_ROW_PREFETCH=0
// turns it off; read once)
int row_prefetch() {
  static const int on = [] {
    const char* e = getenv("FUSE_ROW_PREFETCH");
    return e && *e == '0' ? 0 : 1;
  }();
  return on;
}

int ln_kernel(int64_t hidden, fuse_dtype dt, int flags, LnKernel* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(hidden, static_cast<int>(dt), flags);
  if (auto it = g_kernels.find(key); it != g_kernels.end()) {
    stat_hit();
    *out = it->second;
    return FUSE_OK;
  }
  LnKernel k;
  const int bytes = dtype_bytes(dt);
  int vec = 32 / bytes;
  while (vec > 1 && hidden % vec) vec /= 2;
  k.has_vec = vec * bytes >= 4;
  k.vec = k.has_vec ? vec : 1;
  const int64_t nvr = hidden / k.vec;
  k.block = static_cast<int>(std::min<int64_t>(1024, std::max<int64_t>(32, (nvr + 31) / 32 * 32)));
  const int64_t r = (nvr + k.block - 1) / k.block;
  std::string src = fmt(
      "// residual add + LayerNorm + cast, hidden %lld, %s\n"
      "constexpr int DT = %d;\nconstexpr int HIDDEN = %lld;\nconstexpr int BLOCK = %d;\n"
      "constexpr int VEC = %d;\nconstexpr int R = %lld;\n"
      "constexpr bool HAS_RES = %s, HAS_GAMMA = %s, HAS_BETA = %s;\n#define FUSE_LN_VEC %d\n"
      "#define LN_MAX_REGS %d\n#define ROW_PREFETCH %d\n#include \"fuse/layernorm.cuh\"\n",
      (long long)hidden, dtype_name(dt), static_cast<int>(dt), (long long)hidden, k.block, k.vec,
      (long long)r, (flags & 1) ? "true" : "false", (flags & 2) ? "true" : "false",
      (flags & 4) ? "true" : "false", k.has_vec ? 1 : 0, max_regs(k.block, r), row_prefetch());
  if (int rc = jit_compile(src, "layernorm_residual", &k.mod)) return rc;
  g_kernels.emplace(key, k);
  *out = k;
  return FUSE_OK;
}

}  // namespace
}  // namespace fuse

extern "C" int layernorm_residual(const void* x, const void* residual, const void* gamma,
                                  const void* beta, void* out, void* residual_out, int64_t rows,
                                  int64_t hidden, float eps, fuse_dtype dt, void* stream) {
  fuse::NvtxRange nvtx_range("layernorm_residual");
  using namespace fuse;
  if (!valid_dtype(dt)) return fail(FUSE_E_DTYPE, fmt("invalid dtype %d", dt));
  if (rows < 0) return fail(FUSE_E_SHAPE, "rows < 0");
  if (hidden < 1 || hidden > 65536) return fail(FUSE_E_SHAPE, "hidden outside 1..65536");
  if (!(eps >= 0.f)) return fail(FUSE_E_ARG, "eps must be >= 0");
  if ((residual == nullptr) != (residual_out == nullptr))
    return fail(FUSE_E_ARG, "residual and residual_out must both be given or both be NULL");
  if (rows == 0) return FUSE_OK;
  if (!x || !out) return fail(FUSE_E_NULL, "NULL x or out");
  const int flags = (residual ? 1 : 0) | (gamma ? 2 : 0) | (beta ? 4 : 0);
  LnKernel k;
  if (int rc = ln_kernel(hidden, dt, flags, &k)) return rc;
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  const uintptr_t need = static_cast<uintptr_t>(std::min(32, k.vec * dtype_bytes(dt)));
  bool vec = k.has_vec;
  for (const void* p : {x, residual, gamma, beta, static_cast<const void*>(out),
                        static_cast<const void*>(residual_out)})
    vec = vec && reinterpret_cast<uintptr_t>(p) % need == 0;  // NULL is aligned
  CUfunction fn;
  if (int rc = jit_function(*k.mod, vec ? "layernorm_vec" : "layernorm_scalar", d, &fn)) return rc;
  long long nrows = rows;
  void* args[] = {&x, &residual, &gamma, &beta, &out, &residual_out, &nrows, &eps};
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(rows, 0x7fffffff));
  return launch(fn, grid, static_cast<unsigned>(k.block), 0, stream, args);
}
