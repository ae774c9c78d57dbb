// rmsnorm.cpp -- residual add + RMSNorm + cast entry point.
//
// "TeleTron" section 3.3 fuses the residual add into the normalisation with a
// per-row reduction accumulated in higher precision; section 4.2 gives the
// scale rsqrt(sum_sq / K + 1e-6) and the block-per-row layout with vector
// loads of 4-8 elements per thread.  Here the row length, vector width and
// block size are baked into the generated source; each row is one CTA, x and
// residual are read once with 32-byte loads, and both outputs are written
// once.
#include <algorithm>
#include <cstdlib>
#include <map>

#include "internal.h"

namespace fuse {
namespace {

struct RmsKernel {
  std::shared_ptr<Module> mod;
  int block = 256, vec = 1;
  bool has_vec = false;
};

std::mutex g_mu;
std::map<std::pair<int64_t, int>, RmsKernel> g_kernels;

// the first-row L2 prefetch before the launch-order wait (FUSE_ROW_PREFETCH=0
// turns it off; read once)
int row_prefetch() {
  static const int on = [] {
    const char* e = getenv("FUSE_ROW_PREFETCH");
    return e && *e == '0' ? 0 : 1;
  }();
  return on;
}

int rms_kernel(int64_t hidden, fuse_dtype dt, RmsKernel* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(hidden, static_cast<int>(dt));
  if (auto it = g_kernels.find(key); it != g_kernels.end()) {
    stat_hit();
    *out = it->second;
    return FUSE_OK;
  }
  RmsKernel k;
  const int bytes = dtype_bytes(dt);
  int vec = 32 / bytes;
  while (vec > 1 && hidden % vec) vec /= 2;
  k.has_vec = vec * bytes >= 4;
  k.vec = k.has_vec ? vec : 1;
  const int64_t nvr = hidden / k.vec;
  k.block = static_cast<int>(std::min<int64_t>(1024, std::max<int64_t>(32, (nvr + 31) / 32 * 32)));
  const int64_t r = (nvr + k.block - 1) / k.block;
  std::string src = fmt(
      "// residual add + RMSNorm + cast, hidden %lld, %s\n"
      "constexpr int DT = %d;\nconstexpr int HIDDEN = %lld;\nconstexpr int BLOCK = %d;\n"
      "constexpr int VEC = %d;\nconstexpr int R = %lld;\n#define FUSE_RMS_VEC %d\n"
      "#define ROW_PREFETCH %d\n#include \"fuse/rmsnorm.cuh\"\n",
      (long long)hidden, dtype_name(dt), static_cast<int>(dt), (long long)hidden, k.block, k.vec,
      (long long)r, k.has_vec ? 1 : 0, row_prefetch());
  if (int rc = jit_compile(src, "rmsnorm_residual", &k.mod)) return rc;
  g_kernels.emplace(key, k);
  *out = k;
  return FUSE_OK;
}

}  // namespace
}  // namespace fuse

extern "C" int rmsnorm_residual(const void* x, const void* residual, const void* weight, void* out,
                                void* residual_out, int64_t rows, int64_t hidden, float eps,
                                fuse_dtype dt, void* stream) {
  fuse::NvtxRange nvtx_range("rmsnorm_residual");
  using namespace fuse;
  if (!valid_dtype(dt)) return fail(FUSE_E_DTYPE, fmt("invalid dtype %d", dt));
  if (rows < 0) return fail(FUSE_E_SHAPE, "rows < 0");
  if (hidden < 1 || hidden > 65536) return fail(FUSE_E_SHAPE, "hidden outside 1..65536");
  if (!(eps >= 0.f)) return fail(FUSE_E_ARG, "eps must be >= 0");
  if (rows == 0) return FUSE_OK;
  if (!x || !residual || !weight || !out || !residual_out)
    return fail(FUSE_E_NULL, "NULL tensor pointer");
  RmsKernel k;
  if (int rc = rms_kernel(hidden, dt, &k)) return rc;
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  const uintptr_t need = static_cast<uintptr_t>(std::min(32, k.vec * dtype_bytes(dt)));
  bool vec = k.has_vec;
  for (const void* p : {x, residual, weight, static_cast<const void*>(out),
                        static_cast<const void*>(residual_out)})
    vec = vec && reinterpret_cast<uintptr_t>(p) % need == 0;
  CUfunction fn;
  if (int rc = jit_function(*k.mod, vec ? "rmsnorm_vec" : "rmsnorm_scalar", d, &fn)) return rc;
  long long nrows = rows;
  void* args[] = {&x, &residual, &weight, &out, &residual_out, &nrows, &eps};
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(rows, 0x7fffffff));
  return launch(fn, grid, static_cast<unsigned>(k.block), 0, stream, args);
}
