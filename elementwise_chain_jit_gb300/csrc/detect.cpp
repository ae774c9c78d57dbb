// detect.cpp -- detection-head decode entry point.
//
// "DeepJIT ... 串行小核墙" section 1.1 describes the tail of a detection head
// (sigmoid, exp, mul, add, slice, concat, cast) split into a hundred small
// kernels after the backbone; section 5.2 runs the fused replacement on the
// same stream right after the engine, whose output is NCHW fp32.  Here all
// scales, anchors and channels decode in one launch: the per-scale shapes,
// strides, anchors and output row offsets are baked into the generated
// source, and the channel -> last transpose goes through shared memory so
// that both the reads (along cells) and the writes (whole output rows) are
// coalesced.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <sstream>

#include "internal.h"

namespace fuse {
namespace {

struct DetectKernel {
  std::shared_ptr<Module> mod;
  unsigned grid = 0;
  int block = 256;
};

std::mutex g_mu;
std::map<std::string, DetectKernel> g_kernels;

std::string key_of(const int* hw, const float* strides, const float* anchors, int ns, int na,
                   int no, fuse_dtype dt) {
  std::string k = fmt("%d/%d/%d/%d/", ns, na, no, static_cast<int>(dt));
  k.append(reinterpret_cast<const char*>(hw), sizeof(int) * 2 * ns);
  k.append(reinterpret_cast<const char*>(strides), sizeof(float) * ns);
  k.append(reinterpret_cast<const char*>(anchors), sizeof(float) * 2 * ns * na);
  return k;
}

int detect_kernel(const int* hw, const float* strides, const float* anchors, int ns, int na, int no,
                  fuse_dtype dt, DetectKernel* out) {
  std::string key = key_of(hw, strides, anchors, ns, na, no, dt);
  if (auto it = g_kernels.find(key); it != g_kernels.end()) {
    stat_hit();
    *out = it->second;
    return FUSE_OK;
  }
  DetectKernel k;
  // Cells per tile: up to 128, a multiple of 8, with the tile of tc * no
  // floats inside 48 KB.  Threads per CTA: the fewest that still give no
  // thread more (channel, 8-cell) items than 512 threads would, so the items
  // spread evenly (1360 items of the 85-output head: 454 threads, 3 each).
  // Measured on GB300 for the 3-scale 85-output head, launched back to back:
  // 5.53 us against 5.83 for 64-cell tiles of 256 threads (three runs each);
  // 340 threads of exactly 2 items each took 6.5 us.  FUSE_DETECT_TC and
  // FUSE_DETECT_BLOCK override.
  int tc = std::min(128, (12288 / no) / 8 * 8);
  if (const char* e = getenv("FUSE_DETECT_TC"); e && *e) {
    int v = atoi(e) / 8 * 8;
    if (v >= 8 && v * no * 4 <= 49152) tc = v;
  }
  {
    const int items = no * (tc / 8);
    const int per = (items + 511) / 512;
    k.block = std::max(32, (items + per - 1) / per);
  }
  if (const char* e = getenv("FUSE_DETECT_BLOCK"); e && *e) {
    int v = atoi(e);
    if (v >= 32 && v <= 1024) k.block = v;
  }
  std::ostringstream s;
  s << "// detection-head decode: " << ns << " scales, " << na << " anchors, " << no
    << " outputs per anchor, " << dtype_name(dt) << " in, f32 out\n";
  s << "constexpr int DT = " << dt << ";\nconstexpr int NA = " << na << ";\nconstexpr int NO = " << no
    << ";\nconstexpr int TC = " << tc << ";\nconstexpr int BLOCK = " << k.block << ";\n";
  s << "#include \"fuse/detect.cuh\"\n\n";
  s << "template <bool VEC>\n__device__ __forceinline__ void dispatch(const Feats& f, float* out, "
       "float* tile) {\n  const int b = blockIdx.x;\n";
  int64_t cta = 0, row0 = 0;
  for (int sc = 0; sc < ns; ++sc) {
    const int H = hw[2 * sc], W = hw[2 * sc + 1];
    const int64_t HW = int64_t(H) * W;
    const int64_t tiles = (HW + tc - 1) / tc;
    const int64_t end = cta + tiles * na;
    s << "  if (b < " << end << ") {  // scale " << sc << ": " << H << " x " << W << ", stride "
      << strides[sc] << ", rows from " << row0 << "\n";
    s << "    const int r = b - " << cta << ", a = r / " << tiles << ", c0 = (r % " << tiles
      << ") * TC;\n    float aw = 0.f, ah = 0.f;\n    switch (a) {\n";
    for (int a = 0; a < na; ++a)
      s << "      case " << a << ": aw = " << hex_float(anchors[(sc * na + a) * 2])
        << "; ah = " << hex_float(anchors[(sc * na + a) * 2 + 1]) << "; break;\n";
    s << "    }\n    tile_work<VEC, " << H << ", " << W << ">(f.p[" << sc << "], out, a, c0, "
      << hex_float(strides[sc]) << ", aw, ah, " << row0 << "LL + (long long)a * " << HW
      << " + c0, tile);\n    return;\n  }\n";
    cta = end;
    row0 += HW * na;
  }
  s << "}\n\n";
  for (const char* v : {"vec", "scalar"})
    s << "extern \"C\" __global__ void __launch_bounds__(BLOCK) detect_" << v
      << "(const Feats f, float* out) {\n  pdl_enter();\n  __shared__ __align__(16) float tile[TC * NO];\n  dispatch<"
      << (v[0] == 'v' ? "true" : "false") << ">(f, out, tile);\n}\n";
  if (cta > 0x7fffffff) return fail(FUSE_E_SHAPE, "too many tiles");
  k.grid = static_cast<unsigned>(cta);
  if (int rc = jit_compile(s.str(), "detect_decode", &k.mod)) return rc;
  g_kernels.emplace(key, k);
  *out = k;
  return FUSE_OK;
}

}  // namespace
}  // namespace fuse

extern "C" int detect_decode(const void* const* feats, const int* hw, const float* strides,
                             const float* anchors, int nscales, int na, int no, fuse_dtype in_dt,
                             void* out, void* stream) {
  fuse::NvtxRange nvtx_range("detect_decode");
  using namespace fuse;
  if (!valid_dtype(in_dt)) return fail(FUSE_E_DTYPE, fmt("invalid dtype %d", in_dt));
  if (nscales < 1 || nscales > 8) return fail(FUSE_E_SHAPE, "nscales outside 1..8");
  if (na < 1 || na > 16) return fail(FUSE_E_SHAPE, "na outside 1..16");
  if (no < 5 || no > 1024) return fail(FUSE_E_SHAPE, "no outside 5..1024");
  if (!hw || !strides || !anchors) return fail(FUSE_E_NULL, "NULL hw/strides/anchors");
  for (int s = 0; s < nscales; ++s) {
    if (hw[2 * s] < 1 || hw[2 * s + 1] < 1 || int64_t(hw[2 * s]) * hw[2 * s + 1] > (1 << 24))
      return fail(FUSE_E_SHAPE, fmt("scale %d: H and W must be >= 1 with H*W <= 2^24", s));
    if (!std::isfinite(strides[s])) return fail(FUSE_E_ARG, "non-finite stride");
  }
  for (int i = 0; i < 2 * nscales * na; ++i)
    if (!std::isfinite(anchors[i])) return fail(FUSE_E_ARG, "non-finite anchor");
  if (!feats || !out) return fail(FUSE_E_NULL, "NULL feats or out");
  bool vec = fuse::aligned16(out);
  const uintptr_t need = static_cast<uintptr_t>(std::min(32, 8 * dtype_bytes(in_dt)));
  for (int s = 0; s < nscales; ++s) {
    if (!feats[s]) return fail(FUSE_E_NULL, fmt("feats[%d] is NULL", s));
    vec = vec && reinterpret_cast<uintptr_t>(feats[s]) % need == 0;
  }
  DetectKernel k;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (int rc = detect_kernel(hw, strides, anchors, nscales, na, no, in_dt, &k)) return rc;
  }
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  CUfunction fn;
  if (int rc = jit_function(*k.mod, vec ? "detect_vec" : "detect_scalar", d, &fn)) return rc;
  struct {
    const void* p[8];
  } f{};
  for (int s = 0; s < nscales; ++s) f.p[s] = feats[s];
  void* args[] = {&f, &out};
  return launch(fn, k.grid, static_cast<unsigned>(k.block), 0, stream, args);
}
