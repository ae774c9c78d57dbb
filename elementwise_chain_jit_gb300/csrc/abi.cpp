// abi.cpp -- diagnostics entry points and ChannelShuffle.
//
// ChannelShuffle ("算子与运行时", section 2) on contiguous NCHW is a
// permutation of whole H*W planes.  It runs through the chain engine as the
// spec "shuffle:G" with no ops: a bit copy whose input index is the shuffle's
// gather, with 16/32-byte coalesced accesses on both sides.  The handle is a
// shape bucket over the batch dimension N (one compile per (C, H, W, G,
// dtype), N passed with the launch), so a batch that changes from call to
// call compiles nothing after the first.  The pages' own
// remedy for the slow reshape/transpose (shared-memory reordering before
// coalesced writes, section 2.1) is not needed on NCHW, where each plane is
// already contiguous in both layouts.
#include <map>
#include <tuple>

#include "internal.h"

namespace fuse {
void read_stats(int64_t* c, int64_t* h, int64_t* l, double* ms);
int chain_compile(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dt,
                  fuse_chain** out, bool bucket);
int chain_launch(fuse_chain* h, const void* const* inputs, int n_in, void* output, void* stream,
                 int64_t rows);

namespace {
std::mutex g_shuffle_mu;
// (c, h, w, groups, dtype, 64-bit indices) -> bucket handle
std::map<std::tuple<int64_t, int64_t, int64_t, int, int, bool>, fuse_chain*> g_shuffle;
constexpr int64_t kMaxShuffleElems = int64_t(1) << 40;  // the chain engine's limit
}  // namespace
}  // namespace fuse

extern "C" {

const char* fuse_last_error(void) { return fuse::last_error_cstr(); }

int fuse_stats(int64_t* compiles, int64_t* cache_hits, int64_t* launches, double* compile_ms) {
  fuse::read_stats(compiles, cache_hits, launches, compile_ms);
  return FUSE_OK;
}

int fuse_device_sms(int* sms) {
  if (!sms) return fuse::fail(FUSE_E_NULL, "sms is NULL");
  *sms = fuse::default_sms();
  return FUSE_OK;
}

int channel_shuffle(const void* in, void* out, int64_t n, int64_t c, int64_t h, int64_t w,
                    int groups, fuse_dtype dt, void* stream) {
  fuse::NvtxRange nvtx_range("channel_shuffle");
  using namespace fuse;
  if (!valid_dtype(dt)) return fail(FUSE_E_DTYPE, fmt("invalid dtype %d", dt));
  if (n < 0 || c < 0 || h < 0 || w < 0) return fail(FUSE_E_SHAPE, "negative dimension");
  if (groups <= 0) return fail(FUSE_E_ARG, "groups must be positive");
  if (c % groups) return fail(FUSE_E_SHAPE, "channels not divisible by groups");
  if (n == 0 || c == 0 || h == 0 || w == 0) return FUSE_OK;
  // (no product is formed before it is known to stay below 2^40)
  if (c > kMaxShuffleElems / h || c * h > kMaxShuffleElems / w ||
      n > kMaxShuffleElems / (c * h * w))
    return fail(FUSE_E_SHAPE, "more than 2^40 elements");
  if (!in || !out) return fail(FUSE_E_NULL, "NULL tensor pointer");
  if (in == out) return fail(FUSE_E_ARG, "channel_shuffle cannot run in place");
  // the batch bucket: every N whose elements stay below 2^31 shares one
  // kernel with 32-bit indices; larger N take a second one with 64-bit
  // indices, up to the engine's 2^40 elements
  const int64_t plane = c * h * w;
  const int64_t n32 = ((int64_t(1) << 31) - 1) / plane;
  const bool wide = n > n32;
  const int64_t cap = wide ? kMaxShuffleElems / plane : n32;
  fuse_chain* hnd = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_shuffle_mu);
    auto key = std::make_tuple(c, h, w, groups, static_cast<int>(dt), wide);
    auto it = g_shuffle.find(key);
    if (it != g_shuffle.end()) {
      hnd = it->second;
      stat_hit();
    } else {
      int64_t shape[4] = {cap, c, h, w};
      std::string spec = fmt("shuffle:%d", groups);
      if (int rc = chain_compile(spec.c_str(), shape, 4, dt, &hnd, true)) return rc;
      g_shuffle.emplace(key, hnd);
    }
  }
  const void* ins[1] = {in};
  return chain_launch(hnd, ins, 1, out, stream, n);
}

}  // extern "C"

// ------------------------------------------------------------------ self test

namespace {
// one warp waits on an mbarrier that nothing arrives at, through the same
// bounded wait as every wait in the library's kernels, and records code 1
const char* kSelftestSource =
    "#include \"fuse/sync.cuh\"\n"
    "extern \"C\" __global__ void bounded_wait_selftest(unsigned spins, int* err) {\n"
    "  __shared__ unsigned long long bar;\n"
    "  const u32 b = smem_u32(&bar);\n"
    "  if (threadIdx.x == 0) mbar_init(b, 1);\n"
    "  __syncthreads();\n"
    "  const bool ok = __all_sync(0xffffffffu, mbar_wait(b, 0, spins));\n"
    "  if (!ok && threadIdx.x == 0) atomicExch(err, 1);\n"
    "}\n";
std::mutex g_selftest_mu;
std::shared_ptr<fuse::Module> g_selftest;
}  // namespace

extern "C" int fuse_selftest_bounded_wait(int64_t spins, void* stream) {
  using namespace fuse;
  if (spins < 1 || spins > (int64_t(1) << 30)) return fail(FUSE_E_ARG, "spins outside 1..2^30");
  std::shared_ptr<Module> mod;
  {
    std::lock_guard<std::mutex> lk(g_selftest_mu);
    if (!g_selftest)
      if (int rc = jit_compile(kSelftestSource, "bounded_wait_selftest", &g_selftest)) return rc;
    mod = g_selftest;
  }
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  CUfunction fn;
  if (int rc = jit_function(*mod, "bounded_wait_selftest", d, &fn)) return rc;
  CUdeviceptr err;
  if (int rc = device_error_word(d.ordinal, &err)) return rc;
  unsigned sp = static_cast<unsigned>(spins);
  void* args[] = {&sp, &err};
  return launch(fn, 1, 32, 0, stream, args);
}
