// rms_linear.cpp -- RMSNorm -> Linear -> scale entry point (tcgen05).
//
// "TeleTron" section 4.2 ("RMSNorm + Linear + scale" fused): the RMSNorm
// factor of each row is computed inside the GEMM's tile loop and applied in
// the epilogue, and the contraction runs on the tensor cores (tcgen05.mma with
// TMEM accumulators, operands staged by TMA).  gamma is folded into the
// weight (w' = dt(w * gamma)): once by the caller through rmsnorm_linear_fold,
// or, when gamma is passed, into a stream-ordered scratch copy for the call.
// The kernel is generated per (K, N, dtype, bias) and compiled by NVRTC for
// sm_103a like every other kernel of the library.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <map>
#include <tuple>
#include <vector>

#include "internal.h"

namespace fuse {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kSmemOptinSm103 = 227 * 1024;  // shared memory a CTA may opt in to
// the persistent CTA-pair kernel: stages of x (128 x 64) and half a w tile
// (128 x 64) per CTA, accumulator buffers of 256 TMEM columns, runs of
// column blocks that share one computation of the row statistics, and a
// 32 x 64 output block (128-byte rows, 128-byte swizzle) per epilogue warp
// staged for the TMA store
constexpr int kPairStages = 6, kPairAcc = 2, kPairRun = 2, kOutRows = 32, kOutCols = 64;
// its dynamic shared memory: 1 KB alignment slack, the stages, rstd[2][128],
// the epilogue's staging blocks, the mbarriers and the TMEM address slot
constexpr int kPairSmem = 1024 + kPairStages * (kBM + kBN / 2) * kBK * 2 + 2 * 128 * 4 +
                          4 * 2 * kOutRows * kOutCols * 2 + 8 * (3 * kPairStages + 8) + 16;
static_assert(kPairSmem <= kSmemOptinSm103, "the persistent kernel's layout must fit a CTA");

std::mutex g_mu;
std::map<std::tuple<int64_t, int64_t, int, int>, std::shared_ptr<Module>> g_kernels;

int rl_module(int64_t K, int64_t N, fuse_dtype dt, bool has_bias, std::shared_ptr<Module>* out) {
  auto key = std::make_tuple(K, N, static_cast<int>(dt), has_bias ? 1 : 0);
  if (auto it = g_kernels.find(key); it != g_kernels.end()) {
    stat_hit();
    *out = it->second;
    return FUSE_OK;
  }
  std::string src = fmt(
      "// RMSNorm -> Linear -> scale, K %lld, N %lld, %s, tcgen05\n"
      "constexpr int DT = %d;\nconstexpr long long KDIM = %lldLL;\nconstexpr long long NDIM = %lldLL;\n"
      "constexpr int PSTAGES = %d, PAIR_NACC = %d, PAIR_RUN = %d;\n"
      "constexpr bool HAS_BIAS = %s;\n"
      "#include \"fuse/rms_linear.cuh\"\n",
      (long long)K, (long long)N, dtype_name(dt), static_cast<int>(dt), (long long)K, (long long)N,
      kPairStages, kPairAcc, kPairRun, has_bias ? "true" : "false");
  std::shared_ptr<Module> mod;
  if (int rc = jit_compile(src, "rmsnorm_linear", &mod)) return rc;
  g_kernels.emplace(key, mod);
  *out = mod;
  return FUSE_OK;
}

int encode_kmajor(const DriverApi* api, CUtensorMap* map, const void* ptr, fuse_dtype dt,
                  int64_t rows, int64_t K, uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t elem[2] = {1, 1};
  CUresult r = api->TensorMapEncodeTiled(
      map, dt == FUSE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
      const_cast<void*>(ptr), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuTensorMapEncodeTiled");
  return FUSE_OK;
}

// The output [M, N] as the destination of 32-row x 64-column TMA stores from
// 128-byte swizzled staging blocks.
int encode_out(const DriverApi* api, CUtensorMap* map, void* ptr, fuse_dtype dt, int64_t M,
               int64_t N) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
  cuuint32_t box[2] = {kOutCols, kOutRows};
  cuuint32_t elem[2] = {1, 1};
  CUresult r = api->TensorMapEncodeTiled(
      map, dt == FUSE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
      ptr, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuTensorMapEncodeTiled(out)");
  return FUSE_OK;
}

// The kernel deals runs of column blocks to its clusters round-robin: the
// first mp_long row pairs in runs of 2 * kPairRun blocks, the rest in runs of
// kPairRun.  A long run computes the row statistics once for twice the
// blocks, but coarse runs can leave the last clusters' loads uneven.  Picks
// the largest mp_long whose most loaded cluster has no more blocks than with
// short runs only (every value up to 512 row pairs, 64 evenly spaced ones
// beyond), cached per shape; also returns the number of runs.
int64_t pick_mp_long(int64_t m_pairs, int64_t nt, int64_t clusters, int64_t* runs_out) {
  static std::mutex mu;
  static std::map<std::tuple<int64_t, int64_t, int64_t>, std::pair<int64_t, int64_t>> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(m_pairs, nt, clusters);
  if (auto it = cache.find(key); it != cache.end()) {
    *runs_out = it->second.second;
    return it->second.first;
  }
  const int64_t c = std::max<int64_t>(1, clusters), run_s = kPairRun, run_l = 2 * kPairRun;
  std::vector<int64_t> load(static_cast<size_t>(c));
  auto simulate = [&](int64_t mp_long, int64_t* nruns) {
    std::fill(load.begin(), load.end(), 0);
    int64_t idx = 0;
    for (int64_t mp = 0; mp < m_pairs; ++mp) {
      const int64_t run = mp < mp_long ? run_l : run_s;
      for (int64_t n = 0; n < nt; n += run) load[static_cast<size_t>(idx++ % c)] += std::min(run, nt - n);
    }
    *nruns = idx;
    return *std::max_element(load.begin(), load.end());
  };
  int64_t runs0;
  const int64_t bound = simulate(0, &runs0);
  int64_t best = 0, best_runs = runs0;
  const int64_t step = m_pairs <= 512 ? 1 : (m_pairs + 63) / 64;
  for (int64_t mp = m_pairs; mp > 0; mp = mp > step ? mp - step : 0) {
    int64_t nruns;
    if (simulate(mp, &nruns) <= bound) {
      best = mp;
      best_runs = nruns;
      break;
    }
  }
  cache.emplace(key, std::make_pair(best, best_runs));
  *runs_out = best_runs;
  return best;
}

// How many 2-CTA clusters of the persistent kernel fit on the device at
// once (some SMs may be left over when a GPC has an odd number of them).
int max_clusters(const DriverApi* api, CUfunction fn, int smem, int* out) {
  static std::map<CUfunction, int> cache;
  if (auto it = cache.find(fn); it != cache.end()) {
    *out = it->second;
    return FUSE_OK;
  }
  CUlaunchConfig cfg = {};
  cfg.gridDimX = 2;
  cfg.gridDimY = cfg.gridDimZ = 1;
  cfg.blockDimX = 320;
  cfg.blockDimY = cfg.blockDimZ = 1;
  cfg.sharedMemBytes = static_cast<unsigned>(smem);
  int n = 0;
  CUresult r = api->OccupancyMaxActiveClusters(&n, fn, &cfg);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuOccupancyMaxActiveClusters");
  if (n < 1) return fail(FUSE_E_CUDA, "no 2-CTA cluster of rmsnorm_linear fits on this device");
  cache.emplace(fn, n);
  *out = n;
  return FUSE_OK;
}

// A device's pool for the folded-weight scratch of calls that pass gamma:
// the library's own (the process's default pool keeps its settings), with no
// release threshold, so a scratch block stays mapped for the next call
// instead of being unmapped at every synchronisation.  It holds at most what
// the calls that overlap on the GPU needed at once.
int scratch_pool(const DriverApi* api, int device, CUmemoryPool* out) {
  static std::mutex mu;
  static CUmemoryPool pools[64] = {};
  if (device < 0 || device >= 64) return fail(FUSE_E_ARG, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(mu);
  if (!pools[device]) {
    CUmemPoolProps props = {};
    props.allocType = CU_MEM_ALLOCATION_TYPE_PINNED;
    props.handleTypes = CU_MEM_HANDLE_TYPE_NONE;
    props.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    props.location.id = device;
    CUmemoryPool pool;
    CUresult r = api->MemPoolCreate(&pool, &props);
    if (r != CUDA_SUCCESS) return cuda_fail(r, "cuMemPoolCreate");
    cuuint64_t keep = ~cuuint64_t(0);
    r = api->MemPoolSetAttribute(pool, CU_MEMPOOL_ATTR_RELEASE_THRESHOLD, &keep);
    if (r != CUDA_SUCCESS) return cuda_fail(r, "cuMemPoolSetAttribute");
    pools[device] = pool;
  }
  *out = pools[device];
  return FUSE_OK;
}

// The persistent CTA-pair kernel on a weight with gamma already folded in.
int launch_folded(const void* x, const void* w, const void* bias, void* out, int64_t M, int64_t N,
                  int64_t K, float eps, float scale, fuse_dtype dt, void* stream) {
  std::shared_ptr<Module> mod;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (int rc = rl_module(K, N, dt, bias != nullptr, &mod)) return rc;
  }
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  CUfunction fn;
  if (int rc = jit_function(*mod, "rms_linear_persistent", d, &fn)) return rc;
  CUdeviceptr err;
  if (int rc = device_error_word(d.ordinal, &err)) return rc;
  CUresult r = api->FuncSetAttribute(fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, kPairSmem);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuFuncSetAttribute(shared memory)");
  int clusters = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (int rc = max_clusters(api, fn, kPairSmem, &clusters)) return rc;
  }
  // x in 128-row tiles; each CTA of a pair loads one 128-row half of a w tile
  alignas(64) CUtensorMap mx, mw, mo;
  if (int rc = encode_kmajor(api, &mx, x, dt, M, K, kBM)) return rc;
  if (int rc = encode_kmajor(api, &mw, w, dt, N, K, kBN / 2)) return rc;
  if (int rc = encode_out(api, &mo, out, dt, M, N)) return rc;
  const int64_t m_tiles64 = (M + kBM - 1) / kBM, n_tiles = (N + kBN - 1) / kBN;
  int m_tiles = static_cast<int>(m_tiles64);
  int64_t runs;
  int mp_long = static_cast<int>(pick_mp_long((m_tiles64 + 1) / 2, n_tiles, clusters, &runs));
  const unsigned grid = 2u * static_cast<unsigned>(std::min<int64_t>(runs, clusters));
  void* args[] = {&mx, &mw, &mo, &bias, &m_tiles, &eps, &scale, &err, &mp_long};
  // programmatic dependent launch, as for the other kernels (FUSE_PDL=0 off):
  // the kernel's set-up overlaps the previous kernel, which it waits for
  // before its first global access
  static const bool pdl = [] {
    const char* e = getenv("FUSE_PDL");
    return !(e && *e == '0');
  }();
  CUlaunchAttribute attr = {};
  attr.id = CU_LAUNCH_ATTRIBUTE_PROGRAMMATIC_STREAM_SERIALIZATION;
  attr.value.programmaticStreamSerializationAllowed = 1;
  CUlaunchConfig cfg = {};
  cfg.gridDimX = grid;
  cfg.gridDimY = cfg.gridDimZ = 1;
  cfg.blockDimX = 320;
  cfg.blockDimY = cfg.blockDimZ = 1;
  cfg.sharedMemBytes = kPairSmem;
  cfg.hStream = reinterpret_cast<CUstream>(stream);
  cfg.attrs = pdl ? &attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  r = api->LaunchKernelEx(&cfg, fn, args, nullptr);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuLaunchKernelEx(rmsnorm_linear)");
  stat_launch();
  return FUSE_OK;
}

}  // namespace
}  // namespace fuse

extern "C" int rmsnorm_linear(const void* x, const void* gamma, const void* w, const void* bias,
                              void* out, int64_t M, int64_t N, int64_t K, float eps, float scale,
                              fuse_dtype dt, void* stream) {
  fuse::NvtxRange nvtx_range("rmsnorm_linear");
  using namespace fuse;
  if (dt != FUSE_F16 && dt != FUSE_BF16)
    return fail(FUSE_E_DTYPE, "rmsnorm_linear runs on the tensor cores: f16 or bf16 only");
  if (M < 0 || N < 0 || K < 0) return fail(FUSE_E_SHAPE, "negative size");
  // TMA takes the ragged edges: rows and columns past the tensors load as
  // zeros and are clipped on store; its row strides must be multiples of 16
  // bytes
  if (N % 8 || K % 8 || K == 0)
    return fail(FUSE_E_SHAPE, fmt("need N %% 8 == 0, K %% 8 == 0 and K > 0 (got N %lld, K %lld)",
                                  (long long)N, (long long)K));
  const int64_t m_tiles = (M + kBM - 1) / kBM, n_tiles = (N + kBN - 1) / kBN;
  // TMA tile coordinates are 32-bit
  if (K > (int64_t(1) << 20) || M > INT32_MAX - kBM || m_tiles * n_tiles > INT32_MAX)
    return fail(FUSE_E_SHAPE, "M, K or the tile count too large");
  if (!(eps >= 0.f) || !std::isfinite(scale)) return fail(FUSE_E_ARG, "bad eps or scale");
  if (M == 0 || N == 0) return FUSE_OK;
  if (!x || !w || !out) return fail(FUSE_E_NULL, "NULL tensor pointer");
  for (const void* p : {x, gamma, w, bias, static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(p) % 16)
      return fail(FUSE_E_ARG, "rmsnorm_linear needs 16-byte aligned tensors (TMA)");
  if (gamma == nullptr) return launch_folded(x, w, bias, out, M, N, K, eps, scale, dt, stream);
  // gamma given: fold it into a scratch copy of w allocated on the stream
  // and released on the stream after the product, so that calls on
  // different streams never share it
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  CUmemoryPool pool = nullptr;
  if (int rc = scratch_pool(api, d.ordinal, &pool)) return rc;
  CUdeviceptr wf = 0;
  CUresult r = api->MemAllocFromPoolAsync(&wf, static_cast<size_t>(N) * static_cast<size_t>(K) * 2,
                                          pool, reinterpret_cast<CUstream>(stream));
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuMemAllocFromPoolAsync(folded weight)");
  void* wfp = reinterpret_cast<void*>(wf);
  int rc = rmsnorm_linear_fold(w, gamma, wfp, N, K, dt, stream);
  if (rc == FUSE_OK) rc = launch_folded(x, wfp, bias, out, M, N, K, eps, scale, dt, stream);
  r = api->MemFreeAsync(wf, reinterpret_cast<CUstream>(stream));
  if (rc != FUSE_OK) return rc;
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuMemFreeAsync(folded weight)");
  return FUSE_OK;
}

extern "C" int rmsnorm_linear_fold(const void* w, const void* gamma, void* w_out, int64_t N,
                                   int64_t K, fuse_dtype dt, void* stream) {
  fuse::NvtxRange nvtx_range("rmsnorm_linear_fold");
  using namespace fuse;
  if (dt != FUSE_F16 && dt != FUSE_BF16) return fail(FUSE_E_DTYPE, "f16 or bf16 only");
  if (N < 0 || K < 1 || K > (int64_t(1) << 20)) return fail(FUSE_E_SHAPE, "bad N or K");
  if (N == 0) return FUSE_OK;
  if (!w || !gamma || !w_out) return fail(FUSE_E_NULL, "NULL tensor pointer");
  std::shared_ptr<Module> mod;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (int rc = rl_module(K, kBN, dt, false, &mod)) return rc;
  }
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  CUfunction fn;
  if (int rc = jit_function(*mod, "rms_linear_fold", d, &fn)) return rc;
  long long total = N * K;
  void* args[] = {&w, &gamma, &w_out, &total};
  // 8 elements (16 bytes) per access when the rows and pointers allow it
  const bool vec = K % 8 == 0 && aligned16(w) && aligned16(gamma) && aligned16(w_out);
  const int64_t items = vec ? total / 8 : total;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(d.sms * 8LL, (items + 255) / 256));
  if (vec) {
    CUfunction fv;
    if (int rc = jit_function(*mod, "rms_linear_fold_vec", d, &fv)) return rc;
    return launch(fv, grid, 256, 0, stream, args);
  }
  return launch(fn, grid, 256, 0, stream, args);
}
