// runtime.cpp -- status and counters, the run-time-resolved CUDA driver API,
// device checks, and the NVRTC compile cache ("DeepJIT ... 串行小核墙",
// section 3.2: NVRTC -> module -> function, primary context shared with the
// framework; section 3.3: a map keyed by source + arch + options; section
// 6.2: an in-memory cache and an optional on-disk cache of compiled code;
// section 6.3: no -use_fast_math by default; section 6.4: modules are never
// unloaded while a stream might still run them).
#include <dlfcn.h>
#include <unistd.h>
#include <nvrtc.h>

#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <unordered_map>
#include <unordered_set>

#include "internal.h"

namespace fuse {

// Kernel template headers, embedded at build time: {name, text} pairs.
struct EmbeddedHeader {
  const char* name;
  const char* text;
};
#include "kernels_embedded.inc"  // defines kEmbeddedHeaders[], kNumEmbeddedHeaders

// ------------------------------------------------------------------ status

namespace {
thread_local std::string t_last_error;
std::atomic<int64_t> g_compiles{0}, g_hits{0}, g_launches{0}, g_errors{0};
std::atomic<int64_t> g_compile_us{0};
}  // namespace

int fail(int code, const std::string& msg) {
  t_last_error = msg;
  g_errors.fetch_add(1, std::memory_order_relaxed);
  return code;
}

void clear_error() { t_last_error.clear(); }

std::string fmt(const char* f, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, f);
  vsnprintf(buf, sizeof buf, f, ap);
  va_end(ap);
  return buf;
}

void stat_compile(double ms) {
  g_compiles.fetch_add(1, std::memory_order_relaxed);
  g_compile_us.fetch_add(static_cast<int64_t>(ms * 1000.0), std::memory_order_relaxed);
}
void stat_hit() { g_hits.fetch_add(1, std::memory_order_relaxed); }
void stat_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

const char* last_error_cstr() { return t_last_error.c_str(); }

void read_stats(int64_t* c, int64_t* h, int64_t* l, double* ms) {
  if (c) *c = g_compiles.load();
  if (h) *h = g_hits.load();
  if (l) *l = g_launches.load();
  if (ms) *ms = g_compile_us.load() / 1000.0;
}

// ------------------------------------------------------------------ helpers

int dtype_bytes(fuse_dtype dt) { return dt == FUSE_F32 ? 4 : 2; }
const char* dtype_name(fuse_dtype dt) {
  return dt == FUSE_F32 ? "f32" : dt == FUSE_F16 ? "f16" : "bf16";
}
bool valid_dtype(int dt) { return dt == FUSE_F32 || dt == FUSE_F16 || dt == FUSE_BF16; }

std::string hex_float(float v) {
  char buf[64];
  snprintf(buf, sizeof buf, "%af", static_cast<double>(v));
  return buf;
}

// ------------------------------------------------------------------ driver

namespace {
DriverApi g_api;
int g_driver_status = FUSE_E_CUDA;
std::string g_driver_msg;
std::once_flag g_driver_once;

void load_driver() {
  void* h = dlopen("libcuda.so.1", RTLD_NOW | RTLD_LOCAL);
  if (!h) {
    g_driver_msg = "CUDA driver (libcuda.so.1) not found: no GPU driver on this machine";
    return;
  }
  using GetProc = decltype(&::cuGetProcAddress);
  auto gpa = reinterpret_cast<GetProc>(dlsym(h, "cuGetProcAddress_v2"));
  if (!gpa) {
    g_driver_msg = "CUDA driver too old: cuGetProcAddress_v2 missing";
    return;
  }
  bool ok = true;
  auto get = [&](const char* sym, void** slot) {
    CUdriverProcAddressQueryResult q;
    if (gpa(sym, slot, 12080, CU_GET_PROC_ADDRESS_DEFAULT, &q) != CUDA_SUCCESS || !*slot) {
      g_driver_msg = fmt("CUDA driver lacks %s", sym);
      ok = false;
    }
  };
#define FUSE_GET(field, sym) get(sym, reinterpret_cast<void**>(&g_api.field))
  FUSE_GET(Init, "cuInit");
  FUSE_GET(DeviceGet, "cuDeviceGet");
  FUSE_GET(DeviceGetCount, "cuDeviceGetCount");
  FUSE_GET(DeviceGetAttribute, "cuDeviceGetAttribute");
  FUSE_GET(DevicePrimaryCtxRetain, "cuDevicePrimaryCtxRetain");
  FUSE_GET(CtxGetCurrent, "cuCtxGetCurrent");
  FUSE_GET(CtxSetCurrent, "cuCtxSetCurrent");
  FUSE_GET(CtxGetDevice, "cuCtxGetDevice");
  FUSE_GET(ModuleLoadData, "cuModuleLoadData");
  FUSE_GET(ModuleGetFunction, "cuModuleGetFunction");
  FUSE_GET(LaunchKernel, "cuLaunchKernel");
  FUSE_GET(LaunchKernelEx, "cuLaunchKernelEx");
  FUSE_GET(FuncSetAttribute, "cuFuncSetAttribute");
  FUSE_GET(FuncGetAttribute, "cuFuncGetAttribute");
  FUSE_GET(MemAlloc, "cuMemAlloc");
  FUSE_GET(MemFree, "cuMemFree");
  FUSE_GET(GetErrorName, "cuGetErrorName");
  FUSE_GET(GetErrorString, "cuGetErrorString");
  FUSE_GET(OccupancyMaxActiveBlocksPerMultiprocessor, "cuOccupancyMaxActiveBlocksPerMultiprocessor");
  FUSE_GET(StreamCreate, "cuStreamCreate");
  FUSE_GET(StreamSynchronize, "cuStreamSynchronize");
  FUSE_GET(StreamDestroy, "cuStreamDestroy");
  FUSE_GET(StreamBeginCapture, "cuStreamBeginCapture");
  FUSE_GET(StreamEndCapture, "cuStreamEndCapture");
  FUSE_GET(GraphInstantiateWithFlags, "cuGraphInstantiateWithFlags");
  FUSE_GET(GraphLaunch, "cuGraphLaunch");
  FUSE_GET(GraphExecDestroy, "cuGraphExecDestroy");
  FUSE_GET(GraphDestroy, "cuGraphDestroy");
  FUSE_GET(GraphGetNodes, "cuGraphGetNodes");
  FUSE_GET(TensorMapEncodeTiled, "cuTensorMapEncodeTiled");
  FUSE_GET(CtxSynchronize, "cuCtxSynchronize");
  FUSE_GET(MemcpyDtoH, "cuMemcpyDtoH");
  FUSE_GET(MemsetD32, "cuMemsetD32");
  FUSE_GET(OccupancyMaxActiveClusters, "cuOccupancyMaxActiveClusters");
  FUSE_GET(MemFreeAsync, "cuMemFreeAsync");
  FUSE_GET(MemPoolCreate, "cuMemPoolCreate");
  FUSE_GET(MemPoolSetAttribute, "cuMemPoolSetAttribute");
  FUSE_GET(MemAllocFromPoolAsync, "cuMemAllocFromPoolAsync");
#undef FUSE_GET
  if (!ok) return;
  {
    CUdriverProcAddressQueryResult q;
    if (gpa("cuFuncIsLoaded", reinterpret_cast<void**>(&g_api.FuncIsLoaded), 12040,
            CU_GET_PROC_ADDRESS_DEFAULT, &q) != CUDA_SUCCESS)
      g_api.FuncIsLoaded = nullptr;
    if (gpa("cuFuncLoad", reinterpret_cast<void**>(&g_api.FuncLoad), 12040,
            CU_GET_PROC_ADDRESS_DEFAULT, &q) != CUDA_SUCCESS)
      g_api.FuncLoad = nullptr;
    if (gpa("cuCtxGetId", reinterpret_cast<void**>(&g_api.CtxGetId), 12000,
            CU_GET_PROC_ADDRESS_DEFAULT, &q) != CUDA_SUCCESS)
      g_api.CtxGetId = nullptr;
  }
  CUresult r = g_api.Init(0);
  if (r != CUDA_SUCCESS) {
    const char* name = "?";
    g_api.GetErrorName(r, &name);
    g_driver_msg = fmt("cuInit failed: %s (no usable GPU)", name);
    return;
  }
  g_driver_status = FUSE_OK;
}
}  // namespace

int driver(const DriverApi** api) {
  std::call_once(g_driver_once, load_driver);
  if (g_driver_status != FUSE_OK) return fail(g_driver_status, g_driver_msg);
  *api = &g_api;
  return FUSE_OK;
}

int cuda_fail(CUresult r, const char* what) {
  const char* name = "?";
  const char* desc = "";
  if (g_driver_status == FUSE_OK) {
    g_api.GetErrorName(r, &name);
    g_api.GetErrorString(r, &desc);
  }
  return fail(FUSE_E_CUDA, fmt("%s failed: %s (%s)", what, name, desc ? desc : ""));
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_known[kMaxDevices];
}  // namespace

int current_device(DeviceInfo* info) {
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  CUcontext ctx = nullptr;
  CUresult r = api->CtxGetCurrent(&ctx);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuCtxGetCurrent");
  if (!ctx) {
    int n = 0;
    r = api->DeviceGetCount(&n);
    if (r != CUDA_SUCCESS) return cuda_fail(r, "cuDeviceGetCount");
    if (n == 0) return fail(FUSE_E_CUDA, "no CUDA device visible");
    CUdevice d0;
    if ((r = api->DeviceGet(&d0, 0)) != CUDA_SUCCESS) return cuda_fail(r, "cuDeviceGet");
    if ((r = api->DevicePrimaryCtxRetain(&ctx, d0)) != CUDA_SUCCESS)
      return cuda_fail(r, "cuDevicePrimaryCtxRetain");
    if ((r = api->CtxSetCurrent(ctx)) != CUDA_SUCCESS) return cuda_fail(r, "cuCtxSetCurrent");
  }
  CUdevice dev;
  if ((r = api->CtxGetDevice(&dev)) != CUDA_SUCCESS) return cuda_fail(r, "cuCtxGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FUSE_E_CUDA, "device ordinal out of range");
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_known[dev]) {
      DeviceInfo d{};
      d.ordinal = dev;
      api->DeviceGetAttribute(&d.sms, CU_DEVICE_ATTRIBUTE_MULTIPROCESSOR_COUNT, dev);
      api->DeviceGetAttribute(&d.cc_major, CU_DEVICE_ATTRIBUTE_COMPUTE_CAPABILITY_MAJOR, dev);
      api->DeviceGetAttribute(&d.cc_minor, CU_DEVICE_ATTRIBUTE_COMPUTE_CAPABILITY_MINOR, dev);
      api->DeviceGetAttribute(&d.max_smem_optin,
                              CU_DEVICE_ATTRIBUTE_MAX_SHARED_MEMORY_PER_BLOCK_OPTIN, dev);
      g_dev[dev] = d;
      g_dev_known[dev] = true;
    }
    *info = g_dev[dev];
  }
  if (info->cc_major != 10 || info->cc_minor != 3)
    return fail(FUSE_E_ARCH, fmt("device %d is sm_%d%d; this library is built for sm_103 only",
                                 info->ordinal, info->cc_major, info->cc_minor));
  return FUSE_OK;
}

int default_sms() {
  const DriverApi* api;
  std::call_once(g_driver_once, load_driver);
  if (g_driver_status != FUSE_OK) return 152;
  api = &g_api;
  CUcontext ctx = nullptr;
  if (api->CtxGetCurrent(&ctx) != CUDA_SUCCESS || !ctx) {
    int n = 0;
    if (api->DeviceGetCount(&n) != CUDA_SUCCESS || n == 0) return 152;
  }
  DeviceInfo d;
  std::string saved = t_last_error;
  if (current_device(&d) != FUSE_OK) {
    t_last_error = saved;
    return 152;
  }
  return d.sms;
}

// ------------------------------------------------------------------ jit

namespace {
std::mutex g_cache_mu;
std::condition_variable g_cache_cv;
std::unordered_map<std::string, std::shared_ptr<Module>> g_cache;
std::unordered_set<std::string> g_in_flight;  // keys a thread is compiling now

uint64_t fnv1a(const std::string& s) {
  uint64_t h = 1469598103934665603ull;
  for (unsigned char c : s) {
    h ^= c;
    h *= 1099511628211ull;
  }
  return h;
}

std::vector<std::string> nvrtc_options() {
  std::vector<std::string> o = {"--gpu-architecture=sm_103a", "--std=c++17", "--fmad=true"};
  if (const char* e = getenv("FUSE_LINEINFO"); e && *e == '1') o.push_back("-lineinfo");
  if (const char* e = getenv("FUSE_PTXAS_VERBOSE"); e && *e == '1')
    o.push_back("--ptxas-options=-v");
  // extra NVRTC options, space-separated (part of the cache key like the rest)
  if (const char* e = getenv("FUSE_NVRTC_OPTIONS"); e && *e) {
    std::string all(e), cur;
    for (char c : all + " ") {
      if (c == ' ') {
        if (!cur.empty()) o.push_back(cur);
        cur.clear();
      } else {
        cur += c;
      }
    }
  }
  return o;
}

// What else decides the cubin besides the generated source and the options:
// the text of the embedded headers the source includes and the NVRTC
// version.  Part of every cache key, so that a cache directory filled by
// another build of the library (headers changed) or another NVRTC is
// recompiled rather than loaded.
const std::string& toolchain_tag() {
  static const std::string tag = [] {
    std::string all;
    for (int i = 0; i < kNumEmbeddedHeaders; ++i) {
      all += kEmbeddedHeaders[i].name;
      all += '\0';
      all += kEmbeddedHeaders[i].text;
      all += '\0';
    }
    int major = 0, minor = 0;
    nvrtcVersion(&major, &minor);
    return fmt("headers %016llx nvrtc %d.%d\n", static_cast<unsigned long long>(fnv1a(all)),
               major, minor);
  }();
  return tag;
}

// Optional on-disk cache of cubins (FUSE_CACHE_DIR): file name is the hash
// of the full key; the file holds the key length and a second hash so that
// a collision is detected rather than loaded, and a hash of the cubin so that
// a damaged file is recompiled rather than handed to the driver.
std::string disk_path(const std::string& key) {
  const char* dir = getenv("FUSE_CACHE_DIR");
  if (!dir || !*dir) return {};
  return fmt("%s/fuse_%016llx.cubin", dir, static_cast<unsigned long long>(fnv1a(key)));
}

struct DiskHeader {
  char magic[8];
  uint64_t key_len, key_hash2, cubin_len, cubin_hash;
};

uint64_t bytes_hash(const std::vector<char>& v) {
  uint64_t h = 1469598103934665603ull;
  for (char c : v) {
    h ^= static_cast<unsigned char>(c);
    h *= 1099511628211ull;
  }
  return h;
}

uint64_t hash2(const std::string& key) { return fnv1a("salt:" + key + ":salt"); }

bool disk_load(const std::string& key, std::vector<char>* cubin) {
  std::string p = disk_path(key);
  if (p.empty()) return false;
  std::ifstream f(p, std::ios::binary);
  if (!f) return false;
  DiskHeader h;
  if (!f.read(reinterpret_cast<char*>(&h), sizeof h)) return false;
  if (memcmp(h.magic, "FUSECUB2", 8) != 0 || h.key_len != key.size() || h.key_hash2 != hash2(key) ||
      h.cubin_len == 0 || h.cubin_len > (uint64_t(1) << 30))
    return false;
  cubin->resize(h.cubin_len);
  if (!f.read(cubin->data(), static_cast<std::streamsize>(h.cubin_len)) ||
      bytes_hash(*cubin) != h.cubin_hash) {
    cubin->clear();
    return false;
  }
  return true;
}

void disk_store(const std::string& key, const std::vector<char>& cubin) {
  std::string p = disk_path(key);
  if (p.empty()) return;
  std::string tmp = p + fmt(".tmp%d", static_cast<int>(getpid()));
  std::ofstream f(tmp, std::ios::binary);
  if (!f) return;  // unwritable cache directory: keep going without it
  DiskHeader h;
  memcpy(h.magic, "FUSECUB2", 8);
  h.key_len = key.size();
  h.key_hash2 = hash2(key);
  h.cubin_len = cubin.size();
  h.cubin_hash = bytes_hash(cubin);
  f.write(reinterpret_cast<const char*>(&h), sizeof h);
  f.write(cubin.data(), static_cast<std::streamsize>(cubin.size()));
  f.close();
  if (f) std::rename(tmp.c_str(), p.c_str());
  else std::remove(tmp.c_str());
}
}  // namespace

namespace {

// NVRTC (or the disk cache) for one source, outside the cache lock.
int compile_module(const std::string& key, const std::string& source, const std::string& name,
                   const std::vector<std::string>& opts, Module* m, bool* from_disk) {
  m->name = name;
  *from_disk = disk_load(key, &m->cubin);
  if (*from_disk) return FUSE_OK;
  if (const char* e = getenv("FUSE_VERBOSE"); e && *e == '1')
    fprintf(stderr, "[fuse] compiling %s:\n%s\n", name.c_str(), source.c_str());
  std::vector<const char*> hdr_text, hdr_name;
  for (int i = 0; i < kNumEmbeddedHeaders; ++i) {
    hdr_text.push_back(kEmbeddedHeaders[i].text);
    hdr_name.push_back(kEmbeddedHeaders[i].name);
  }
  nvrtcProgram prog;
  nvrtcResult r = nvrtcCreateProgram(&prog, source.c_str(), (name + ".cu").c_str(),
                                     kNumEmbeddedHeaders, hdr_text.data(), hdr_name.data());
  if (r != NVRTC_SUCCESS)
    return fail(FUSE_E_COMPILE, fmt("nvrtcCreateProgram: %s", nvrtcGetErrorString(r)));
  std::vector<const char*> copt;
  for (auto& o : opts) copt.push_back(o.c_str());
  r = nvrtcCompileProgram(prog, static_cast<int>(copt.size()), copt.data());
  size_t log_size = 0;
  nvrtcGetProgramLogSize(prog, &log_size);
  m->log.resize(log_size);
  if (log_size) nvrtcGetProgramLog(prog, &m->log[0]);
  while (!m->log.empty() && m->log.back() == '\0') m->log.pop_back();
  if (r != NVRTC_SUCCESS) {
    nvrtcDestroyProgram(&prog);
    return fail(FUSE_E_COMPILE,
                fmt("NVRTC failed on %s: %s\n", name.c_str(), nvrtcGetErrorString(r)) + m->log);
  }
  size_t n = 0;
  nvrtcGetCUBINSize(prog, &n);
  m->cubin.resize(n);
  nvrtcGetCUBIN(prog, m->cubin.data());
  nvrtcDestroyProgram(&prog);
  disk_store(key, m->cubin);
  if (const char* e = getenv("FUSE_PTXAS_VERBOSE"); e && *e == '1')
    fprintf(stderr, "[fuse] %s:\n%s\n", name.c_str(), m->log.c_str());
  return FUSE_OK;
}

}  // namespace

int jit_compile(const std::string& source, const std::string& name, std::shared_ptr<Module>* out,
                bool* compiled) {
  if (compiled) *compiled = false;
  std::vector<std::string> opts = nvrtc_options();
  std::string key = "sm_103a\n" + toolchain_tag();
  for (auto& o : opts) key += o + "\n";
  key += source;
  {
    std::unique_lock<std::mutex> lk(g_cache_mu);
    for (;;) {
      auto it = g_cache.find(key);
      if (it != g_cache.end()) {
        stat_hit();
        *out = it->second;
        return FUSE_OK;
      }
      if (!g_in_flight.count(key)) break;
      g_cache_cv.wait(lk);  // another thread compiles this source: take its module
    }
    g_in_flight.insert(key);
  }
  // distinct sources compile in parallel; the same source only once
  auto m = std::make_shared<Module>();
  bool from_disk = false;
  auto t0 = std::chrono::steady_clock::now();
  const int rc = compile_module(key, source, name, opts, m.get(), &from_disk);
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    g_in_flight.erase(key);
    if (rc == FUSE_OK) g_cache.emplace(key, m);
  }
  g_cache_cv.notify_all();  // waiters find the module, or compile (and fail) themselves
  if (rc != FUSE_OK) return rc;
  double ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  if (from_disk) stat_hit();  // a disk load counts as a cache hit, not a compile
  else stat_compile(ms);
  if (compiled) *compiled = !from_disk;
  *out = m;
  return FUSE_OK;
}

int jit_function(Module& m, const char* fn_name, const DeviceInfo& dev, CUfunction* fn) {
  std::lock_guard<std::mutex> lk(m.mu);
  Module::Loaded* ld = nullptr;
  for (auto& l : m.loaded)
    if (l.device == dev.ordinal) ld = &l;
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  if (!ld) {
    CUmodule mod;
    CUresult r = api->ModuleLoadData(&mod, m.cubin.data());
    if (r != CUDA_SUCCESS) return cuda_fail(r, ("cuModuleLoadData(" + m.name + ")").c_str());
    m.loaded.push_back({dev.ordinal, mod, {}});
    ld = &m.loaded.back();
  }
  for (auto& f : ld->fns)
    if (f.first == fn_name) {
      *fn = f.second;
      return FUSE_OK;
    }
  CUfunction f;
  CUresult r = api->ModuleGetFunction(&f, ld->mod, fn_name);
  if (r != CUDA_SUCCESS) return cuda_fail(r, fmt("cuModuleGetFunction(%s)", fn_name).c_str());
  ld->fns.emplace_back(fn_name, f);
  *fn = f;
  return FUSE_OK;
}

int launch(CUfunction fn, unsigned grid, unsigned block, unsigned smem, void* stream, void** args) {
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  if (grid == 0) return FUSE_OK;
  // programmatic dependent launch: the kernel's CTAs may be scheduled while
  // the previous kernel on the stream finishes; the kernel itself waits for
  // that kernel (griddepcontrol.wait, its first statement) before touching
  // memory.  FUSE_PDL=0 launches in plain stream order.
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
  cfg.blockDimX = block;
  cfg.blockDimY = cfg.blockDimZ = 1;
  cfg.sharedMemBytes = smem;
  cfg.hStream = reinterpret_cast<CUstream>(stream);
  cfg.attrs = pdl ? &attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  CUresult r = api->LaunchKernelEx(&cfg, fn, args, nullptr);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuLaunchKernelEx");
  stat_launch();
  return FUSE_OK;
}

}  // namespace fuse

// ------------------------------------------------------------------ device error word

namespace fuse {
namespace {
std::mutex g_err_mu;
CUdeviceptr g_err_words[64];  // per device; set by kernels, read by fuse_device_error
}  // namespace

int device_error_word(int device, CUdeviceptr* out) {
  if (device < 0 || device >= 64) return fail(FUSE_E_ARG, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_words[device]) {
    const DriverApi* api;
    if (int rc = driver(&api)) return rc;
    CUdeviceptr p;
    CUresult r = api->MemAlloc(&p, 16);
    if (r != CUDA_SUCCESS) return cuda_fail(r, "cuMemAlloc(error word)");
    if ((r = api->MemsetD32(p, 0, 4)) != CUDA_SUCCESS) return cuda_fail(r, "cuMemsetD32");
    g_err_words[device] = p;
  }
  *out = g_err_words[device];
  return FUSE_OK;
}
}  // namespace fuse

extern "C" int fuse_device_error(int* code) {
  using namespace fuse;
  if (!code) return fail(FUSE_E_NULL, "code is NULL");
  *code = 0;
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_words[d.ordinal]) return FUSE_OK;
  CUresult r = api->CtxSynchronize();
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuCtxSynchronize");
  if ((r = api->MemcpyDtoH(code, g_err_words[d.ordinal], 4)) != CUDA_SUCCESS)
    return cuda_fail(r, "cuMemcpyDtoH(error word)");
  if ((r = api->MemsetD32(g_err_words[d.ordinal], 0, 4)) != CUDA_SUCCESS)
    return cuda_fail(r, "cuMemsetD32(error word)");
  return FUSE_OK;
}
