// internal.h -- shared declarations of the fused-chain library's host side.
#pragma once

#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "fuse.h"

namespace fuse {

// ------------------------------------------------------------------ status
// Sets the calling thread's last-error message, counts the error and
// returns `code` (so call sites read `return fail(FUSE_E_ARG, "...")`).
int fail(int code, const std::string& msg);
void clear_error();
const char* last_error_cstr();  // the calling thread's last-error message
std::string fmt(const char* f, ...) __attribute__((format(printf, 1, 2)));

struct Stats {
  int64_t compiles, cache_hits, launches, errors;
  double compile_ms;
};
void stat_compile(double ms);
void stat_hit();
void stat_launch();

// ------------------------------------------------------------------ driver
// The CUDA driver API is resolved at run time (dlopen of libcuda.so.1 and
// cuGetProcAddress), so the library loads on machines without a GPU driver;
// calls that need the device then fail with FUSE_E_CUDA.
struct DriverApi {
  decltype(&::cuInit) Init;
  decltype(&::cuDeviceGet) DeviceGet;
  decltype(&::cuDeviceGetCount) DeviceGetCount;
  decltype(&::cuDeviceGetAttribute) DeviceGetAttribute;
  decltype(&::cuDevicePrimaryCtxRetain) DevicePrimaryCtxRetain;
  decltype(&::cuCtxGetCurrent) CtxGetCurrent;
  decltype(&::cuCtxSetCurrent) CtxSetCurrent;
  decltype(&::cuCtxGetDevice) CtxGetDevice;
  decltype(&::cuModuleLoadData) ModuleLoadData;
  decltype(&::cuModuleGetFunction) ModuleGetFunction;
  decltype(&::cuLaunchKernel) LaunchKernel;
  decltype(&::cuLaunchKernelEx) LaunchKernelEx;
  decltype(&::cuFuncSetAttribute) FuncSetAttribute;
  decltype(&::cuFuncGetAttribute) FuncGetAttribute;
  decltype(&::cuMemAlloc) MemAlloc;
  decltype(&::cuMemFree) MemFree;
  decltype(&::cuGetErrorName) GetErrorName;
  decltype(&::cuGetErrorString) GetErrorString;
  decltype(&::cuOccupancyMaxActiveBlocksPerMultiprocessor) OccupancyMaxActiveBlocksPerMultiprocessor;
  decltype(&::cuStreamCreate) StreamCreate;
  decltype(&::cuStreamSynchronize) StreamSynchronize;
  decltype(&::cuStreamDestroy) StreamDestroy;
  decltype(&::cuStreamBeginCapture) StreamBeginCapture;
  decltype(&::cuStreamEndCapture) StreamEndCapture;
  decltype(&::cuGraphInstantiateWithFlags) GraphInstantiateWithFlags;
  decltype(&::cuGraphLaunch) GraphLaunch;
  decltype(&::cuGraphExecDestroy) GraphExecDestroy;
  decltype(&::cuGraphDestroy) GraphDestroy;
  decltype(&::cuGraphGetNodes) GraphGetNodes;
  decltype(&::cuTensorMapEncodeTiled) TensorMapEncodeTiled;
  decltype(&::cuCtxSynchronize) CtxSynchronize;
  decltype(&::cuMemcpyDtoH) MemcpyDtoH;
  decltype(&::cuMemsetD32) MemsetD32;
  decltype(&::cuOccupancyMaxActiveClusters) OccupancyMaxActiveClusters;
  decltype(&::cuMemFreeAsync) MemFreeAsync;
  decltype(&::cuMemPoolCreate) MemPoolCreate;
  decltype(&::cuMemPoolSetAttribute) MemPoolSetAttribute;
  decltype(&::cuMemAllocFromPoolAsync) MemAllocFromPoolAsync;
  // optional (NULL on drivers before CUDA 12.4)
  decltype(&::cuFuncIsLoaded) FuncIsLoaded;
  decltype(&::cuFuncLoad) FuncLoad;
  decltype(&::cuCtxGetId) CtxGetId;
};

// Returns FUSE_OK and the API table, or FUSE_E_CUDA (driver missing).
int driver(const DriverApi** api);

// Error message for a failed driver call.
int cuda_fail(CUresult r, const char* what);

struct DeviceInfo {
  int ordinal;
  int sms;
  int cc_major, cc_minor;
  int max_smem_optin;
};

// Makes a context current on the calling thread (the primary context of
// device 0 when none is), checks that the device is sm_103 and returns its
// description.  FUSE_E_CUDA without a driver/device, FUSE_E_ARCH on another
// architecture.
int current_device(DeviceInfo* info);

// SM count of the current device, or 152 when there is none.
int default_sms();

// ------------------------------------------------------------------ jit
// A compiled module: the sm_103a cubin of one generated source, loaded
// lazily on each device that uses it.  Modules are never unloaded.
struct Module {
  std::string name;
  std::vector<char> cubin;
  std::string log;
  std::mutex mu;
  struct Loaded {
    int device;
    CUmodule mod;
    std::vector<std::pair<std::string, CUfunction>> fns;
  };
  std::vector<Loaded> loaded;
};

// Compile `source` (cache key: source + arch + options) or fetch it from the
// cache.  `name` is used in messages only.
// Thread-safe: the same source compiles once (later callers wait for it),
// distinct sources compile in parallel.  *compiled (if given) tells whether
// NVRTC ran, as opposed to a memory or disk cache hit.
int jit_compile(const std::string& source, const std::string& name, std::shared_ptr<Module>* out,
                bool* compiled = nullptr);

// The kernel `fn_name` of module m on the current device (loads the module
// there on first use).
int jit_function(Module& m, const char* fn_name, const DeviceInfo& dev, CUfunction* fn);

// Launch on `stream` and count it.
int launch(CUfunction fn, unsigned grid, unsigned block, unsigned smem, void* stream, void** args);

// The device's error word (allocated on first use): kernels with bounded
// waits or debug bounds checks write a nonzero code there instead of
// trapping; fuse_device_error() reads and clears it.
//   1 a bounded wait ran out, 2 too little shared memory for the layout,
//   3 an index outside its tensor (FUSE_DEBUG_BOUNDS)
int device_error_word(int device, CUdeviceptr* out);

// A named range around an ABI call, for timeline profilers (NVTX v3,
// header-only; a few nanoseconds when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ------------------------------------------------------------------ helpers
int dtype_bytes(fuse_dtype dt);
const char* dtype_name(fuse_dtype dt);
bool valid_dtype(int dt);
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
std::string hex_float(float v);  // exact C++ literal of an fp32 value ("0x1p-1f")

}  // namespace fuse
