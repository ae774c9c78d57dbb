// graph.cpp -- a sequence of the library's launches recorded once and
// replayed as one CUDA graph.
//
// "DeepJIT ... 串行小核墙" section 5.3 runs the fused kernels in sequence
// outside the engine and records the launches with stream capture into a CUDA
// graph; section 3.1 notes that a graph removes launch overhead but not the
// memory round trips, so it complements fusion rather than replacing it.
// fuse_graph_begin/end wrap stream capture on the caller's stream: every
// library call made on that stream in between (chains, the fixed entry
// points) becomes a node of one graph, replayed by fuse_graph_launch with a
// single submission.
#include "internal.h"

struct fuse_graph {
  CUgraph graph = nullptr;
  CUgraphExec exec = nullptr;
  size_t nodes = 0;
};

extern "C" {

int fuse_graph_begin(void* stream) {
  using namespace fuse;
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  CUresult r = api->StreamBeginCapture(reinterpret_cast<CUstream>(stream),
                                       CU_STREAM_CAPTURE_MODE_THREAD_LOCAL);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuStreamBeginCapture");
  return FUSE_OK;
}

int fuse_graph_end(void* stream, fuse_graph** out) {
  using namespace fuse;
  if (!out) return fail(FUSE_E_NULL, "out is NULL");
  *out = nullptr;
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  auto g = new fuse_graph();
  CUresult r = api->StreamEndCapture(reinterpret_cast<CUstream>(stream), &g->graph);
  if (r != CUDA_SUCCESS) {
    delete g;
    return cuda_fail(r, "cuStreamEndCapture (a call inside the capture may have been illegal "
                        "during capture, e.g. a first-use compile or table build)");
  }
  r = api->GraphGetNodes(g->graph, nullptr, &g->nodes);
  if (r == CUDA_SUCCESS) r = api->GraphInstantiateWithFlags(&g->exec, g->graph, 0);
  if (r != CUDA_SUCCESS) {
    api->GraphDestroy(g->graph);
    delete g;
    return cuda_fail(r, "cuGraphInstantiate");
  }
  *out = g;
  return FUSE_OK;
}

int fuse_graph_launch(fuse_graph* g, void* stream) {
  fuse::NvtxRange nvtx_range("fuse_graph_launch");
  using namespace fuse;
  if (!g || !g->exec) return fail(FUSE_E_ARG, "NULL graph");
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  CUresult r = api->GraphLaunch(g->exec, reinterpret_cast<CUstream>(stream));
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuGraphLaunch");
  stat_launch();
  return FUSE_OK;
}

int fuse_graph_nodes(fuse_graph* g, int64_t* nodes) {
  using namespace fuse;
  if (!g) return fail(FUSE_E_ARG, "NULL graph");
  if (!nodes) return fail(FUSE_E_NULL, "nodes is NULL");
  *nodes = static_cast<int64_t>(g->nodes);
  return FUSE_OK;
}

int fuse_graph_release(fuse_graph* g) {
  using namespace fuse;
  if (!g) return FUSE_OK;
  const DriverApi* api;
  if (driver(&api) == FUSE_OK) {
    if (g->exec) api->GraphExecDestroy(g->exec);
    if (g->graph) api->GraphDestroy(g->graph);
  }
  delete g;
  return FUSE_OK;
}

}  // extern "C"
