// The whole forward as one CUDA graph owned by the library: engram_forward's kernel chain (hash +
// gather, projection, gate, each launched with programmatic dependent launch) captured once on a
// private stream, instantiated, and replayed by one cudaGraphLaunch per step. A decode loop then
// costs one host call and one graph launch per step instead of three kernel launches.
//
// Everything a step reads or writes is a pointer captured at creation: the caller refills x,
// tokens (and the mask) in place between launches. The cache lengths live on the device and each
// replay advances them, as consecutive engram_forward calls do.
#include <cuda_runtime.h>

#include <cstdio>
#include <new>

#include "engram.h"
#include "kernels.h"

struct engram_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  int device;
};

namespace {

// records the message engram_last_error() returns
int graph_fail(int code, const char* what, cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, e == cudaSuccess ? "failed" : cudaGetErrorString(e));
  return engram::set_last_error(code, msg);
}

}  // namespace

ENGRAM_API int engram_forward_graph_create(
    const engram_desc_t* desc, const engram_tables_t* tables, const engram_weights_t* weights,
    const uint16_t* x, const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
    int32_t* cache_len, int32_t capacity, const uint8_t* token_mask, uint16_t* out,
    int32_t* hash_ids_out, float* gate_out, uint16_t* kv_out, void* workspace,
    size_t workspace_bytes, engram_graph_t** graph_out) {
  if (graph_out == nullptr) return graph_fail(ENGRAM_EINVAL, "graph_out is NULL", cudaSuccess);
  *graph_out = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return graph_fail(ENGRAM_ECUDA, "cudaGetDevice", e);
  cudaStream_t s = nullptr;
  if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess)
    return graph_fail(ENGRAM_ECUDA, "cudaStreamCreateWithFlags", e);
  // relaxed: the first call on a device may still resolve device symbols and set kernel
  // attributes, which are not stream work and need not be captured
  if ((e = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed)) != cudaSuccess) {
    cudaStreamDestroy(s);
    return graph_fail(ENGRAM_ECUDA, "cudaStreamBeginCapture", e);
  }
  // argument errors are engram_forward's own (and so is its engram_last_error message)
  const int rc = engram_forward(desc, tables, weights, x, tokens, B, T, cache, cache_len, capacity,
                                token_mask, out, hash_ids_out, gate_out, kv_out, workspace,
                                workspace_bytes, s);
  cudaGraph_t g = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &g);   // ends the capture whatever happened
  cudaStreamDestroy(s);
  if (rc != ENGRAM_OK || end != cudaSuccess || g == nullptr) {
    if (g) cudaGraphDestroy(g);
    return rc != ENGRAM_OK ? rc
                           : graph_fail(ENGRAM_ECUDA, "stream capture of engram_forward", end);
  }
  cudaGraphExec_t exec = nullptr;
  if ((e = cudaGraphInstantiate(&exec, g, 0)) != cudaSuccess) {
    cudaGraphDestroy(g);
    return graph_fail(ENGRAM_ECUDA, "cudaGraphInstantiate", e);
  }
  engram_graph_t* h = new (std::nothrow) engram_graph_t{g, exec, dev};
  if (h == nullptr) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(g);
    return graph_fail(ENGRAM_EINVAL, "host allocation of the graph handle", cudaSuccess);
  }
  *graph_out = h;
  return ENGRAM_OK;
}

ENGRAM_API int engram_graph_launch(const engram_graph_t* graph, void* stream) {
  if (graph == nullptr) return graph_fail(ENGRAM_EINVAL, "graph is NULL", cudaSuccess);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return graph_fail(ENGRAM_ECUDA, "cudaGetDevice", e);
  if (dev != graph->device)
    return graph_fail(ENGRAM_EINVAL, "the graph belongs to another device", cudaSuccess);
  if ((e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return graph_fail(ENGRAM_ECUDA, "cudaGraphLaunch", e);
  return ENGRAM_OK;
}

ENGRAM_API int engram_graph_destroy(engram_graph_t* graph) {
  if (graph == nullptr) return ENGRAM_OK;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
  return ENGRAM_OK;
}
