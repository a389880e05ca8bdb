// Layer sequences (a DiT block stack with selectively skipped dense layers) and their CUDA graphs: host code
// only.  Every layer is checked before anything is enqueued; the graph is one stream capture of the same
// sequence of lynx_linear / lynx_linear_dense calls, so a replay runs exactly the kernels an eager run would.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "../../include/lynx.h"
#include "kernels.h"

struct lynx_graph_s {
  cudaGraphExec_t exec;
};

namespace lynx {
namespace {

size_t layer_workspace_bytes(const lynx_layer& l) {
  if (l.sparse) return lynx_workspace_bytes(l.M, l.N, l.K, l.R);
  return (l.LA || l.LB) ? lynx_dense_workspace_bytes(l.M, l.R) : 0;
}

int layer_status(const lynx_layer& l, const void* ws, size_t ws_bytes) {
  return l.sparse ? linear_arg_status(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, ws_bytes)
                  : dense_arg_status(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, ws_bytes);
}

// LYNX_OK when every layer would launch; else the first failure, its index in *failed.
int check_layers(const lynx_layer* layers, int32_t n, const void* ws, size_t ws_bytes, int32_t* failed) {
  if (failed) *failed = -1;
  if (n > 0 && !layers) return LYNX_ERR_NULL;
  if (n < 0) return LYNX_ERR_SHAPE;
  for (int32_t i = 0; i < n; ++i) {
    if (int e = layer_status(layers[i], ws, ws_bytes)) {
      if (failed) *failed = i;
      return e;
    }
  }
  return LYNX_OK;
}

int enqueue_layers(const lynx_layer* layers, int32_t n, void* ws, size_t ws_bytes, void* stream) {
  for (int32_t i = 0; i < n; ++i) {
    const lynx_layer& l = layers[i];
    const int e = l.sparse ? lynx_linear(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, ws_bytes, stream)
                           : lynx_linear_dense(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, ws_bytes, stream);
    if (e) return e;
  }
  return LYNX_OK;
}

}  // namespace
}  // namespace lynx

using namespace lynx;

extern "C" {

size_t lynx_layers_workspace_bytes(const lynx_layer* layers, int32_t n) {
  if (!layers || n < 1) return 0;
  size_t b = 0;
  for (int32_t i = 0; i < n; ++i) {
    const size_t w = layer_workspace_bytes(layers[i]);
    if (w > b) b = w;
  }
  return b;
}

int lynx_run_layers(const lynx_layer* layers, int32_t n, void* workspace, size_t workspace_bytes, void* stream,
                    int32_t* failed_layer) {
  if (int e = check_layers(layers, n, workspace, workspace_bytes, failed_layer)) return e;
  return enqueue_layers(layers, n, workspace, workspace_bytes, stream);
}

int lynx_graph_create(const lynx_layer* layers, int32_t n, void* workspace, size_t workspace_bytes,
                      lynx_graph* graph_out, int32_t* failed_layer) {
  if (failed_layer) *failed_layer = -1;
  if (!graph_out) return LYNX_ERR_NULL;
  *graph_out = nullptr;
  if (!layers) return LYNX_ERR_NULL;
  if (n < 1) return LYNX_ERR_SHAPE;
  if (int e = check_layers(layers, n, workspace, workspace_bytes, failed_layer)) return e;

  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return LYNX_ERR_CUDA;
  clear_stage_request();  // no stage-timing events inside the graph
  int status = LYNX_OK;
  cudaGraph_t graph = nullptr;
  // Relaxed mode: the launch helpers may set a kernel attribute or query occupancy on their first use.
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    status = LYNX_ERR_CUDA;
  } else {
    status = enqueue_layers(layers, n, workspace, workspace_bytes, s);
    const cudaError_t end = cudaStreamEndCapture(s, &graph);  // always ends the capture
    if (status == LYNX_OK && end != cudaSuccess) status = LYNX_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (status == LYNX_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) status = LYNX_ERR_CUDA;
  if (graph) cudaGraphDestroy(graph);
  cudaStreamDestroy(s);
  if (status != LYNX_OK) {
    if (exec) cudaGraphExecDestroy(exec);
    cudaGetLastError();  // clear the (non-sticky) last-error state a failed capture leaves behind
    return status;
  }
  lynx_graph_s* g = new (std::nothrow) lynx_graph_s{exec};
  if (!g) {
    cudaGraphExecDestroy(exec);
    return LYNX_ERR_CUDA;
  }
  *graph_out = g;
  return LYNX_OK;
}

int lynx_graph_launch(lynx_graph graph, void* stream) {
  if (!graph) return LYNX_ERR_NULL;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LYNX_OK : LYNX_ERR_CUDA;
}

int lynx_graph_destroy(lynx_graph graph) {
  if (!graph) return LYNX_OK;
  const cudaError_t e = cudaGraphExecDestroy(graph->exec);
  delete graph;
  return e == cudaSuccess ? LYNX_OK : LYNX_ERR_CUDA;
}

}  // extern "C"
