// Layer sequences (a DiT block stack with selectively skipped dense layers and fused MLP pairs) and their CUDA
// graphs: host code only.  Every layer is checked before anything is enqueued (seq_status); the launches come
// from seq_enqueue (lynx_api.cu), and the graph is one stream capture of the same launches, so a replay runs
// exactly the kernels an eager run would.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "../../include/lynx.h"
#include "kernels.h"

struct lynx_graph_s {
  cudaGraphExec_t exec;
};

using namespace lynx;

extern "C" {

size_t lynx_layers_workspace_bytes(const lynx_layer* layers, int32_t n) { return seq_workspace_bytes(layers, n); }

int lynx_run_layers(const lynx_layer* layers, int32_t n, void* workspace, size_t workspace_bytes, void* stream,
                    int32_t* failed_layer) {
  if (int e = seq_status(layers, n, workspace, workspace_bytes, failed_layer)) return e;
  return seq_enqueue(layers, n, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int lynx_graph_create(const lynx_layer* layers, int32_t n, void* workspace, size_t workspace_bytes,
                      lynx_graph* graph_out, int32_t* failed_layer) {
  if (failed_layer) *failed_layer = -1;
  if (!graph_out) return LYNX_ERR_NULL;
  *graph_out = nullptr;
  if (!layers) return LYNX_ERR_NULL;
  if (n < 1) return LYNX_ERR_SHAPE;
  if (int e = seq_status(layers, n, workspace, workspace_bytes, failed_layer)) return e;

  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return LYNX_ERR_CUDA;
  clear_stage_request();  // no stage-timing events inside the graph
  int status = LYNX_OK;
  cudaGraph_t graph = nullptr;
  // Relaxed mode: the launch helpers may set a kernel attribute or query occupancy on their first use.
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    status = LYNX_ERR_CUDA;
  } else {
    status = seq_enqueue(layers, n, workspace, workspace_bytes, s);
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

int lynx_debug_pair_offsets(const lynx_layer* layers, int32_t n, int32_t i, size_t* offsets) {
  return seq_pair_offsets(layers, n, i, offsets);
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
