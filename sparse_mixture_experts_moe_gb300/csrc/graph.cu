// CUDA-graph replay of moe_forward_ex: the layer's kernels (with their programmatic-dependent-
// launch edges) are captured once on a private stream and replayed with one host call, so a
// small batch is no longer bound by the host's per-kernel launch cost.
#include <cuda_runtime.h>

#include <new>

#include "moe.h"

struct moe_graph_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

extern "C" {

moe_status moe_forward_graph_create(const void* x, const void* w_r, const float* b_r, const void* w1,
                                    const void* w2, int T, int d, int F, int E, int k, moe_dtype dt,
                                    moe_dtype out_dt, moe_path path, int flags, int capacity, void* out,
                                    int32_t* topk_idx, float* topk_gate, int32_t* counts, float* router_stats,
                                    void* workspace, size_t ws_bytes, moe_graph* graph) {
  if (graph == nullptr) return MOE_ERR_INVALID_ARG;
  *graph = nullptr;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MOE_ERR_CUDA;
  // relaxed: the launch path sets kernel attributes and queries the device while capturing
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return MOE_ERR_CUDA;
  }
  const moe_status st = moe_forward_ex(x, w_r, b_r, w1, w2, T, d, F, E, k, dt, out_dt, path, flags, capacity, out,
                                       topk_idx, topk_gate, counts, router_stats, workspace, ws_bytes, cs);
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (st != MOE_OK || ec != cudaSuccess) {
    if (g != nullptr) cudaGraphDestroy(g);
    cudaGetLastError();  // the capture's own error must not leak into the caller's next check
    return st != MOE_OK ? st : MOE_ERR_CUDA;
  }
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  moe_graph h = new (std::nothrow) moe_graph_s;
  if (h == nullptr) {
    cudaGraphExecDestroy(ex);
    cudaGraphDestroy(g);
    return MOE_ERR_CUDA;
  }
  h->graph = g;
  h->exec = ex;
  *graph = h;
  return MOE_OK;
}

moe_status moe_graph_capture_begin(void** capture_stream) {
  if (capture_stream == nullptr) return MOE_ERR_INVALID_ARG;
  *capture_stream = nullptr;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return MOE_ERR_CUDA;
  }
  *capture_stream = cs;
  return MOE_OK;
}

moe_status moe_graph_capture_end(void* capture_stream, moe_graph* graph) {
  if (capture_stream == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t cs = (cudaStream_t)capture_stream;
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (graph == nullptr || ec != cudaSuccess) {
    if (g != nullptr) cudaGraphDestroy(g);
    cudaGetLastError();
    return graph == nullptr ? MOE_ERR_INVALID_ARG : MOE_ERR_CUDA;
  }
  *graph = nullptr;
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  moe_graph h = new (std::nothrow) moe_graph_s;
  if (h == nullptr) {
    cudaGraphExecDestroy(ex);
    cudaGraphDestroy(g);
    return MOE_ERR_CUDA;
  }
  h->graph = g;
  h->exec = ex;
  *graph = h;
  return MOE_OK;
}

moe_status moe_graph_launch(moe_graph graph, void* stream) {
  if (graph == nullptr || graph->exec == nullptr) return MOE_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_graph_destroy(moe_graph graph) {
  if (graph == nullptr) return MOE_OK;
  if (graph->exec != nullptr) cudaGraphExecDestroy(graph->exec);
  if (graph->graph != nullptr) cudaGraphDestroy(graph->graph);
  delete graph;
  return MOE_OK;
}

}  // extern "C"
