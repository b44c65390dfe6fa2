// Replayable steps: the asynchronous work of a sequence of library calls on one
// stream, recorded once into a CUDA graph and launched as a whole afterwards.
//
// A decode loop makes the same calls every step on the same buffers; only the
// values in device memory (queries, new K/V rows, lengths, selections) change.
// Each call validates its arguments on the host and launches its kernels; a
// recorded step skips all of that and costs one graph launch. The kernels' own
// programmatic-dependent-launch edges are recorded as such, so the replayed
// step overlaps each kernel's start with the previous one as the live calls do.
#include <new>

#include "se_internal.h"

struct se_graph_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

namespace {

se_status_t graph_fail(const char* fn, cudaError_t e) {
  se::set_error_detail(fn, cudaGetErrorString(e));
  return SE_ERR_CUDA;
}

}  // namespace

extern "C" se_status_t se_capture_begin(void* stream) {
  static const char* fn = "se_capture_begin";
  if (!stream) {
    se::set_error_detail(fn, "capturing needs a stream other than the legacy default stream");
    return SE_ERR_INVALID_ARG;
  }
  // The per-device context (device properties, the device error word) is set
  // up here, outside the recording, so that no call made during it allocates.
  int sm_count = 0;
  unsigned* err = nullptr;
  cudaError_t e = se::device_context(&sm_count, &err);
  if (e != cudaSuccess) return graph_fail(fn, e);
  e = cudaStreamBeginCapture(static_cast<cudaStream_t>(stream), cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return graph_fail(fn, e);
  return SE_OK;
}

extern "C" se_status_t se_capture_end(void* stream, se_graph_t* graph) {
  static const char* fn = "se_capture_end";
  if (!stream || !graph) {
    se::set_error_detail(fn, "NULL stream or graph");
    return SE_ERR_INVALID_ARG;
  }
  *graph = nullptr;
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(static_cast<cudaStream_t>(stream), &g);
  if (e != cudaSuccess) return graph_fail(fn, e);
  cudaGraphExec_t x = nullptr;
  e = cudaGraphInstantiate(&x, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return graph_fail(fn, e);
  }
  se_graph_s* h = new (std::nothrow) se_graph_s;
  if (!h) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    se::set_error_detail(fn, "out of host memory");
    return SE_ERR_CUDA;
  }
  h->graph = g;
  h->exec = x;
  *graph = h;
  return SE_OK;
}

extern "C" se_status_t se_graph_launch(se_graph_t graph, void* stream) {
  static const char* fn = "se_graph_launch";
  if (!graph) {
    se::set_error_detail(fn, "graph is NULL");
    return SE_ERR_INVALID_ARG;
  }
  const cudaError_t e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return graph_fail(fn, e);
  return SE_OK;
}

extern "C" void se_graph_destroy(se_graph_t graph) {
  if (!graph) return;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
}
