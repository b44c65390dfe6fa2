// Replayable steps: the asynchronous work of a sequence of library calls on one
// stream, recorded once into a CUDA graph and launched as a whole afterwards.
//
// A decode loop makes the same calls every step on the same buffers; only the
// values in device memory (queries, new K/V rows, lengths, selections) change.
// Each call validates its arguments on the host and launches its kernels; a
// recorded step skips all of that and costs one graph launch. The kernels' own
// programmatic-dependent-launch edges are recorded as such, so the replayed
// step overlaps each kernel's start with the previous one as the live calls do.
#include <algorithm>
#include <new>

#include "se_internal.h"
#include "se_ptx.cuh"

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

namespace {

// Copies of up to kKernelCopyMax bytes between device memory and page-locked
// host memory run as a kernel: the SMs load and store the host side directly
// over the GPU's link to host memory, all 16-byte pieces in flight at once,
// which for the few hundred KB of a decode step's inputs or output takes a
// fraction of a copy engine's start-up. The kernel waits for the previous
// kernel of the stream (which may have written the source) before its loads.
constexpr size_t kKernelCopyMax = size_t(8) << 20;
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                              size_t n16) {
  se::pdl_enter();
  for (size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x; i < n16; i += (size_t)gridDim.x * kCopyThreads)
    dst[i] = src[i];
}

__global__ void __launch_bounds__(kCopyThreads) copy1_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                                             size_t n) {
  se::pdl_enter();
  for (size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x; i < n; i += (size_t)gridDim.x * kCopyThreads)
    dst[i] = src[i];
}

// The address through which kernels reach p: itself for device (or managed)
// memory, the mapped address for page-locked host memory; NULL otherwise.
void* device_view(const void* p, bool* host) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  *host = at.type == cudaMemoryTypeHost;
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return const_cast<void*>(p);
  if (at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}

}  // namespace

extern "C" se_status_t se_copy_async(void* dst, const void* src, size_t bytes, void* stream) {
  static const char* fn = "se_copy_async";
  if (bytes == 0) return SE_OK;
  if (!dst || !src) {
    se::set_error_detail(fn, "NULL dst or src");
    return SE_ERR_INVALID_ARG;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bytes <= kKernelCopyMax) {
    bool dst_host = false, src_host = false;
    void* d = device_view(dst, &dst_host);
    const void* s = device_view(src, &src_host);
    if (d && s && (dst_host || src_host)) {
      int sm_count = 0;
      unsigned* err = nullptr;
      cudaError_t e = se::device_context(&sm_count, &err);
      if (e != cudaSuccess) return graph_fail(fn, e);
      const bool wide = ((reinterpret_cast<uintptr_t>(d) | reinterpret_cast<uintptr_t>(s) | bytes) & 15) == 0;
      const size_t n = wide ? bytes / 16 : bytes;
      const size_t blocks = std::min<size_t>((n + kCopyThreads - 1) / kCopyThreads, (size_t)sm_count * 8);
      e = wide ? se::launch_pdl(copy16_kernel, dim3((unsigned)blocks), dim3(kCopyThreads), 0, st,
                                static_cast<uint4*>(d), static_cast<const uint4*>(s), n)
               : se::launch_pdl(copy1_kernel, dim3((unsigned)blocks), dim3(kCopyThreads), 0, st,
                                static_cast<uint8_t*>(d), static_cast<const uint8_t*>(s), n);
      if (e != cudaSuccess) return graph_fail(fn, e);
      return SE_OK;
    }
  }
  // Otherwise the copy engine; cudaMemcpyDefault: the direction follows from
  // the unified addresses of device memory and of page-locked host memory.
  const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, st);
  if (e != cudaSuccess) return graph_fail(fn, e);
  return SE_OK;
}
