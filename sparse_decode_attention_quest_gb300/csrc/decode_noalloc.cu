// se_sparse_paged_decode_noalloc: the sparse paged decode for callers that
// cannot allocate device memory.
//
// se_sparse_paged_decode asks the caller for a workspace that holds the
// per-split partial outputs and log-sum-exps. Some callers cannot provide one:
// a plugin in an inference runtime that is handed its inputs and outputs but no
// scratch buffer, a process whose device memory is owned by another framework's
// caching allocator, or a serving loop that forbids cudaMalloc after start-up
// because it can synchronise the device and stall other streams. This entry
// point keeps the partials in a fixed array inside the library instead, and
// calls no allocator of any kind.
//
// The array is a file-scope __device__ array of kNoAllocScratchBytes (8 MiB).
// Every GPU that loads the library holds it until the process exits. Its device
// address is looked up once per device, by the first call made on that device
// (with that device current); make that first call before any stream capture.
// All calls on a device share the array and it keeps the last call's contents.
// The decode writes every partial it later reads; its per-item arrival counters
// must start at zero, so each call clears them (an asynchronous memset on the
// caller's stream, no allocation) before its launch. Two calls that overlap on
// the GPU (different streams, no ordering) race on the array and both results
// are undefined. The looked-up address stays valid for the life of the device's
// primary context: after cudaDeviceReset the library must not be called on that
// device again in the same process.
#include <mutex>

#include "se_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

// Split partials of se_sparse_paged_decode_noalloc. In host code this name is a
// host-side stand-in, not a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_decode_scratch on the current device, looked up once.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

se_status_t reject(se_status_t st, const char* what) {
  se::set_error_detail("se_sparse_paged_decode_noalloc", what);
  return st;
}

}  // namespace

extern "C" se_status_t se_sparse_paged_decode_noalloc(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                                      const int32_t* block_table, int32_t bt_stride,
                                                      const int32_t* seq_lens, int32_t batch,
                                                      const int32_t* sel_pages, const int32_t* sel_counts,
                                                      int32_t sel_stride, float sm_scale, void* out, float* out_lse,
                                                      void* stream) {
  bool latent = false;
  const se_status_t st = se::check_decode_call("se_sparse_paged_decode_noalloc", kv, q, num_q_heads, block_table,
                                               bt_stride, seq_lens, batch, sel_pages, sel_counts, sel_stride,
                                               sm_scale, out, out_lse, &latent);
  if (st != SE_OK) return st;
  if (latent)
    return reject(SE_ERR_UNSUPPORTED, "a latent cache needs se_sparse_paged_decode with a caller workspace; this "
                                      "entry covers head_dim = head_dim_v = 128 with <= 16 query heads per KV head");

  int sm_count = 0;
  unsigned* err = nullptr;
  cudaError_t e = se::device_context(&sm_count, &err);
  if (e != cudaSuccess) return reject(SE_ERR_CUDA, cudaGetErrorString(e));
  const se::DecodePlan plan = se::plan_gqa_decode(batch, kv->num_kv_heads, sel_stride, sm_count);
  const size_t need = se::gqa_decode_workspace_bytes(batch, num_q_heads, kv->head_dim_v, plan);
  if (need > kNoAllocScratchBytes)
    return reject(SE_ERR_WORKSPACE, "these sizes need more split scratch than the built-in 8 MiB array; "
                                    "use se_sparse_paged_decode with a caller workspace");
  if ((size_t)batch * kv->num_kv_heads > se::gqa_decode_max_items())
    return reject(SE_ERR_UNSUPPORTED, "too many (request, KV head) items for one launch");
  if (batch == 0) return SE_OK;
  void* scratch = nullptr;
  e = scratch_address(&scratch);
  if (e != cudaSuccess) return reject(SE_ERR_CUDA, cudaGetErrorString(e));

  // The arrival counters of the split merge start at zero on every call.
  const size_t counters = se::gqa_decode_arrivals_offset(batch, num_q_heads, kv->head_dim_v, plan);
  e = cudaMemsetAsync(static_cast<unsigned char*>(scratch) + counters, 0,
                      (size_t)batch * kv->num_kv_heads * sizeof(uint32_t), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return reject(SE_ERR_CUDA, cudaGetErrorString(e));

  se::KvView view;
  view.k = static_cast<const uint16_t*>(kv->k);
  view.v = static_cast<const uint16_t*>(kv->v);
  view.summary = static_cast<uint16_t*>(kv->summary);
  view.num_pages = kv->num_pages;
  view.num_kv_heads = kv->num_kv_heads;
  view.head_dim = kv->head_dim;
  view.head_dim_v = kv->head_dim_v;
  view.row_stride_k = kv->row_stride_k;
  view.row_stride_v = kv->row_stride_v;
  e = se::launch_gqa_decode(view, static_cast<const uint16_t*>(q), num_q_heads, block_table, bt_stride, seq_lens,
                            batch, sel_pages, sel_counts, sel_stride, sm_scale, static_cast<uint16_t*>(out), out_lse,
                            scratch, plan, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return reject(SE_ERR_CUDA, cudaGetErrorString(e));
  return SE_OK;
}
