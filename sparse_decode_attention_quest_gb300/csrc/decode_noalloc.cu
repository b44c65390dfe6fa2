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
// All calls on a device share the array and it keeps the last call's contents:
// the decode writes every partial it later reads, so nothing needs clearing,
// but two calls that overlap on the GPU (different streams, no ordering) race
// on it and both results are undefined.
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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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
  if (!kv || !kv->k || !kv->v) return reject(SE_ERR_INVALID_ARG, "kv, kv->k or kv->v is NULL");
  if (!aligned16(kv->k) || !aligned16(kv->v)) return reject(SE_ERR_INVALID_ARG, "cache not 16-byte aligned");
  if (kv->page_size != se::kPageSize || kv->num_pages < 0 || kv->num_kv_heads < 1)
    return reject(SE_ERR_INVALID_ARG, "bad page_size / num_pages / num_kv_heads");
  if (kv->row_stride_k < kv->head_dim || kv->row_stride_v < kv->head_dim_v || (kv->row_stride_k % 8) ||
      (kv->row_stride_v % 8))
    return reject(SE_ERR_INVALID_ARG, "row strides must cover the head dims and be multiples of 8");
  if ((long long)kv->num_pages * kv->num_kv_heads * se::kPageSize >= (1ll << 31))
    return reject(SE_ERR_UNSUPPORTED, "cache holds 2^31 or more token rows");
  if (batch < 0 || sel_stride < 1 || bt_stride < 1) return reject(SE_ERR_INVALID_ARG, "bad sizes");
  if (num_q_heads < 1 || num_q_heads % kv->num_kv_heads)
    return reject(SE_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  if (batch > 0 && (!q || !block_table || !seq_lens || !sel_pages || !sel_counts || !out))
    return reject(SE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(q) || !aligned16(out) || !aligned16(out_lse) || !aligned16(sel_pages))
    return reject(SE_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (!(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f)
    return reject(SE_ERR_INVALID_ARG, "sm_scale not finite");
  if (!(kv->head_dim == 128 && kv->head_dim_v == 128 && num_q_heads / kv->num_kv_heads <= 16))
    return reject(SE_ERR_UNSUPPORTED, "only head_dim = head_dim_v = 128 with <= 16 query heads per KV head");

  int sm_count = 0;
  unsigned* err = nullptr;
  cudaError_t e = se::device_context(&sm_count, &err);
  if (e != cudaSuccess) return reject(SE_ERR_CUDA, cudaGetErrorString(e));
  const se::DecodePlan plan = se::plan_gqa_decode(batch, kv->num_kv_heads, sel_stride, sm_count);
  const size_t need = se::gqa_decode_workspace_bytes(batch, num_q_heads, kv->head_dim_v, plan);
  if (need > kNoAllocScratchBytes)
    return reject(SE_ERR_WORKSPACE, "these sizes need more split scratch than the built-in 8 MiB array; "
                                    "use se_sparse_paged_decode with a caller workspace");
  if (batch == 0) return SE_OK;
  void* scratch = nullptr;
  e = scratch_address(&scratch);
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
  if ((size_t)batch * kv->num_kv_heads > se::gqa_decode_max_items())
    return reject(SE_ERR_UNSUPPORTED, "too many (request, KV head) items for one launch");
  e = se::launch_gqa_decode(view, static_cast<const uint16_t*>(q), num_q_heads, block_table, bt_stride, seq_lens,
                            batch, sel_pages, sel_counts, sel_stride, sm_scale, static_cast<uint16_t*>(out), out_lse,
                            scratch, plan, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return reject(SE_ERR_CUDA, cudaGetErrorString(e));
  return SE_OK;
}
