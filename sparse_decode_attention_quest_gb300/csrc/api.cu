// Host entry points of the C ABI declared in include/sparse_engine.h:
// argument validation (before any launch), per-device cached properties,
// tensor-map encoding for the TMA copies, and dispatch to the kernels.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "se_internal.h"

// The library's device error word (SE_DEVERR_* bits), one per device context.
__device__ unsigned se_device_error_word;

namespace {

using se::KvView;

thread_local char g_detail[256] = "";

se_status_t fail(se_status_t st, const char* fn, const char* what) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s", fn, what);
  return st;
}

se_status_t cuda_fail(const char* fn, cudaError_t e) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s (%s)", fn, cudaGetErrorName(e), cudaGetErrorString(e));
  return SE_ERR_CUDA;
}

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  unsigned* err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

// Properties of the current device, queried once per device.
cudaError_t current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), se_device_error_word);
    if (e != cudaSuccess) return e;
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D view of a paged cache (or any row-major bf16 matrix) as rows of
// `row_stride` bf16, boxes of 64 columns x `box_rows` rows with 128-byte swizzle.
bool encode_page_map(CUtensorMap* map, const void* base, long long rows, int width, int row_stride,
                     int box_rows = se::kPageSize) {
  auto fn = encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_stride * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view of a bf16 cache of `rows` rows, `row_stride` elements apart, as
// (64 dims, row, 64-dim chunk) with the chunks 128 bytes apart. A box of
// 64 x box_rows x chunks copies box_rows rows, every chunk, with a single
// request, into [chunk][row][128 bytes] with 128-byte swizzle: a SnapKV page
// of one head (16 rows x 2 chunks, 4 KB), or half a latent page (8 rows x 9
// chunks, 9 KB).
bool encode_row_chunks_map(CUtensorMap* map, const void* base, long long rows, int row_stride, int chunks,
                           int box_rows) {
  auto fn = encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)chunks};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D view of SnapKV window queries bf16 [batch][window][num_q_heads][128]: boxes of
// 64 dims x `group` heads x `window` positions x 1 request (128-byte swizzle), so one
// box holds a KV head's window rows r = w * group + g for 64 of the dims.
bool encode_window_map(CUtensorMap* map, const void* base, int batch, int window, int num_q_heads, int group) {
  auto fn = encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[4] = {128, (cuuint64_t)num_q_heads, (cuuint64_t)window, (cuuint64_t)batch};
  cuuint64_t strides[3] = {128 * 2, (cuuint64_t)num_q_heads * 128 * 2, (cuuint64_t)window * num_q_heads * 128 * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)group, (cuuint32_t)window, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int pages_of(long long tokens) { return (int)((tokens + se::kPageSize - 1) / se::kPageSize); }

// Common checks of a paged cache view.
se_status_t check_kv(const char* fn, const se_paged_kv_t* kv, bool need_summary) {
  if (!kv) return fail(SE_ERR_INVALID_ARG, fn, "kv is NULL");
  if (!kv->k || !kv->v) return fail(SE_ERR_INVALID_ARG, fn, "kv->k / kv->v is NULL");
  if (need_summary && !kv->summary) return fail(SE_ERR_INVALID_ARG, fn, "kv->summary is NULL");
  if (!aligned16(kv->k) || !aligned16(kv->v) || (kv->summary && !aligned16(kv->summary)))
    return fail(SE_ERR_INVALID_ARG, fn, "cache pointers must be 16-byte aligned");
  if (kv->page_size != se::kPageSize) return fail(SE_ERR_INVALID_ARG, fn, "page_size must be 16");
  if (kv->num_pages < 0 || kv->num_kv_heads < 1) return fail(SE_ERR_INVALID_ARG, fn, "bad num_pages/num_kv_heads");
  if (kv->head_dim < 8 || kv->head_dim_v < 8 || (kv->head_dim % 8) || (kv->head_dim_v % 8))
    return fail(SE_ERR_INVALID_ARG, fn, "head dims must be positive multiples of 8");
  if (kv->row_stride_k < kv->head_dim || kv->row_stride_v < kv->head_dim_v || (kv->row_stride_k % 8) ||
      (kv->row_stride_v % 8))
    return fail(SE_ERR_INVALID_ARG, fn, "row strides must cover the head dims and be multiples of 8");
  if ((long long)kv->num_pages * kv->num_kv_heads * se::kPageSize >= (1ll << 31))
    return fail(SE_ERR_UNSUPPORTED, fn, "cache holds 2^31 or more token rows");
  if (kv->head_dim != 128 && kv->head_dim != 576) return fail(SE_ERR_UNSUPPORTED, fn, "head_dim must be 128 or 576");
  return SE_OK;
}

KvView view_of(const se_paged_kv_t* kv) {
  KvView v;
  v.k = static_cast<const uint16_t*>(kv->k);
  v.v = static_cast<const uint16_t*>(kv->v);
  v.summary = static_cast<uint16_t*>(kv->summary);
  v.num_pages = kv->num_pages;
  v.num_kv_heads = kv->num_kv_heads;
  v.head_dim = kv->head_dim;
  v.head_dim_v = kv->head_dim_v;
  v.row_stride_k = kv->row_stride_k;
  v.row_stride_v = kv->row_stride_v;
  return v;
}

size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

int score_stride_for(int max_seq_len) { return pages_of(max_seq_len) > 0 ? pages_of(max_seq_len) : 1; }

se_status_t check_batch_common(const char* fn, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* seq_lens, int32_t batch, int32_t max_seq_len) {
  if (batch < 0) return fail(SE_ERR_INVALID_ARG, fn, "batch < 0");
  if (max_seq_len < 0) return fail(SE_ERR_INVALID_ARG, fn, "max_seq_len < 0");
  if (batch > 0 && (!block_table || !seq_lens)) return fail(SE_ERR_INVALID_ARG, fn, "block_table/seq_lens NULL");
  if (bt_stride < pages_of(max_seq_len) || bt_stride < 1)
    return fail(SE_ERR_INVALID_ARG, fn, "bt_stride < ceil(max_seq_len / 16)");
  return SE_OK;
}

}  // namespace

extern "C" {

const char* se_status_string(int status) {
  switch (status) {
    case SE_OK: return "SE_OK";
    case SE_ERR_INVALID_ARG: return "SE_ERR_INVALID_ARG";
    case SE_ERR_UNSUPPORTED: return "SE_ERR_UNSUPPORTED";
    case SE_ERR_WORKSPACE: return "SE_ERR_WORKSPACE";
    case SE_ERR_CUDA: return "SE_ERR_CUDA";
    case SE_ERR_DEVICE: return "SE_ERR_DEVICE";
    default: return "SE_ERR_UNKNOWN";
  }
}

const char* se_last_error_detail(void) { return g_detail; }

se_status_t se_read_device_error(uint32_t* out, int clear) {
  if (!out) return fail(SE_ERR_INVALID_ARG, "se_read_device_error", "out is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail("se_read_device_error", e);
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, se_device_error_word, sizeof(v));
  if (e != cudaSuccess) return cuda_fail("se_read_device_error", e);
  if (clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(se_device_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail("se_read_device_error", e);
  }
  *out = v;
  return SE_OK;
}

se_status_t se_quest_build_summaries(const se_paged_kv_t* kv, const int32_t* block_table, int32_t bt_stride,
                                     const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                     void* stream) {
  static const char* fn = "se_quest_build_summaries";
  se_status_t st = check_kv(fn, kv, true);
  if (st != SE_OK) return st;
  st = check_batch_common(fn, block_table, bt_stride, seq_lens, batch, max_seq_len);
  if (st != SE_OK) return st;
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  e = se::launch_build_summaries(view_of(kv), block_table, bt_stride, seq_lens, batch, max_seq_len, d->err,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

se_status_t se_quest_update_summaries(const se_paged_kv_t* kv, const void* k_new, const void* v_new,
                                      const int32_t* block_table, int32_t bt_stride,
                                      const int32_t* seq_lens_before, int32_t batch, void* stream) {
  return se_quest_update_summaries_ex(kv, k_new, v_new, block_table, bt_stride, seq_lens_before, batch, 0u, stream);
}

se_status_t se_quest_update_summaries_ex(const se_paged_kv_t* kv, const void* k_new, const void* v_new,
                                         const int32_t* block_table, int32_t bt_stride,
                                         const int32_t* seq_lens_before, int32_t batch, uint32_t flags,
                                         void* stream) {
  static const char* fn = "se_quest_update_summaries_ex";
  if (flags & ~(uint32_t)SE_APPEND_OVERLAP_PREVIOUS) return fail(SE_ERR_INVALID_ARG, fn, "unknown flags");
  se_status_t st = check_kv(fn, kv, false);  // summary NULL: the K/V rows only
  if (st != SE_OK) return st;
  if (batch < 0) return fail(SE_ERR_INVALID_ARG, fn, "batch < 0");
  if (batch > 0 && (!k_new || !block_table || !seq_lens_before))
    return fail(SE_ERR_INVALID_ARG, fn, "k_new/block_table/seq_lens_before NULL");
  if (bt_stride < 1) return fail(SE_ERR_INVALID_ARG, fn, "bt_stride < 1");
  const bool latent = kv->v == kv->k;
  if (!latent && batch > 0 && !v_new) return fail(SE_ERR_INVALID_ARG, fn, "v_new NULL for a separate value cache");
  if (latent && v_new) return fail(SE_ERR_INVALID_ARG, fn, "v_new must be NULL when kv->v == kv->k");
  if (!aligned16(k_new) || !aligned16(v_new)) return fail(SE_ERR_INVALID_ARG, fn, "k_new/v_new not 16-byte aligned");
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  e = se::launch_append_update(view_of(kv), static_cast<uint16_t*>(kv->k), static_cast<uint16_t*>(kv->v),
                               static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
                               block_table, bt_stride, seq_lens_before, batch,
                               (flags & SE_APPEND_OVERLAP_PREVIOUS) != 0, d->err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

namespace {

// Shared body of se_quest_score_pages and se_quest_score_pages_ws (pn: the
// multiplier workspace, or null).
se_status_t score_pages_impl(const char* fn, const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                             const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens, int32_t batch,
                             int32_t max_seq_len, float* scores, int32_t score_stride, float* pn, void* stream) {
  se_status_t st = check_kv(fn, kv, true);
  if (st != SE_OK) return st;
  st = check_batch_common(fn, block_table, bt_stride, seq_lens, batch, max_seq_len);
  if (st != SE_OK) return st;
  if (num_q_heads < 1 || num_q_heads % kv->num_kv_heads)
    return fail(SE_ERR_INVALID_ARG, fn, "num_q_heads must be a positive multiple of num_kv_heads");
  if (batch > 0 && (!q || !scores)) return fail(SE_ERR_INVALID_ARG, fn, "q/scores NULL");
  if (!aligned16(q) || !aligned16(scores)) return fail(SE_ERR_INVALID_ARG, fn, "q/scores not 16-byte aligned");
  if (score_stride < score_stride_for(max_seq_len)) return fail(SE_ERR_INVALID_ARG, fn, "score_stride too small");
  if (!se::score_pages_supported(kv->num_kv_heads, kv->head_dim))
    return fail(SE_ERR_UNSUPPORTED, fn, "scoring needs head_dim 128 with 1..8 KV heads, or head_dim 576 with one");
  if (batch > 16384) return fail(SE_ERR_UNSUPPORTED, fn, "batch > 16384");
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  e = se::launch_score_pages(view_of(kv), static_cast<const uint16_t*>(q), num_q_heads, block_table, bt_stride,
                             seq_lens, batch, max_seq_len, scores, score_stride, pn, d->sm_count, d->err,
                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

}  // namespace

se_status_t se_quest_score_pages(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                 const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                 int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                                 void* stream) {
  return score_pages_impl("se_quest_score_pages", kv, q, num_q_heads, block_table, bt_stride, seq_lens, batch,
                          max_seq_len, scores, score_stride, nullptr, stream);
}

size_t se_quest_score_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t head_dim) {
  if (batch < 0 || num_kv_heads < 0 || head_dim < 0) return 0;
  return round16(se::score_pn_bytes(batch, num_kv_heads, head_dim));
}

se_status_t se_quest_score_pages_ws(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                    const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                    int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  static const char* fn = "se_quest_score_pages_ws";
  if (!kv) return fail(SE_ERR_INVALID_ARG, fn, "kv is NULL");
  if (batch < 0) return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  const size_t need = se_quest_score_workspace_size(batch, kv->num_kv_heads, kv->head_dim);
  if (workspace_bytes < need) return fail(SE_ERR_WORKSPACE, fn, "workspace too small");
  if (need > 0 && !workspace) return fail(SE_ERR_INVALID_ARG, fn, "workspace NULL");
  if (!aligned16(workspace)) return fail(SE_ERR_INVALID_ARG, fn, "workspace not 16-byte aligned");
  return score_pages_impl(fn, kv, q, num_q_heads, block_table, bt_stride, seq_lens, batch, max_seq_len, scores,
                          score_stride, need > 0 ? static_cast<float*>(workspace) : nullptr, stream);
}

se_status_t se_quest_topk_pages_windowed(const float* scores, int32_t score_stride, const int32_t* seq_lens,
                                         int32_t batch, int32_t num_kv_heads, int32_t max_seq_len, int32_t topk_pages,
                                         int32_t sink_tokens, int32_t recent_tokens, int32_t* out_pages,
                                         int32_t* out_counts, int32_t sel_stride, void* stream) {
  static const char* fn = "se_quest_topk_pages_windowed";
  if (batch < 0 || num_kv_heads < 1 || max_seq_len < 0) return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  if (topk_pages < 1) return fail(SE_ERR_INVALID_ARG, fn, "topk_pages < 1");
  if (sink_tokens < 0 || recent_tokens < 0 || sink_tokens > (1 << 30) || recent_tokens > (1 << 30))
    return fail(SE_ERR_INVALID_ARG, fn, "sink_tokens / recent_tokens out of range");
  if ((long long)sel_stride < se_quest_kept_pages_max(topk_pages, sink_tokens, recent_tokens))
    return fail(SE_ERR_INVALID_ARG, fn, "sel_stride < se_quest_kept_pages_max(topk_pages, sink, recent)");
  if (score_stride < score_stride_for(max_seq_len)) return fail(SE_ERR_INVALID_ARG, fn, "score_stride too small");
  if (batch > 0 && (!scores || !seq_lens || !out_pages || !out_counts))
    return fail(SE_ERR_INVALID_ARG, fn, "NULL pointer");
  if (!aligned16(scores) || !aligned16(out_pages) || !aligned16(out_counts))
    return fail(SE_ERR_INVALID_ARG, fn, "pointers must be 16-byte aligned");
  if (se::topk_smem_bytes(max_seq_len) > 200 * 1024)
    return fail(SE_ERR_UNSUPPORTED, fn, "more than 51200 candidate pages per request");
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  e = se::launch_topk_pages(scores, score_stride, seq_lens, batch, num_kv_heads, max_seq_len, topk_pages,
                            sink_tokens, recent_tokens, out_pages, out_counts, sel_stride, d->err,
                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

se_status_t se_quest_topk_pages(const float* scores, int32_t score_stride, const int32_t* seq_lens,
                                int32_t batch, int32_t num_kv_heads, int32_t max_seq_len, int32_t topk_pages,
                                int32_t* out_pages, int32_t* out_counts, int32_t sel_stride, void* stream) {
  return se_quest_topk_pages_windowed(scores, score_stride, seq_lens, batch, num_kv_heads, max_seq_len, topk_pages,
                                      0, 0, out_pages, out_counts, sel_stride, stream);
}

long long se_quest_kept_pages_max(int32_t topk_pages, int32_t sink_tokens, int32_t recent_tokens) {
  if (topk_pages < 0 || sink_tokens < 0 || recent_tokens < 0) return -1;
  const long long ps = se::kPageSize;
  return (sink_tokens + ps - 1) / ps + topk_pages + (recent_tokens + ps - 1) / ps + 1;
}

size_t se_quest_select_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len) {
  if (batch < 0 || num_kv_heads < 0 || max_seq_len < 0) return 0;
  return round16((size_t)batch * num_kv_heads * score_stride_for(max_seq_len) * sizeof(float));
}

se_status_t se_quest_select_pages_windowed(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                           const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                           int32_t batch, int32_t max_seq_len, int32_t topk_pages,
                                           int32_t sink_tokens, int32_t recent_tokens, int32_t* out_pages,
                                           int32_t* out_counts, int32_t sel_stride, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  static const char* fn = "se_quest_select_pages_windowed";
  if (!kv) return fail(SE_ERR_INVALID_ARG, fn, "kv is NULL");
  if (batch < 0 || max_seq_len < 0) return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  const size_t need = se_quest_select_workspace_size(batch, kv->num_kv_heads, max_seq_len);
  if (workspace_bytes < need) return fail(SE_ERR_WORKSPACE, fn, "workspace too small");
  if (need > 0 && !workspace) return fail(SE_ERR_INVALID_ARG, fn, "workspace NULL");
  if (topk_pages < 1 || sink_tokens < 0 || recent_tokens < 0 ||
      (long long)sel_stride < se_quest_kept_pages_max(topk_pages, sink_tokens, recent_tokens))
    return fail(SE_ERR_INVALID_ARG, fn, "topk_pages < 1, negative window or sel_stride too small");
  float* scores = static_cast<float*>(workspace);
  const int stride = score_stride_for(max_seq_len);
  se_status_t st = se_quest_score_pages(kv, q, num_q_heads, block_table, bt_stride, seq_lens, batch, max_seq_len,
                                        scores, stride, stream);
  if (st != SE_OK) return st;
  return se_quest_topk_pages_windowed(scores, stride, seq_lens, batch, kv->num_kv_heads, max_seq_len, topk_pages,
                                      sink_tokens, recent_tokens, out_pages, out_counts, sel_stride, stream);
}

se_status_t se_quest_select_pages(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                  const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                  int32_t batch, int32_t max_seq_len, int32_t topk_pages, int32_t* out_pages,
                                  int32_t* out_counts, int32_t sel_stride, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return se_quest_select_pages_windowed(kv, q, num_q_heads, block_table, bt_stride, seq_lens, batch, max_seq_len,
                                        topk_pages, 0, 0, out_pages, out_counts, sel_stride, workspace,
                                        workspace_bytes, stream);
}

se_status_t se_quest_fused_step(const se_paged_kv_t* kv, const void* k_new, const void* v_new, const void* q,
                                int32_t num_q_heads, const int32_t* block_table, int32_t bt_stride,
                                const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, int32_t topk_pages,
                                int32_t sink_tokens, int32_t recent_tokens, float sm_scale, void* out,
                                float* out_lse, int32_t* sel_pages, int32_t* sel_counts, int32_t sel_stride,
                                void* stream) {
  static const char* fn = "se_quest_fused_step";
  se_status_t st = check_kv(fn, kv, true);
  if (st != SE_OK) return st;
  if (batch < 0 || max_seq_len < 0 || bt_stride < 1) return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  if (num_q_heads < 1 || num_q_heads % kv->num_kv_heads)
    return fail(SE_ERR_INVALID_ARG, fn, "num_q_heads must be a positive multiple of num_kv_heads");
  if (kv->head_dim != 128 || kv->head_dim_v != 128 || kv->v == kv->k || num_q_heads / kv->num_kv_heads > 16)
    return fail(SE_ERR_UNSUPPORTED, fn, "head_dim = head_dim_v = 128, separate K and V, <= 16 query heads per KV head");
  if (topk_pages < 1 || sink_tokens < 0 || recent_tokens < 0)
    return fail(SE_ERR_INVALID_ARG, fn, "topk_pages < 1 or negative window");
  const long long kept_max = se_quest_kept_pages_max(topk_pages, sink_tokens, recent_tokens);
  if ((long long)sel_stride < kept_max) return fail(SE_ERR_INVALID_ARG, fn, "sel_stride < se_quest_kept_pages_max");
  if (kept_max > se::fused_max_kept()) return fail(SE_ERR_UNSUPPORTED, fn, "more than 2048 kept pages");
  if (pages_of(max_seq_len) - 1 > se::fused_max_candidates())
    return fail(SE_ERR_UNSUPPORTED, fn, "more than 8192 candidate pages per request");
  if (bt_stride < pages_of(max_seq_len)) return fail(SE_ERR_INVALID_ARG, fn, "bt_stride < pages of max_seq_len");
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(SE_ERR_INVALID_ARG, fn, "k_new and v_new: both or neither");
  if (batch > 0 && (!q || !block_table || !seq_lens || !out || !sel_pages || !sel_counts))
    return fail(SE_ERR_INVALID_ARG, fn, "NULL pointer");
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(sel_pages) ||
      !aligned16(out_lse))
    return fail(SE_ERR_INVALID_ARG, fn, "pointers must be 16-byte aligned");
  if (!std::isfinite(sm_scale)) return fail(SE_ERR_INVALID_ARG, fn, "sm_scale not finite");
  if (batch == 0) return SE_OK;
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  e = se::launch_quest_fused(view_of(kv), static_cast<uint16_t*>(kv->k), static_cast<uint16_t*>(kv->v),
                             static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
                             static_cast<const uint16_t*>(q), num_q_heads, block_table, bt_stride, seq_lens, batch,
                             max_seq_len, topk_pages, sink_tokens, recent_tokens, sm_scale,
                             static_cast<uint16_t*>(out), out_lse, sel_pages, sel_counts, sel_stride, d->sm_count,
                             d->err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

se_status_t se_sparse_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t head_dim_v, int32_t sel_stride, int32_t* nsplit,
                                  int32_t* pages_per_split, int32_t* launches) {
  static const char* fn = "se_sparse_decode_plan";
  if (!nsplit || !pages_per_split || !launches) return fail(SE_ERR_INVALID_ARG, fn, "NULL output");
  if (batch < 0 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads || sel_stride < 1)
    return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  const bool mla = se::mla_decode_supported(num_kv_heads, head_dim, head_dim_v, num_q_heads);
  if (!(head_dim == 128 && head_dim_v == 128 && num_q_heads / num_kv_heads <= 16) && !mla)
    return fail(SE_ERR_UNSUPPORTED, fn, "shape not implemented");
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  const se::DecodePlan plan = mla ? se::plan_mla_decode(sel_stride, d->sm_count)
                                  : se::plan_gqa_decode(batch, num_kv_heads, sel_stride, d->sm_count);
  *nsplit = plan.nsplit;
  *pages_per_split = plan.pages_per_split;
  *launches = batch == 0 ? 0 : (mla ? 2 : 1);  // latent: the decode kernel and the split merge
  return SE_OK;
}

size_t se_sparse_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim_v, int32_t sel_stride) {
  if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim_v < 1 || sel_stride < 1) return 0;
  // The split layout does not depend on the device. A latent cache is the one
  // shape with a 512-wide value and one KV head.
  if (num_kv_heads == 1 && head_dim_v == 512 && se::mla_decode_supported(1, 576, 512, num_q_heads))
    return round16(se::mla_decode_workspace_bytes(batch, num_q_heads, se::plan_mla_decode(sel_stride, 1)));
  const se::DecodePlan plan = se::plan_gqa_decode(batch, num_kv_heads, sel_stride, 1);
  return round16(se::gqa_decode_workspace_bytes(batch, num_q_heads, head_dim_v, plan));
}

se_status_t se_sparse_paged_decode(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                   const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                   int32_t batch, const int32_t* sel_pages, const int32_t* sel_counts,
                                   int32_t sel_stride, float sm_scale, void* out, float* out_lse,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  static const char* fn = "se_sparse_paged_decode";
  bool mla = false;
  se_status_t st = se::check_decode_call(fn, kv, q, num_q_heads, block_table, bt_stride, seq_lens, batch, sel_pages,
                                         sel_counts, sel_stride, sm_scale, out, out_lse, &mla);
  if (st != SE_OK) return st;
  if (!aligned16(workspace)) return fail(SE_ERR_INVALID_ARG, fn, "workspace must be 16-byte aligned");
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (mla) {
    const se::DecodePlan plan = se::plan_mla_decode(sel_stride, d->sm_count);
    const size_t need = se::mla_decode_workspace_bytes(batch, num_q_heads, plan);
    if (workspace_bytes < need) return fail(SE_ERR_WORKSPACE, fn, "workspace too small");
    if (need > 0 && !workspace) return fail(SE_ERR_INVALID_ARG, fn, "workspace NULL");
    if ((size_t)batch > se::mla_decode_max_items())
      return fail(SE_ERR_UNSUPPORTED, fn, "too many requests for one launch");
    if (batch == 0) return SE_OK;
    // Tile copies: 8 rows x all 9 chunks of 64 dims (half a page) of the cache,
    // 64 dims x all heads of the queries.
    CUtensorMap kvmap, qmap;
    if (!encode_row_chunks_map(&kvmap, kv->k, (long long)kv->num_pages * se::kPageSize, kv->row_stride_k,
                               kv->head_dim / 64, se::kPageSize / 2) ||
        !encode_page_map(&qmap, q, (long long)batch * num_q_heads, kv->head_dim, kv->head_dim, num_q_heads))
      return fail(SE_ERR_CUDA, fn, "cuTensorMapEncodeTiled failed");
    e = se::launch_mla_decode(kvmap, qmap, view_of(kv), static_cast<const uint16_t*>(q), num_q_heads, block_table,
                              bt_stride,
                              seq_lens, batch, sel_pages, sel_counts, sel_stride, sm_scale,
                              static_cast<uint16_t*>(out), out_lse, workspace, plan, d->err,
                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
  }
  const se::DecodePlan plan = se::plan_gqa_decode(batch, kv->num_kv_heads, sel_stride, d->sm_count);
  const size_t need = se::gqa_decode_workspace_bytes(batch, num_q_heads, kv->head_dim_v, plan);
  if (workspace_bytes < need) return fail(SE_ERR_WORKSPACE, fn, "workspace too small");
  if (need > 0 && !workspace) return fail(SE_ERR_INVALID_ARG, fn, "workspace NULL");
  if ((size_t)batch * kv->num_kv_heads > se::gqa_decode_max_items())
    return fail(SE_ERR_UNSUPPORTED, fn, "too many (request, KV head) items for one launch");
  if (batch == 0) return SE_OK;
  e = se::launch_gqa_decode(view_of(kv), static_cast<const uint16_t*>(q), num_q_heads, block_table, bt_stride,
                            seq_lens, batch, sel_pages, sel_counts, sel_stride, sm_scale,
                            static_cast<uint16_t*>(out), out_lse, workspace, plan, d->err,
                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}


}  // extern "C"

// ------------------------------------------------------------------ SnapKV
namespace {

se_status_t check_snapkv_shape(const char* fn, const se_paged_kv_t* kv, int32_t num_q_heads, int32_t window,
                               int32_t batch, int32_t max_len) {
  se_status_t st = check_kv(fn, kv, false);
  if (st != SE_OK) return st;
  if (kv->head_dim != 128 || kv->head_dim_v != 128)
    return fail(SE_ERR_UNSUPPORTED, fn, "SnapKV needs head_dim = head_dim_v = 128");
  if (num_q_heads < 1 || num_q_heads % kv->num_kv_heads)
    return fail(SE_ERR_INVALID_ARG, fn, "num_q_heads must be a positive multiple of num_kv_heads");
  if (window < 1) return fail(SE_ERR_INVALID_ARG, fn, "window < 1");
  if (window * (num_q_heads / kv->num_kv_heads) > 128)
    return fail(SE_ERR_UNSUPPORTED, fn, "window x query heads per KV head must be <= 128");
  if (batch < 0 || max_len < 0) return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  if ((long long)batch * kv->num_kv_heads > 4096) return fail(SE_ERR_UNSUPPORTED, fn, "more than 4096 pairs");
  return SE_OK;
}

int snap_score_stride(int max_len, int window) { return max_len - window > 1 ? max_len - window : 1; }

}  // namespace

extern "C" {

size_t se_snapkv_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t window, int32_t max_prompt_len) {
  if (batch < 0 || num_kv_heads < 1 || window < 1 || max_prompt_len < 0) return 0;
  const int pairs = batch * num_kv_heads;
  return round16(se::snapkv_part_bytes(pairs, max_prompt_len)) +
         round16((size_t)pairs * snap_score_stride(max_prompt_len, window) * sizeof(float));
}

se_status_t se_snapkv_window_scores(const se_paged_kv_t* src, const void* q_window, int32_t num_q_heads,
                                    int32_t window, const int32_t* block_table, int32_t bt_stride,
                                    const int32_t* prompt_lens, int32_t batch, int32_t max_prompt_len, float sm_scale,
                                    float* scores, int32_t score_stride, float* row_lse, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  static const char* fn = "se_snapkv_window_scores";
  se_status_t st = check_snapkv_shape(fn, src, num_q_heads, window, batch, max_prompt_len);
  if (st != SE_OK) return st;
  st = check_batch_common(fn, block_table, bt_stride, prompt_lens, batch, max_prompt_len);
  if (st != SE_OK) return st;
  if (batch > 0 && (!q_window || !scores)) return fail(SE_ERR_INVALID_ARG, fn, "q_window/scores NULL");
  if (!aligned16(q_window) || !aligned16(scores) || !aligned16(row_lse) || !aligned16(workspace))
    return fail(SE_ERR_INVALID_ARG, fn, "pointers must be 16-byte aligned");
  if (score_stride < snap_score_stride(max_prompt_len, window))
    return fail(SE_ERR_INVALID_ARG, fn, "score_stride < max_prompt_len - window");
  if (!std::isfinite(sm_scale)) return fail(SE_ERR_INVALID_ARG, fn, "sm_scale not finite");
  const size_t need = se::snapkv_part_bytes(batch * src->num_kv_heads, max_prompt_len);
  if (workspace_bytes < need) return fail(SE_ERR_WORKSPACE, fn, "workspace too small");
  if (need > 0 && !workspace) return fail(SE_ERR_INVALID_ARG, fn, "workspace NULL");
  if (batch == 0) return SE_OK;
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  CUtensorMap kmap, qmap;
  const long long rows = (long long)src->num_pages * src->num_kv_heads * se::kPageSize;
  if (!encode_row_chunks_map(&kmap, src->k, rows > 0 ? rows : 1, src->row_stride_k, 2, se::kPageSize) ||
      !encode_window_map(&qmap, q_window, batch, window, num_q_heads, num_q_heads / src->num_kv_heads))
    return fail(SE_ERR_CUDA, fn, "cuTensorMapEncodeTiled failed");
  e = se::launch_snapkv_scores(kmap, qmap, view_of(src), static_cast<const uint16_t*>(q_window), num_q_heads, window,
                               block_table, bt_stride, prompt_lens, batch, max_prompt_len, sm_scale, scores,
                               score_stride, row_lse, workspace, d->sm_count, d->err,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

se_status_t se_debug_snapkv_wait_probe(uint32_t limit_us) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(SE_ERR_INVALID_ARG, "se_debug_snapkv_wait_probe", "limit_us must be in 1 .. 1000000");
  se::set_snapkv_wait_probe(limit_us);
  return SE_OK;
}

se_status_t se_snapkv_select_windowed(const float* scores, int32_t score_stride, const int32_t* prompt_lens,
                                      int32_t batch, int32_t num_kv_heads, int32_t window, int32_t max_prompt_len,
                                      int32_t pool_kernel, int32_t keep_topk, int32_t sink_tokens,
                                      int32_t recent_tokens, int32_t* kept_pos, int32_t kept_stride,
                                      int32_t* kept_counts, void* stream) {
  static const char* fn = "se_snapkv_select_windowed";
  if (batch < 0 || num_kv_heads < 1 || window < 1 || max_prompt_len < 0) return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  if (pool_kernel < 1 || pool_kernel % 2 == 0) return fail(SE_ERR_INVALID_ARG, fn, "pool_kernel must be odd");
  if (keep_topk < 1) return fail(SE_ERR_INVALID_ARG, fn, "keep_topk < 1");
  if (sink_tokens < 0 || recent_tokens < window || sink_tokens > (1 << 30) || recent_tokens > (1 << 30))
    return fail(SE_ERR_INVALID_ARG, fn, "sink_tokens < 0 or recent_tokens < window");
  if ((long long)kept_stride < (long long)sink_tokens + keep_topk + recent_tokens)
    return fail(SE_ERR_INVALID_ARG, fn, "kept_stride < sink_tokens + keep_topk + recent_tokens");
  if (score_stride < snap_score_stride(max_prompt_len, window))
    return fail(SE_ERR_INVALID_ARG, fn, "score_stride < max_prompt_len - window");
  if (max_prompt_len - window > se::snapkv_select_max_candidates())
    return fail(SE_ERR_UNSUPPORTED, fn, "more than 45056 candidate positions per request");
  if (batch > 0 && (!scores || !prompt_lens || !kept_pos || !kept_counts))
    return fail(SE_ERR_INVALID_ARG, fn, "NULL pointer");
  if (!aligned16(scores) || !aligned16(kept_pos) || !aligned16(kept_counts))
    return fail(SE_ERR_INVALID_ARG, fn, "pointers must be 16-byte aligned");
  if (batch == 0) return SE_OK;
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  e = se::launch_snapkv_select(scores, score_stride, prompt_lens, batch, num_kv_heads, window, max_prompt_len,
                               pool_kernel, keep_topk, sink_tokens, recent_tokens, kept_pos, kept_stride, kept_counts,
                               d->err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

se_status_t se_snapkv_select(const float* scores, int32_t score_stride, const int32_t* prompt_lens, int32_t batch,
                             int32_t num_kv_heads, int32_t window, int32_t max_prompt_len, int32_t pool_kernel,
                             int32_t keep_topk, int32_t* kept_pos, int32_t kept_stride, int32_t* kept_counts,
                             void* stream) {
  return se_snapkv_select_windowed(scores, score_stride, prompt_lens, batch, num_kv_heads, window, max_prompt_len,
                                   pool_kernel, keep_topk, 0, window, kept_pos, kept_stride, kept_counts, stream);
}

se_status_t se_snapkv_compact(const se_paged_kv_t* src, const int32_t* src_block_table, int32_t src_bt_stride,
                              const int32_t* prompt_lens, int32_t batch, const se_paged_kv_t* dst,
                              const int32_t* dst_block_table, int32_t dst_bt_stride, const int32_t* kept_pos,
                              int32_t kept_stride, const int32_t* kept_counts, void* stream) {
  static const char* fn = "se_snapkv_compact";
  se_status_t st = check_kv(fn, src, false);
  if (st != SE_OK) return st;
  st = check_kv(fn, dst, false);
  if (st != SE_OK) return st;
  if (src->head_dim != 128 || src->head_dim_v != 128 || dst->head_dim != 128 || dst->head_dim_v != 128 ||
      dst->row_stride_k != 128 || dst->row_stride_v != 128 || dst->num_kv_heads != src->num_kv_heads)
    return fail(SE_ERR_UNSUPPORTED, fn, "compaction needs d 128 caches with dense destination rows");
  if (batch < 0 || kept_stride < 1 || src_bt_stride < 1 || dst_bt_stride < 1)
    return fail(SE_ERR_INVALID_ARG, fn, "bad sizes");
  if (batch > 0 && (!src_block_table || !prompt_lens || !dst_block_table || !kept_pos || !kept_counts))
    return fail(SE_ERR_INVALID_ARG, fn, "NULL pointer");
  if (batch == 0) return SE_OK;
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  e = se::launch_snapkv_gather(view_of(src), static_cast<uint16_t*>(dst->k), static_cast<uint16_t*>(dst->v),
                               dst->num_pages, src_block_table, src_bt_stride, dst_block_table, dst_bt_stride,
                               prompt_lens, batch, kept_pos, kept_stride, kept_counts, d->err,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SE_OK : cuda_fail(fn, e);
}

se_status_t se_snapkv_score_and_compact_windowed(const se_paged_kv_t* src, const void* q_window,
                                                 int32_t num_q_heads, int32_t window, const int32_t* src_block_table,
                                                 int32_t src_bt_stride, const int32_t* prompt_lens, int32_t batch,
                                                 int32_t max_prompt_len, int32_t pool_kernel, int32_t keep_topk,
                                                 int32_t sink_tokens, int32_t recent_tokens, float sm_scale,
                                                 const se_paged_kv_t* dst, const int32_t* dst_block_table,
                                                 int32_t dst_bt_stride, int32_t* kept_pos, int32_t kept_stride,
                                                 int32_t* kept_counts, void* workspace, size_t workspace_bytes,
                                                 void* stream) {
  static const char* fn = "se_snapkv_score_and_compact_windowed";
  if (!src) return fail(SE_ERR_INVALID_ARG, fn, "src is NULL");
  const size_t need = se_snapkv_workspace_size(batch, src->num_kv_heads, window, max_prompt_len);
  if (workspace_bytes < need) return fail(SE_ERR_WORKSPACE, fn, "workspace too small");
  if (need > 0 && !workspace) return fail(SE_ERR_INVALID_ARG, fn, "workspace NULL");
  const size_t part = round16(se::snapkv_part_bytes(batch * src->num_kv_heads, max_prompt_len));
  float* scores = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + part);
  const int stride = snap_score_stride(max_prompt_len, window);
  se_status_t st = se_snapkv_window_scores(src, q_window, num_q_heads, window, src_block_table, src_bt_stride,
                                           prompt_lens, batch, max_prompt_len, sm_scale, scores, stride, nullptr,
                                           workspace, part, stream);
  if (st != SE_OK) return st;
  st = se_snapkv_select_windowed(scores, stride, prompt_lens, batch, src->num_kv_heads, window, max_prompt_len,
                                 pool_kernel, keep_topk, sink_tokens, recent_tokens, kept_pos, kept_stride,
                                 kept_counts, stream);
  if (st != SE_OK) return st;
  return se_snapkv_compact(src, src_block_table, src_bt_stride, prompt_lens, batch, dst, dst_block_table,
                           dst_bt_stride, kept_pos, kept_stride, kept_counts, stream);
}

se_status_t se_snapkv_score_and_compact(const se_paged_kv_t* src, const void* q_window, int32_t num_q_heads,
                                        int32_t window, const int32_t* src_block_table, int32_t src_bt_stride,
                                        const int32_t* prompt_lens, int32_t batch, int32_t max_prompt_len,
                                        int32_t pool_kernel, int32_t keep_topk, float sm_scale,
                                        const se_paged_kv_t* dst, const int32_t* dst_block_table,
                                        int32_t dst_bt_stride, int32_t* kept_pos, int32_t kept_stride,
                                        int32_t* kept_counts, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  return se_snapkv_score_and_compact_windowed(src, q_window, num_q_heads, window, src_block_table, src_bt_stride,
                                              prompt_lens, batch, max_prompt_len, pool_kernel, keep_topk, 0, window,
                                              sm_scale, dst, dst_block_table, dst_bt_stride, kept_pos, kept_stride,
                                              kept_counts, workspace, workspace_bytes, stream);
}

}  // extern "C"

// Internal accessors for entry points defined in other translation units.
namespace se {

cudaError_t device_context(int* sm_count, unsigned** err) {
  DeviceInfo* d = nullptr;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return e;
  *sm_count = d->sm_count;
  *err = d->err;
  return cudaSuccess;
}


void set_error_detail(const char* fn, const char* what) { fail(SE_OK, fn, what); }

se_status_t check_decode_call(const char* fn, const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                              const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens, int32_t batch,
                              const int32_t* sel_pages, const int32_t* sel_counts, int32_t sel_stride,
                              float sm_scale, const void* out, const float* out_lse, bool* latent) {
  se_status_t st = check_kv(fn, kv, false);
  if (st != SE_OK) return st;
  if (batch < 0) return fail(SE_ERR_INVALID_ARG, fn, "batch < 0");
  if (num_q_heads < 1 || num_q_heads % kv->num_kv_heads)
    return fail(SE_ERR_INVALID_ARG, fn, "num_q_heads must be a positive multiple of num_kv_heads");
  if (sel_stride < 1 || bt_stride < 1) return fail(SE_ERR_INVALID_ARG, fn, "sel_stride/bt_stride < 1");
  if (batch > 0 && (!q || !block_table || !seq_lens || !sel_pages || !sel_counts || !out))
    return fail(SE_ERR_INVALID_ARG, fn, "NULL pointer");
  if (!aligned16(q) || !aligned16(out) || !aligned16(out_lse) || !aligned16(sel_pages))
    return fail(SE_ERR_INVALID_ARG, fn, "pointers must be 16-byte aligned");
  if (!std::isfinite(sm_scale)) return fail(SE_ERR_INVALID_ARG, fn, "sm_scale not finite");
  const int group = num_q_heads / kv->num_kv_heads;
  const bool gqa = kv->head_dim == 128 && kv->head_dim_v == 128 && group <= 16;
  const bool mla = mla_decode_supported(kv->num_kv_heads, kv->head_dim, kv->head_dim_v, num_q_heads);
  if (!gqa && !mla)
    return fail(SE_ERR_UNSUPPORTED, fn,
                "head_dim = head_dim_v = 128 with <= 16 query heads per KV head, or a latent cache (576/512, one "
                "KV head, 16..64 query heads in multiples of 16)");
  if (mla && kv->v != kv->k) return fail(SE_ERR_INVALID_ARG, fn, "a latent cache needs kv->v == kv->k");
  *latent = mla;
  return SE_OK;
}

}  // namespace se
