// Internal declarations shared by the host entry points (api.cu) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/sparse_engine.h"

namespace se {

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream finishes; it waits (pdl_wait) before
// touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kPageSize = 16;
// Bounded waits: an mbarrier wait gives up after this much wall time or polls.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitLimitIters = 1u << 28;

// Device-visible copy of the cache layout (plain values, passed by value).
struct KvView {
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* summary;
  int32_t num_pages;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t head_dim_v;
  int32_t row_stride_k;
  int32_t row_stride_v;
};

// ---- quest_summary.cu
cudaError_t launch_build_summaries(const KvView& kv, const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, unsigned* err,
                                   cudaStream_t stream);
// overlap_previous: the kernel may run alongside the previous kernel of the
// stream (it must touch nothing that kernel reads or writes) and completes after it.
cudaError_t launch_append_update(const KvView& kv, uint16_t* k_mut, uint16_t* v_mut, const uint16_t* k_new,
                                 const uint16_t* v_new, const int32_t* block_table, int32_t bt_stride,
                                 const int32_t* seq_lens_before, int32_t batch, bool overlap_previous,
                                 unsigned* err, cudaStream_t stream);

// ---- quest_score.cu
bool score_pages_supported(int num_kv_heads, int head_dim);
// Bytes of the per-request multipliers (P and N) that pn_ws holds.
size_t score_pn_bytes(int32_t batch, int32_t num_kv_heads, int32_t head_dim);
// pn_ws (score_pn_bytes, 16-byte aligned) or null: with it, a first kernel
// reduces every request's queries once and the scoring kernel reads the result;
// without it, every CTA reduces the queries of the requests it scores.
cudaError_t launch_score_pages(const KvView& kv, const uint16_t* q, int32_t num_q_heads,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                               int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                               float* pn_ws, int sm_count, unsigned* err, cudaStream_t stream);
// ---- quest_topk.cu
// Top-k of the candidate pages: those holding none of the first sink_tokens and
// none of the last recent_tokens tokens (the last page always kept); the kept
// windows are written around the selection.
cudaError_t launch_topk_pages(const float* scores, int32_t score_stride, const int32_t* seq_lens, int32_t batch,
                              int32_t num_kv_heads, int32_t max_seq_len, int32_t topk, int32_t sink_tokens,
                              int32_t recent_tokens, int32_t* out_pages, int32_t* out_counts, int32_t sel_stride,
                              unsigned* err, cudaStream_t stream);
size_t topk_smem_bytes(int32_t max_seq_len);

// ---- sparse_decode.cu
struct DecodePlan {
  int32_t nsplit;           // most CTAs whose slices one item's pages can span (partial slots per row)
  int32_t pages_per_split;  // fewest selected pages per CTA slice
  int32_t grid;             // CTAs launched
};
DecodePlan plan_gqa_decode(int32_t batch, int32_t num_kv_heads, int32_t sel_stride, int sm_count);
size_t gqa_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim_v, const DecodePlan& plan);
// Byte offset in the workspace of the per-item arrival counters (batch x KV heads
// uint32, zero between calls: every call leaves them as it found them).
size_t gqa_decode_arrivals_offset(int32_t batch, int32_t num_q_heads, int32_t head_dim_v, const DecodePlan& plan);
size_t gqa_decode_max_items();
cudaError_t launch_gqa_decode(const KvView& kv, const uint16_t* q, int32_t num_q_heads, const int32_t* block_table,
                              int32_t bt_stride, const int32_t* seq_lens, int32_t batch, const int32_t* sel_pages,
                              const int32_t* sel_counts, int32_t sel_stride, float sm_scale, uint16_t* out,
                              float* out_lse, void* workspace, const DecodePlan& plan, unsigned* err,
                              cudaStream_t stream);

// ---- mla_decode.cu (latent cache: head_dim 576, value = first 512 dims, one KV head)
bool mla_decode_supported(int num_kv_heads, int head_dim, int head_dim_v, int num_q_heads);
DecodePlan plan_mla_decode(int32_t sel_stride, int sm_count);
size_t mla_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, const DecodePlan& plan);
size_t mla_decode_max_items();
// kvmap: the cache as rows of 576 bf16, boxes of 64 x 16; qmap: the queries as
// batch x num_q_heads rows of 576, boxes of 64 x num_q_heads (both 128-byte swizzle).
cudaError_t launch_mla_decode(const CUtensorMap& kvmap, const CUtensorMap& qmap, const KvView& kv, const uint16_t* q,
                              int32_t num_q_heads, const int32_t* block_table,
                              int32_t bt_stride, const int32_t* seq_lens, int32_t batch, const int32_t* sel_pages,
                              const int32_t* sel_counts, int32_t sel_stride, float sm_scale, uint16_t* out,
                              float* out_lse, void* workspace, const DecodePlan& plan, unsigned* err,
                              cudaStream_t stream);

// ---- quest_fused.cu: append + score + top-k + decode in one launch (a cluster per item)
int fused_max_candidates();
int fused_max_kept();
int fused_cluster_size(int items, int sm_count);
cudaError_t launch_quest_fused(const KvView& kv, uint16_t* k_mut, uint16_t* v_mut, const uint16_t* k_new,
                               const uint16_t* v_new, const uint16_t* q, int32_t num_q_heads,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens, int32_t batch,
                               int32_t max_seq_len, int32_t topk, int32_t sink_tokens, int32_t recent_tokens,
                               float sm_scale, uint16_t* out, float* out_lse, int32_t* sel, int32_t* sel_counts,
                               int32_t sel_stride, int sm_count, unsigned* err, cudaStream_t stream);

// ---- snapkv.cu
int snapkv_max_slices(int max_len);
size_t snapkv_part_bytes(int pairs, int max_len);
int snapkv_select_max_candidates();
// kmap: the key cache as rows of 128 bf16, boxes of 64 x 16; qmap: the window
// queries as [B][W][Hq][128], boxes of 64 dims x G heads x W positions x 1
// (both 128-byte swizzle).
cudaError_t launch_snapkv_scores(const CUtensorMap& kmap, const CUtensorMap& qmap, const KvView& kv, const uint16_t* qwin,
                                 int32_t num_q_heads,
                                 int32_t window, const int32_t* bt, int32_t bt_stride, const int32_t* lens,
                                 int32_t batch, int32_t max_len, float sm_scale, float* scores, int32_t score_stride,
                                 float* row_lse, void* part_ws, int sm_count, unsigned* err, cudaStream_t stream);
// The next launch_snapkv_scores of this host thread runs as a wait probe (limit in us).
void set_snapkv_wait_probe(uint32_t limit_us);
// Keeps positions 0 .. sink - 1 and n - recent .. n - 1 (recent >= window) and the keep best
// pooled candidates between them.
cudaError_t launch_snapkv_select(const float* scores, int32_t score_stride, const int32_t* lens, int32_t batch,
                                 int32_t num_kv_heads, int32_t window, int32_t max_len, int32_t pool, int32_t keep,
                                 int32_t sink, int32_t recent, int32_t* kept, int32_t kept_stride,
                                 int32_t* kept_counts, unsigned* err, cudaStream_t stream);
cudaError_t launch_snapkv_gather(const KvView& src, uint16_t* dk, uint16_t* dv, int32_t dst_num_pages,
                                 const int32_t* src_bt, int32_t src_bt_stride, const int32_t* dst_bt,
                                 int32_t dst_bt_stride, const int32_t* lens, int32_t batch, const int32_t* kept,
                                 int32_t kept_stride, const int32_t* kept_counts, unsigned* err, cudaStream_t stream);

// ---- api.cu: per-device context and helpers shared with other entry points
cudaError_t device_context(int* sm_count, unsigned** err);
void set_error_detail(const char* fn, const char* what);
// Argument checks of a sparse paged decode call (everything but the workspace),
// before any launch; *latent tells which kernel serves the shape.
se_status_t check_decode_call(const char* fn, const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                              const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens, int32_t batch,
                              const int32_t* sel_pages, const int32_t* sel_counts, int32_t sel_stride,
                              float sm_scale, const void* out, const float* out_lse, bool* latent);

}  // namespace se
