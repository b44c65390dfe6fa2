/*
 * sparse_engine.h -- C ABI of the GB300 (sm_103a) sparse decode attention library.
 *
 * The library implements the data-parallel hot path of a sparse-first serving
 * engine as described in "SparseEngine: Sparse-First Inference Engine"
 * (arXiv 2609.39068):
 *   - Quest: query-aware selection of 16-token KV pages from per-page key
 *     summaries, then attention over the selected pages only (Figure 2 caption,
 *     Figure 3 caption, Tables 8-12, Table 14);
 *   - SnapKV: eviction at the end of prefill from observation-window attention
 *     scores with max-pooling, keeping the selected tokens plus the window in
 *     compacted pages (Figure 2 caption, Table 8, Table 10, Table 15 note).
 * The pages do not print either method's equations; each entry point below
 * states the computation it performs.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named in a signature are DEVICE pointers unless the comment says
 *    "host". Structs are passed by host pointer and read during the call only.
 *  - The caller owns every buffer, including workspaces sized by the
 *    *_workspace_size functions. The library allocates no device memory and
 *    keeps no per-call state.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream). Results are valid once the stream has reached the call.
 *  - Arguments are validated on the host before anything is launched: a bad
 *    argument returns SE_ERR_INVALID_ARG (or SE_ERR_UNSUPPORTED for a shape
 *    the kernels do not implement, SE_ERR_WORKSPACE for a short workspace) and
 *    launches nothing. A launch failure returns SE_ERR_CUDA.
 *  - Device pointers must be 16-byte aligned. Device-side contents (lengths,
 *    page ids) are checked in the kernels: a value out of range sets a bit in the
 *    library's device error word, and the offending page or request is skipped.
 *    Read the word with se_read_device_error().
 *  - bf16 is IEEE-style bfloat16 (1-8-7), stored as uint16.
 *  - Page size is 16 tokens.
 */
#ifndef SPARSE_ENGINE_H
#define SPARSE_ENGINE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SE_API __attribute__((visibility("default")))
#else
#define SE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SE_OK = 0,
  SE_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer, stride too small */
  SE_ERR_UNSUPPORTED = 2,  /* valid arguments, shape not implemented (e.g. head_dim) */
  SE_ERR_WORKSPACE = 3,    /* workspace_bytes smaller than the *_workspace_size answer */
  SE_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  SE_ERR_DEVICE = 5        /* the device error word is non-zero (se_read_device_error) */
} se_status_t;

/* Bits of the device error word. */
#define SE_DEVERR_PAGE_RANGE   0x1u  /* a block-table entry outside [0, num_pages) */
#define SE_DEVERR_LENGTH       0x2u  /* a length or selected-page id outside its declared bound */
#define SE_DEVERR_WAIT_TIMEOUT 0x4u  /* a bounded wait (an mbarrier, or another CTA's counter) gave up */

/*
 * Paged KV cache view. Physical page p of KV head h holds tokens in slots
 * 0..15; token slot t of (p, h) starts at element
 *     ((p * num_kv_heads + h) * 16 + t) * row_stride
 * of `k` (resp. `v`). Quest page summaries live beside the pages, indexed by
 * the same physical page id ("the summaries required by Quest" kept with the
 * KV blocks, SparseEngine, Figure 3 caption):
 *     summary[((p * num_kv_heads + h) * 2 + 0) * head_dim + c] = min over the page's valid keys of channel c
 *     summary[((p * num_kv_heads + h) * 2 + 1) * head_dim + c] = max over the same keys
 * A latent (MLA-style) cache sets v == k with head_dim_v < head_dim: the value
 * is the first head_dim_v dims of the key row.
 */
typedef struct {
  void* k;                 /* bf16 */
  void* v;                 /* bf16; may equal k */
  void* summary;           /* bf16 [num_pages][num_kv_heads][2][head_dim]; may be NULL for calls that do not use it */
  int32_t num_pages;       /* physical pages in the pool */
  int32_t num_kv_heads;
  int32_t page_size;       /* must be 16 */
  int32_t head_dim;        /* key/query width: 128, or 576 for a latent cache */
  int32_t head_dim_v;      /* value width: 128, or 512 for a latent cache */
  int32_t row_stride_k;    /* elements between consecutive token rows of k (>= head_dim, multiple of 8) */
  int32_t row_stride_v;    /* elements between consecutive token rows of v (>= head_dim_v, multiple of 8) */
} se_paged_kv_t;

/* Human-readable name of a status code (host, static storage). */
SE_API const char* se_status_string(int status);

/* Details of the last failing call on this host thread: entry point and reason
 * (host, thread-local storage, valid until the next failing call). */
SE_API const char* se_last_error_detail(void);

/*
 * Reads the library's device error word (SE_DEVERR_* bits) for the current
 * device into *out (host) after synchronising the device; clears it when
 * `clear` is non-zero. Returns SE_OK or SE_ERR_CUDA.
 */
SE_API se_status_t se_read_device_error(uint32_t* out, int clear);

/*
 * se_quest_build_summaries -- Quest page summaries from the cached keys.
 * SparseEngine, Figure 3 caption (prefix caching keeps the Quest summaries with
 * the KV blocks) and Table 8 (16-token pages).
 * For every request b, every logical page p < ceil(seq_lens[b] / 16) and every
 * KV head h, writes into kv->summary at physical page block_table[b][p] the
 * per-channel minimum and maximum of the keys of the page's valid tokens
 * (positions < seq_lens[b]); slots past the length are never read.
 *   block_table: int32 [batch][bt_stride]; seq_lens: int32 [batch];
 *   max_seq_len: host upper bound of seq_lens (sizes the grid; a larger device
 *   value sets SE_DEVERR_LENGTH and the request is clipped to it).
 */
SE_API se_status_t se_quest_build_summaries(const se_paged_kv_t* kv, const int32_t* block_table, int32_t bt_stride,
                                     const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                     void* stream);

/*
 * se_quest_update_summaries -- KV append fused with the Quest summary update.
 * SparseEngine, Figure 3 caption (summaries kept with the KV blocks); Table 7
 * (the history of the current position includes the current token).
 * For every request b and KV head h, writes k_new[b][h] (and v_new[b][h]) into
 * the token slot of position seq_lens_before[b] (logical page pos / 16, slot
 * pos % 16, physical page from block_table), and updates that page's summary:
 * set to k_new when the token opens the page (slot 0), otherwise the running
 * min and max with k_new. Re-running the same append is idempotent. The caller
 * advances its lengths afterwards. Requests must not share the written page.
 *   k_new: bf16 [batch][num_kv_heads][head_dim];
 *   v_new: bf16 [batch][num_kv_heads][head_dim_v], or NULL when kv->v == kv->k
 *   (latent cache: the value is part of the key row).
 * With kv->summary NULL only the K/V rows are written: the decode-time append of
 * a cache that keeps no Quest summaries (a SnapKV-compacted cache between its
 * periodic evictions, Table 10: eviction every 1,024 decode steps).
 */
SE_API se_status_t se_quest_update_summaries(const se_paged_kv_t* kv, const void* k_new, const void* v_new,
                                      const int32_t* block_table, int32_t bt_stride,
                                      const int32_t* seq_lens_before, int32_t batch, void* stream);

/*
 * se_quest_update_summaries_ex -- se_quest_update_summaries with flags.
 *   flags: 0, or SE_APPEND_OVERLAP_PREVIOUS: the append's kernel may start
 *   while the previous kernel of `stream` still runs (programmatic dependent
 *   launch, when that kernel allows it) and completes only after it, so work
 *   queued after the call still sees the previous kernel's results. The caller
 *   guarantees that the previous kernel neither reads nor writes anything the
 *   append touches (the written K/V slots and the summary of their page),
 *   e.g. the page selection of the same step: the page a token lands in is the
 *   request's last page, which is never scored (it is always kept). Other bits:
 *   SE_ERR_INVALID_ARG.
 */
#define SE_APPEND_OVERLAP_PREVIOUS 0x1u
SE_API se_status_t se_quest_update_summaries_ex(const se_paged_kv_t* kv, const void* k_new, const void* v_new,
                                                const int32_t* block_table, int32_t bt_stride,
                                                const int32_t* seq_lens_before, int32_t batch, uint32_t flags,
                                                void* stream);

/*
 * se_quest_score_pages -- Quest upper-bound score of every candidate page.
 * SparseEngine, Figure 2 caption and Table 14 (Quest, query-dependent page
 * retrieval); the bound is the published Quest criterion.
 * For request b, KV head h and candidate page p in [0, n_b - 2] with
 * n_b = ceil(seq_lens[b] / 16):
 *     scores[(b * num_kv_heads + h) * score_stride + p]
 *         = sum over the query heads a of h's group, sum over channels c, of
 *           max(q[b][a][c] * min_{p,c}, q[b][a][c] * max_{p,c})
 * (computed as sum_c max_{p,c} * P_c + min_{p,c} * N_c with P_c, N_c the sums of
 * the group's positive and negative query parts; fp32). The last page is not
 * scored: it is always kept.
 *   q: bf16 [batch][num_q_heads][head_dim]; num_q_heads a multiple of num_kv_heads;
 *   scores: fp32, score_stride >= ceil(max_seq_len / 16).
 */
SE_API se_status_t se_quest_score_pages(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                 const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                 int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                                 void* stream);

/*
 * se_quest_score_workspace_size -- bytes of the workspace of
 * se_quest_score_pages_ws: the group sums P_c and N_c of every request and KV
 * head (fp32, batch * num_kv_heads * 2 * head_dim values), then 16 bytes for
 * the counter of the scoring kernel's page pool (reset by every call).
 * 0 for negative sizes.
 */
SE_API size_t se_quest_score_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t head_dim);

/*
 * se_quest_score_pages_ws -- se_quest_score_pages with a workspace for the
 * query multipliers. Same scores, bit for bit. A first kernel sums every
 * request's queries into P_c and N_c once; the scoring kernel then reads them
 * instead of summing the queries of each request in every CTA that scores part
 * of it. That summing waits on the memory latency of the query loads while the
 * summary reads keep HBM busy; with the workspace, a CTA's switch to another
 * request costs one read of the sums. The largest gain is for the latent cache
 * (64 query heads of 576 channels per request). With the workspace the
 * scoring kernel also balances its end: every CTA scores an equal static
 * slice of three quarters of the pages, and the rest go in units of 8 pages
 * to whichever warp is free (the scores do not depend on who computes them).
 *   workspace: device memory the caller owns, 16-byte aligned, at least
 *   se_quest_score_workspace_size(batch, kv->num_kv_heads, kv->head_dim) bytes
 *   (SE_ERR_WORKSPACE when smaller, SE_ERR_INVALID_ARG when NULL or
 *   misaligned); its contents on entry do not matter and are overwritten.
 * The other arguments and errors are those of se_quest_score_pages.
 */
SE_API se_status_t se_quest_score_pages_ws(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                           const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                           int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * se_quest_topk_pages -- per-(request, KV head) page selection.
 * SparseEngine, Table 10 caption (selected budgets exclude separately kept
 * tokens) and Table 10, Quest (Vortex) row (2,048 selected tokens = 128 pages).
 * Among the candidates 0..n_b-2 picks the topk_pages highest scores (equal
 * scores: lower page id first), appends the last page n_b - 1, and writes the
 * page ids in ascending order to out_pages[(b * num_kv_heads + h) * sel_stride
 * + i] and the count to out_counts[b * num_kv_heads + h]. With no more than
 * topk_pages candidates every page is selected (count n_b). A request of
 * length 0 selects nothing (count 0).
 *   sel_stride >= topk_pages + 1.
 */
SE_API se_status_t se_quest_topk_pages(const float* scores, int32_t score_stride, const int32_t* seq_lens,
                                int32_t batch, int32_t num_kv_heads, int32_t max_seq_len, int32_t topk_pages,
                                int32_t* out_pages, int32_t* out_counts, int32_t sel_stride, void* stream);

/*
 * se_quest_topk_pages_windowed -- se_quest_topk_pages with sink and recent keep
 * windows. SparseEngine, Tables 9-12: Quest keeps sink and recent tokens
 * beside its selected budget (e.g. sink 64, recent 512, 1,472 selected =
 * 2,048 total, Tables 11 and 12; sink 64, recent 256, 4,096 selected =
 * 4,416 total, Table 9), and the budget excludes them (Table 10 caption).
 * Page-granular: the pages holding any of the first sink_tokens tokens and
 * the pages holding any of the last recent_tokens tokens are always kept, as
 * is the last page; topk_pages pages are selected among the pages between
 * them (equal scores: lower page id first). Output, ascending: the sink pages,
 * the selected pages, the recent pages; count = all of them (every page when
 * no more than topk_pages candidates remain). sink_tokens = recent_tokens = 0
 * is se_quest_topk_pages.
 *   sel_stride >= se_quest_kept_pages_max(topk_pages, sink_tokens, recent_tokens)
 *               = ceil(sink/16) + topk_pages + ceil(recent/16) + 1.
 */
SE_API se_status_t se_quest_topk_pages_windowed(const float* scores, int32_t score_stride, const int32_t* seq_lens,
                                                int32_t batch, int32_t num_kv_heads, int32_t max_seq_len,
                                                int32_t topk_pages, int32_t sink_tokens, int32_t recent_tokens,
                                                int32_t* out_pages, int32_t* out_counts, int32_t sel_stride,
                                                void* stream);
/* Most pages one (request, KV head) can keep with these windows (-1 for a negative argument). Host only. */
SE_API long long se_quest_kept_pages_max(int32_t topk_pages, int32_t sink_tokens, int32_t recent_tokens);

/*
 * se_quest_select_pages -- se_quest_score_pages followed by se_quest_topk_pages,
 * with the scores kept in the caller's workspace (size from
 * se_quest_select_workspace_size).
 */
SE_API size_t se_quest_select_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len);
SE_API se_status_t se_quest_select_pages(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                  const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                  int32_t batch, int32_t max_seq_len, int32_t topk_pages, int32_t* out_pages,
                                  int32_t* out_counts, int32_t sel_stride, void* workspace,
                                  size_t workspace_bytes, void* stream);
/* se_quest_select_pages with the keep windows of se_quest_topk_pages_windowed. */
SE_API se_status_t se_quest_select_pages_windowed(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                                  const int32_t* block_table, int32_t bt_stride,
                                                  const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                                  int32_t topk_pages, int32_t sink_tokens, int32_t recent_tokens,
                                                  int32_t* out_pages, int32_t* out_counts, int32_t sel_stride,
                                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * se_quest_fused_step -- one Quest decode step in a single launch: the optional
 * KV append with its summary update, the page scores, the windowed top-k and
 * the sparse decode, with the scores kept in on-chip memory (a cluster of CTAs
 * per (request, KV head) shares them over distributed shared memory).
 * SparseEngine, Figure 2 and Figure 3 captions; Tables 9-12 (keep windows);
 * Table 7 (the history includes the current token). The results equal
 * se_quest_update_summaries + se_quest_score_pages +
 * se_quest_topk_pages_windowed + se_sparse_paged_decode:
 *   seq_lens: lengths INCLUDING the new token; with k_new/v_new (bf16
 *     [batch][num_kv_heads][128], both or neither) the token at position
 *     seq_lens[b] - 1 is appended first (no append when both are NULL);
 *   sel_pages / sel_counts: the kept pages as se_quest_topk_pages_windowed writes them;
 *   out: bf16 [batch][num_q_heads][128]; out_lse: fp32 [batch][num_q_heads] or NULL.
 * Shapes: head_dim = head_dim_v = 128, separate K and V caches, up to 16 query
 * heads per KV head, up to 8192 candidate pages per request and 2048 kept pages
 * (se_quest_kept_pages_max); sel_stride >= se_quest_kept_pages_max(...). No workspace.
 */
SE_API se_status_t se_quest_fused_step(const se_paged_kv_t* kv, const void* k_new, const void* v_new, const void* q,
                                       int32_t num_q_heads, const int32_t* block_table, int32_t bt_stride,
                                       const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                       int32_t topk_pages, int32_t sink_tokens, int32_t recent_tokens, float sm_scale,
                                       void* out, float* out_lse, int32_t* sel_pages, int32_t* sel_counts,
                                       int32_t sel_stride, void* stream);

/*
 * se_sparse_paged_decode -- attention of one decode query per request over the
 * selected pages only.
 * SparseEngine, Figure 2 caption (attention execution over the method's view of
 * the cache) and Table 7 (logit z, weight alpha; the history includes the
 * current token).
 * For request b and query head a (KV head h = a / (num_q_heads / num_kv_heads)):
 *     z_j = sm_scale * q[b][a] . k_j over the tokens j < seq_lens[b] of the pages
 *           sel_pages[(b * num_kv_heads + h) * sel_stride + i], i < sel_counts[..]
 *     out[b][a]  = sum_j softmax(z)_j v_j                       (bf16, round to nearest even)
 *     out_lse[b][a] = log sum_j exp(z_j)                        (fp32, natural log; optional)
 * A request with no selected page writes out = 0 and lse = -inf. The pages of
 * one (request, KV head) are split across CTAs and the partial results merged
 * by log-sum-exp in `workspace` (size from se_sparse_decode_workspace_size).
 * The workspace must be zero-filled before its first use (one cudaMemset after
 * allocating it): for head_dim 128 it holds per-item arrival counters that the
 * CTA publishing an item's last partial reads and resets, so every call leaves
 * them zero for the next one; the rest is overwritten by each call. Calls that
 * share a workspace must not overlap on the GPU.
 *   q: bf16 [batch][num_q_heads][head_dim]; out: bf16 [batch][num_q_heads][head_dim_v];
 *   out_lse: fp32 [batch][num_q_heads] or NULL.
 * Shapes: head_dim == head_dim_v == 128 with 1..16 query heads per KV head, or a
 * latent cache (head_dim 576, head_dim_v 512, one KV head, kv->v == kv->k,
 * 16..64 query heads in multiples of 16).
 */
/*
 * se_sparse_decode_plan -- how se_sparse_paged_decode splits the work on the
 * current device for these sizes. The selected pages of all (request, KV head)
 * items are cut into equal slices of at least *pages_per_split pages, one per
 * CTA; *nsplit is the most slices one item can span (the partial results kept
 * per query-head row), and *launches the kernels per call: 1 for head_dim 128
 * (the decode kernel merges the split partials itself), 2 for a latent cache
 * (the decode kernel and the log-sum-exp merge). Host only.
 */
SE_API se_status_t se_sparse_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t head_dim_v, int32_t sel_stride,
                                         int32_t* nsplit, int32_t* pages_per_split, int32_t* launches);
SE_API size_t se_sparse_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim_v, int32_t sel_stride);
SE_API se_status_t se_sparse_paged_decode(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                   const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                   int32_t batch, const int32_t* sel_pages, const int32_t* sel_counts,
                                   int32_t sel_stride, float sm_scale, void* out, float* out_lse,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * SnapKV eviction at the end of prefill (SparseEngine: Sparse-First Inference
 * Engine, Table 8: 32-query scoring window, pooling kernel 7, 2,016 selected +
 * 32 recent tokens; Table 10: probability-based prefill scores; Table 15 note:
 * physical eviction releases KV storage; Figure 3 caption: the compacted state
 * is what Chain Cache resumes from).
 * For request b (prompt length n = prompt_lens[b] >= window) and KV head h, the
 * window queries are the last `window` prompt positions: q_window[b][w][a] is
 * the query of head a at position n - window + w (bf16 [batch][window][Hq][128]).
 * Row r = (w, g) of h's group sees keys j <= n - window + w, with logits
 * z = sm_scale q . k_j. Shapes: head_dim 128 and window * (Hq / Hkv) <= 128.
 *
 * se_snapkv_window_scores: for every candidate j < n - window,
 *     scores[(b * Hkv + h) * score_stride + j] = sum over the window rows and the
 *     group's query heads of softmax_j(z)  (fp32; the softmax of each row is over
 *     all the keys it sees, window keys included),
 *   and optionally row_lse[(b * Hkv + h) * window * G + r] = log sum_j exp(z_rj)
 *   (NULL to skip). score_stride >= max_prompt_len - window. Workspace: the
 *   per-slice row statistics, se_snapkv_workspace_size bytes (any larger size
 *   is fine; the scores buffer of se_snapkv_score_and_compact is not needed
 *   here).
 * se_snapkv_select: max-pools each row of scores with an odd pool_kernel
 *   (stride 1, window clipped to the candidates), keeps the keep_topk best
 *   candidates (equal pooled scores: lower position first) in ascending order,
 *   then appends the window positions n - window .. n - 1; with at most
 *   keep_topk candidates every position is kept. kept_pos int32
 *   [batch][Hkv][kept_stride] (kept_stride >= keep_topk + window), kept_counts
 *   int32 [batch][Hkv]. Up to 45056 candidates per request.
 * se_snapkv_compact: copies the kept K and V rows unchanged into the destination
 *   cache: kept token t of (b, h) goes to page dst_block_table[b][t / 16],
 *   slot t % 16, head h (destination rows dense, 128 wide). The destination
 *   table must map ceil(kept_counts / 16) pages; a kept token past
 *   dst_bt_stride * 16 or a page id out of range sets the device error word
 *   and is skipped.
 * se_snapkv_score_and_compact: the three steps, the scores kept in `workspace`
 *   (se_snapkv_workspace_size bytes).
 * se_snapkv_select_windowed / se_snapkv_score_and_compact_windowed: the same
 *   with explicit keep windows (SparseEngine, Tables 9-12: SnapKV with sink
 *   0/16/64 and recent 64/256/512 tokens beside 4,096 or 15,808 selected, a
 *   16-query observation window in Table 10; Table 10 caption: the budget
 *   excludes them). Positions 0 .. sink_tokens - 1 and n - recent_tokens ..
 *   n - 1 are always kept (recent_tokens >= window); the keep_topk best pooled
 *   candidates among the positions between them are kept in ascending order;
 *   the scores and the pooling are those above (every position before the
 *   window is scored and pooled). Output: sink positions, selected, recent
 *   positions; every position when no more than keep_topk candidates remain.
 *   kept_stride >= sink_tokens + keep_topk + recent_tokens. sink_tokens = 0,
 *   recent_tokens = window is the plain call.
 */
SE_API size_t se_snapkv_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t window,
                                       int32_t max_prompt_len);
SE_API se_status_t se_snapkv_window_scores(const se_paged_kv_t* src, const void* q_window, int32_t num_q_heads,
                                           int32_t window, const int32_t* block_table, int32_t bt_stride,
                                           const int32_t* prompt_lens, int32_t batch, int32_t max_prompt_len,
                                           float sm_scale, float* scores, int32_t score_stride, float* row_lse,
                                           void* workspace, size_t workspace_bytes, void* stream);
SE_API se_status_t se_snapkv_select(const float* scores, int32_t score_stride, const int32_t* prompt_lens,
                                    int32_t batch, int32_t num_kv_heads, int32_t window, int32_t max_prompt_len,
                                    int32_t pool_kernel, int32_t keep_topk, int32_t* kept_pos, int32_t kept_stride,
                                    int32_t* kept_counts, void* stream);
SE_API se_status_t se_snapkv_select_windowed(const float* scores, int32_t score_stride, const int32_t* prompt_lens,
                                             int32_t batch, int32_t num_kv_heads, int32_t window,
                                             int32_t max_prompt_len, int32_t pool_kernel, int32_t keep_topk,
                                             int32_t sink_tokens, int32_t recent_tokens, int32_t* kept_pos,
                                             int32_t kept_stride, int32_t* kept_counts, void* stream);
SE_API se_status_t se_snapkv_compact(const se_paged_kv_t* src, const int32_t* src_block_table, int32_t src_bt_stride,
                                     const int32_t* prompt_lens, int32_t batch, const se_paged_kv_t* dst,
                                     const int32_t* dst_block_table, int32_t dst_bt_stride, const int32_t* kept_pos,
                                     int32_t kept_stride, const int32_t* kept_counts, void* stream);
SE_API se_status_t se_snapkv_score_and_compact(const se_paged_kv_t* src, const void* q_window, int32_t num_q_heads,
                                               int32_t window, const int32_t* src_block_table,
                                               int32_t src_bt_stride, const int32_t* prompt_lens, int32_t batch,
                                               int32_t max_prompt_len, int32_t pool_kernel, int32_t keep_topk,
                                               float sm_scale, const se_paged_kv_t* dst,
                                               const int32_t* dst_block_table, int32_t dst_bt_stride,
                                               int32_t* kept_pos, int32_t kept_stride, int32_t* kept_counts,
                                               void* workspace, size_t workspace_bytes, void* stream);
SE_API se_status_t se_snapkv_score_and_compact_windowed(const se_paged_kv_t* src, const void* q_window,
                                                        int32_t num_q_heads, int32_t window,
                                                        const int32_t* src_block_table, int32_t src_bt_stride,
                                                        const int32_t* prompt_lens, int32_t batch,
                                                        int32_t max_prompt_len, int32_t pool_kernel,
                                                        int32_t keep_topk, int32_t sink_tokens,
                                                        int32_t recent_tokens, float sm_scale,
                                                        const se_paged_kv_t* dst, const int32_t* dst_block_table,
                                                        int32_t dst_bt_stride, int32_t* kept_pos,
                                                        int32_t kept_stride, int32_t* kept_counts, void* workspace,
                                                        size_t workspace_bytes, void* stream);

/*
 * Replayable steps. A decode loop makes the same library calls every step on
 * the same buffers; only the values in device memory change (queries, new K/V
 * rows, lengths, selections), and every kernel of the library reads those
 * values from device memory. These calls record the asynchronous work of a
 * sequence of library calls into a CUDA graph once, so that each later step
 * costs one launch instead of the calls' host-side checks and launches. The
 * pages have no counterpart: this is host plumbing around their hot path.
 *
 * se_capture_begin -- starts recording the work issued on `stream` (a stream
 *   the caller created, not the legacy default stream; thread-local capture
 *   mode). It first sets up this device's library context, so that no call
 *   made while recording allocates. Between begin and end, make the library
 *   calls of one step on `stream`, each exactly as it would be made live:
 *   their argument checks run now, once, and only their kernels and
 *   asynchronous copies and sets are recorded. A call that fails while
 *   recording leaves the capture to be ended and its graph discarded.
 *   se_sparse_paged_decode_noalloc may be recorded after one live call of it
 *   on the device (that call looks up the address of its built-in array).
 * se_capture_end -- ends the recording on `stream` and instantiates it into
 *   *graph (host handle; owned by the caller, freed with se_graph_destroy).
 * se_graph_launch -- runs the recorded step on `stream` (any stream of the
 *   device it was recorded on). Every buffer the recorded calls named must
 *   still exist, and the sizes passed to them (batch, strides, maximum
 *   lengths) still hold; the values in the buffers may change freely between
 *   launches, as in the live calls.
 * se_graph_destroy -- frees a recorded step (NULL: no-op).
 * Errors: SE_ERR_INVALID_ARG for a NULL stream, graph or handle; SE_ERR_CUDA
 * for a failing CUDA call (begin, end, instantiate or launch), with the CUDA
 * error in se_last_error_detail().
 */
typedef struct se_graph_s* se_graph_t;
SE_API se_status_t se_capture_begin(void* stream);
SE_API se_status_t se_capture_end(void* stream, se_graph_t* graph);
SE_API se_status_t se_graph_launch(se_graph_t graph, void* stream);
SE_API void se_graph_destroy(se_graph_t graph);

/*
 * se_copy_async -- copies `bytes` bytes from src to dst on `stream`,
 * asynchronously: device memory to or from page-locked host memory, or device
 * to device (the direction follows from the addresses). Up to 8 MiB between
 * device memory and page-locked host memory, the copy is a kernel of the
 * library whose loads or stores reach the host side directly (a decode step's
 * few hundred KB move in a fraction of a copy engine's start-up); it waits for
 * the previous kernel on `stream` like every kernel of the library. Other
 * copies use the copy engine (cudaMemcpyAsync). Made between
 * se_capture_begin and se_capture_end it is recorded too, so that a step's
 * input upload and result download replay with its kernels in one launch. The
 * pages have no counterpart: this is host plumbing around their hot path.
 * Pageable host memory is not allowed while recording (CUDA refuses it) and
 * makes a live copy synchronous. Ownership: both buffers stay the caller's and
 * must outlive the copy (and every replay of a recording that holds it).
 * Errors: SE_ERR_INVALID_ARG for a NULL dst or src with bytes > 0 (bytes = 0
 * is a no-op); SE_ERR_CUDA for a failing copy, with the CUDA error in
 * se_last_error_detail().
 */
SE_API se_status_t se_copy_async(void* dst, const void* src, size_t bytes, void* stream);

/*
 * se_debug_snapkv_wait_probe -- test hook for the bounded waits; it computes
 * nothing (the pages have no counterpart). In the next se_snapkv_window_scores
 * call issued from this host thread (also inside se_snapkv_score_and_compact*),
 * the first score kernel's MMA-issuing thread of every CTA first waits on an
 * mbarrier phase that nothing completes, and gives up after limit_us
 * microseconds (1 .. 1000000). The kernel then sets SE_DEVERR_WAIT_TIMEOUT in
 * the device error word and issues no tensor-core work for the rest of that
 * launch; its copies still drain and it frees its tensor memory, so the context
 * stays usable. The call's scores are not valid. Later calls are unaffected.
 */
SE_API se_status_t se_debug_snapkv_wait_probe(uint32_t limit_us);

/*
 * se_sparse_paged_decode_noalloc -- se_sparse_paged_decode for callers that
 * cannot allocate device memory. The SparseEngine pages have no counterpart: this
 * is a deployment variant of the decode above.
 * Some callers have no way to provide the decode workspace: a plugin in an
 * inference runtime that receives only its inputs and outputs, a process whose
 * device memory is owned by another framework's caching allocator, or a serving
 * loop that forbids cudaMalloc after start-up because it can synchronise the
 * device. For head_dim = head_dim_v = 128 with up to 16 query heads per KV
 * head, this call computes what se_sparse_paged_decode computes, with the same
 * arguments minus the workspace, and keeps the split partials in a fixed 8 MiB
 * array inside the library (held on every GPU that loads the library until the
 * process exits). A latent cache (576/512) is rejected with SE_ERR_UNSUPPORTED:
 * it needs se_sparse_paged_decode with a caller workspace. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *  - The first call on a device looks up the array's device address, with that
 *    device current; make that first call before any stream capture. The address
 *    is kept for the life of the process: after cudaDeviceReset, do not call the
 *    library on that device again.
 *  - Sizes whose partials exceed 8 MiB are rejected with SE_ERR_WORKSPACE
 *    (use se_sparse_paged_decode with a workspace instead); the bound is
 *    batch * num_q_heads * splits * (head_dim_v + 1) * 4 bytes plus
 *    batch * num_q_heads * 4, splits from se_sparse_decode_plan.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents. Every partial read is first written by the same call; the
 *    split-merge counters, which must start at zero, are cleared by each call
 *    with an asynchronous memset on `stream` before its launch. Two calls that
 *    overlap on the GPU race on the array: order them on one stream or with
 *    events.
 */
SE_API se_status_t se_sparse_paged_decode_noalloc(const se_paged_kv_t* kv, const void* q, int32_t num_q_heads,
                                                  const int32_t* block_table, int32_t bt_stride,
                                                  const int32_t* seq_lens, int32_t batch, const int32_t* sel_pages,
                                                  const int32_t* sel_counts, int32_t sel_stride, float sm_scale,
                                                  void* out, float* out_lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ENGINE_H */
