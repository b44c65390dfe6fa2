// Quest page summaries: the per-channel key minimum and maximum of every
// 16-token page, kept beside the page in the paged cache (SparseEngine:
// Sparse-First Inference Engine, Figure 3 caption: prefix caching keeps the
// summaries Quest needs with the KV blocks; Table 8: 16-token pages).
//
//  * build_summaries_kernel: summaries of every page of every request from the
//    cached keys (end of prefill). Memory-bound copy-like pass: reads the valid
//    key rows once, writes 2 rows per (page, head).
//  * append_update_kernel: the decode-time KV append fused with the summary
//    update of the page the token lands in (one warp per request and KV head).
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kBuildWarps = 8;
constexpr int kBuildPagesPerCta = 16;

__device__ __forceinline__ int clamp_len(int L, int max_len, unsigned* err) {
  if (L < 0 || L > max_len) {
    raise_error(err, SE_DEVERR_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  return L;
}

__global__ void __launch_bounds__(kBuildWarps * 32) build_summaries_kernel(
    KvView kv, const int32_t* __restrict__ block_table, int32_t bt_stride, const int32_t* __restrict__ seq_lens,
    int32_t max_seq_len, unsigned* err) {
  pdl_enter();
  const int b = blockIdx.y;
  const int L = clamp_len(seq_lens[b], max_seq_len, err);
  const int n_pages = (L + kPageSize - 1) / kPageSize;
  const int first = blockIdx.x * kBuildPagesPerCta;
  if (first >= n_pages) return;
  const int last = min(n_pages, first + kBuildPagesPerCta);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = kv.num_kv_heads, D = kv.head_dim;
  for (int idx = warp; idx < (last - first) * H; idx += kBuildWarps) {
    const int p = first + idx / H, h = idx % H;
    const int phys = block_table[(size_t)b * bt_stride + p];
    if (phys < 0 || phys >= kv.num_pages) {
      if (lane == 0) raise_error(err, SE_DEVERR_PAGE_RANGE);
      continue;
    }
    const int valid = min(kPageSize, L - p * kPageSize);
    const size_t blk = (size_t)phys * H + h;
    const uint16_t* rows = kv.k + blk * kPageSize * kv.row_stride_k;
    uint32_t* out = reinterpret_cast<uint32_t*>(kv.summary + blk * 2 * D);
    for (int c = 2 * lane; c < D; c += 64) {
      float mn0 = INFINITY, mn1 = INFINITY, mx0 = -INFINITY, mx1 = -INFINITY;
      for (int t = 0; t < valid; ++t) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(rows + (size_t)t * kv.row_stride_k + c);
        const float lo = bf16_lo(v), hi = bf16_hi(v);
        mn0 = fminf(mn0, lo);
        mx0 = fmaxf(mx0, lo);
        mn1 = fminf(mn1, hi);
        mx1 = fmaxf(mx1, hi);
      }
      // min and max of bf16 values are bf16 values: the round trip is exact.
      out[c >> 1] = pack_bf16x2(mn0, mn1);
      out[(D + c) >> 1] = pack_bf16x2(mx0, mx1);
    }
  }
}

// kOverlap: the kernel may start while the previous kernel of the stream still
// runs (programmatic dependent launch); it touches nothing that kernel reads or
// writes, and waits for it only before it exits, so that the kernels after it
// still see everything before it complete.
template <bool kOverlap>
__global__ void __launch_bounds__(256) append_update_kernel(KvView kv, uint16_t* __restrict__ k_mut,
                                                            uint16_t* __restrict__ v_mut,
                                                            const uint16_t* __restrict__ k_new,
                                                            const uint16_t* __restrict__ v_new,
                                                            const int32_t* __restrict__ block_table,
                                                            int32_t bt_stride,
                                                            const int32_t* __restrict__ seq_lens_before,
                                                            int32_t batch, unsigned* err) {
  if (kOverlap)
    pdl_launch_dependents();
  else
    pdl_enter();
  const int H = kv.num_kv_heads;
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  do {
    if (item >= batch * H) break;
    const int b = item / H, h = item % H;
    const int pos = seq_lens_before[b];
    if (pos < 0 || pos / kPageSize >= bt_stride) {
      if (lane == 0) raise_error(err, SE_DEVERR_LENGTH);
      break;
    }
    const int page = pos / kPageSize, slot = pos % kPageSize;
    const int phys = block_table[(size_t)b * bt_stride + page];
    if (phys < 0 || phys >= kv.num_pages) {
      if (lane == 0) raise_error(err, SE_DEVERR_PAGE_RANGE);
      break;
    }
    const int D = kv.head_dim, Dv = kv.head_dim_v;
    const size_t blk = (size_t)phys * H + h;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(k_new + (size_t)item * D);
    uint32_t* dst = reinterpret_cast<uint32_t*>(k_mut + (blk * kPageSize + slot) * kv.row_stride_k);
    // A cache without Quest summaries (e.g. a SnapKV-compacted one) only gets the rows.
    uint32_t* smin = kv.summary ? reinterpret_cast<uint32_t*>(kv.summary + blk * 2 * D) : nullptr;
    uint32_t* smax = smin + (D >> 1);
    for (int c = lane; c < (D >> 1); c += 32) {
      const uint32_t x = src[c];
      dst[c] = x;
      if (smin == nullptr) continue;
      if (slot == 0) {
        smin[c] = x;
        smax[c] = x;
      } else {
        const uint32_t a = smin[c], z = smax[c];
        smin[c] = pack_bf16x2(fminf(bf16_lo(a), bf16_lo(x)), fminf(bf16_hi(a), bf16_hi(x)));
        smax[c] = pack_bf16x2(fmaxf(bf16_lo(z), bf16_lo(x)), fmaxf(bf16_hi(z), bf16_hi(x)));
      }
    }
    if (v_new != nullptr) {
      const uint32_t* vs = reinterpret_cast<const uint32_t*>(v_new + (size_t)item * Dv);
      uint32_t* vd = reinterpret_cast<uint32_t*>(v_mut + (blk * kPageSize + slot) * kv.row_stride_v);
      for (int c = lane; c < (Dv >> 1); c += 32) vd[c] = vs[c];
    }
  } while (false);
  if (kOverlap) pdl_wait();  // every thread: the grid completes only after the previous one
}

}  // namespace

cudaError_t launch_build_summaries(const KvView& kv, const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, unsigned* err,
                                   cudaStream_t stream) {
  const int max_pages = (max_seq_len + kPageSize - 1) / kPageSize;
  if (batch == 0 || max_pages == 0) return cudaSuccess;
  dim3 grid((max_pages + kBuildPagesPerCta - 1) / kBuildPagesPerCta, batch);
  {
    const cudaError_t le = launch_pdl(build_summaries_kernel, dim3(grid), dim3(kBuildWarps * 32), 0, stream, kv,
                                      block_table, bt_stride, seq_lens, max_seq_len, err);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_append_update(const KvView& kv, uint16_t* k_mut, uint16_t* v_mut, const uint16_t* k_new,
                                 const uint16_t* v_new, const int32_t* block_table, int32_t bt_stride,
                                 const int32_t* seq_lens_before, int32_t batch, bool overlap_previous,
                                 unsigned* err, cudaStream_t stream) {
  const int items = batch * kv.num_kv_heads;
  if (items == 0) return cudaSuccess;
  const cudaError_t le =
      overlap_previous
          ? launch_pdl(append_update_kernel<true>, dim3((items + 7) / 8), dim3(256), 0, stream, kv, k_mut, v_mut,
                       k_new, v_new, block_table, bt_stride, seq_lens_before, batch, err)
          : launch_pdl(append_update_kernel<false>, dim3((items + 7) / 8), dim3(256), 0, stream, kv, k_mut, v_mut,
                       k_new, v_new, block_table, bt_stride, seq_lens_before, batch, err);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace se
