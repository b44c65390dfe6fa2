// Quest page scoring (SparseEngine: Sparse-First Inference Engine, Figure 2
// caption and Table 14: Quest, query-dependent page retrieval; Figure 3 caption:
// the per-page summaries kept beside the KV blocks).
//
// For request b, KV head h and candidate page p (0 .. n_b - 2) the score is the
// Quest upper bound summed over the query heads of h's GQA group:
//     U(p) = sum_c max_{p,c} * P_c + min_{p,c} * N_c,
// where P_c (N_c) is the sum of the group's positive (negative) query parts in
// channel c. This equals the sum over the group of sum_c max(q_c min_c, q_c max_c)
// and needs one multiply-add per summary element: the kernel is HBM-bound.
//
// Work split: the candidate pages of all requests form one flattened range
// (request-major). Each CTA takes an equal slice, so ragged lengths balance.
// The slice is cut at request boundaries into segments. For each segment the
// CTA first computes P and N of the request together (all threads, the group
// cut into runs; double-buffered in shared memory); every lane then keeps the
// multipliers of its own 16-byte chunks in registers. Warps take every eighth
// page of the segment and load U pages at a time with 16-byte loads straight
// into registers, so U page blocks per warp
// are in flight (a page block holds all KV heads of the page, contiguous).
// A page costs T 16-byte loads and 8 T multiply-adds per lane plus a butterfly
// reduce-scatter across the KV heads. Scattered page blocks read this way reach
// close to full HBM bandwidth on GB300, where one issuing warp feeding a
// bulk-copy ring is limited by its per-copy issue cost.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct ScoreArgs {
  KvView kv;
  const uint16_t* q;
  int32_t group;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t max_seq_len;
  float* scores;
  int32_t score_stride;
  unsigned* err;
};

// Largest b in [0, n - 1] with prefix[b] <= x (prefix non-decreasing, prefix[0] = 0): the
// request whose candidate range holds x (empty requests are skipped).
__device__ __forceinline__ int find_request(const int* prefix, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// 8 bf16 values (one 16-byte chunk) times 8 fp32 multipliers, accumulated.
__device__ __forceinline__ float dot8(const uint4 v, const float (&m)[8], float acc) {
  acc = fmaf(bf16_lo(v.x), m[0], acc);
  acc = fmaf(bf16_hi(v.x), m[1], acc);
  acc = fmaf(bf16_lo(v.y), m[2], acc);
  acc = fmaf(bf16_hi(v.y), m[3], acc);
  acc = fmaf(bf16_lo(v.z), m[4], acc);
  acc = fmaf(bf16_hi(v.z), m[5], acc);
  acc = fmaf(bf16_lo(v.w), m[6], acc);
  acc = fmaf(bf16_hi(v.w), m[7], acc);
  return acc;
}

// Runs of query heads the group is cut into for the P/N pre-reduction: about
// two tasks of (KV head, 8 channels, run) per thread, at most one head per run.
__host__ __device__ __forceinline__ int pn_slices(int items, int group) {
  const int s = (2 * kThreads + items - 1) / items;
  return s < group ? s : group;
}

// Positive and negative parts of 8 bf16 query values, accumulated.
__device__ __forceinline__ void add_pos_neg(const uint4 v, float (&P)[8], float (&N)[8]) {
  const float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                      bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    P[e] += fmaxf(x[e], 0.f);
    N[e] += fminf(x[e], 0.f);
  }
}

// Warp sums of T per-lane values (one per KV head), stored by the lanes that
// end up holding them: a butterfly reduce-scatter for T = 1, 2, 4, 8.
template <int T>
__device__ __forceinline__ void reduce_and_store(float (&acc)[T], int lane, float* out, size_t stride, bool good) {
  if ((T & (T - 1)) == 0) {
    constexpr int LOG_T = (T >= 8) ? 3 : (T >= 4) ? 2 : (T >= 2) ? 1 : 0;
#pragma unroll
    for (int k = 0; k < LOG_T; ++k) {
      const int off = 16 >> k;
      const int half = T >> (k + 1);
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int e = 0; e < half; ++e) {
        const float lo_v = acc[e], hi_v = acc[e + half];
        const float send = upper ? lo_v : hi_v;
        acc[e] = (upper ? hi_v : lo_v) + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
#pragma unroll
    for (int off = 16 >> LOG_T; off > 0; off >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], off);
    if ((lane & ((32 >> LOG_T) - 1)) == 0) out[(size_t)(lane >> (5 - LOG_T)) * stride] = good ? acc[0] : -INFINITY;
  } else {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float v = acc[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) out[(size_t)t * stride] = good ? v : -INFINITY;
    }
  }
}

// D: head dim; T: 16-byte chunks per lane per page; U: pages in flight per warp.
// For D = 128 chunk t of every lane belongs to KV head t; for the latent cache
// (D = 576, one KV head) every chunk belongs to the one head.
template <int D, int T, int U, int MIN_BLOCKS>
__global__ void __launch_bounds__(kThreads, MIN_BLOCKS) score_pages_kernel(const ScoreArgs a) {
  // The block-table window of 32 pages is refreshed when k0 crosses a multiple
  // of 32, which k0 (a multiple of U) only hits exactly when U divides 32.
  static_assert(32 % U == 0, "U must divide 32");
  constexpr bool HEAD_PER_CHUNK = (D == 128);
  extern __shared__ __align__(16) uint8_t smem[];
  const int H = a.kv.num_kv_heads;
  const int chunks = H * D / 4;  // 16-byte chunks per page block
  float* pn = reinterpret_cast<float*>(smem);                  // [2][H][2][D]
  float* slice_part = pn + 2 * H * 2 * D;                      // [slices][H][2][D]
  int* prefix = reinterpret_cast<int*>(slice_part + pn_slices(H * D / 8, a.group) * H * 2 * D);  // [batch + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Candidate pages per request, then an exclusive prefix (one warp, chunked).
  for (int b = threadIdx.x; b < a.batch; b += kThreads) {
    int L = a.seq_lens[b];
    if (L < 0 || L > a.max_seq_len) {
      raise_error(a.err, SE_DEVERR_LENGTH);
      L = L < 0 ? 0 : a.max_seq_len;
    }
    prefix[b + 1] = max((L + kPageSize - 1) / kPageSize - 1, 0);
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (a.batch + 31) / 32;
    const int lo = min(a.batch, lane * per), hi = min(a.batch, lo + per);
    int sum = 0;
    for (int b = lo; b < hi; ++b) sum += prefix[b + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - sum;
    if (lane == 0) prefix[0] = 0;
    for (int b = lo; b < hi; ++b) {
      run += prefix[b + 1];
      prefix[b + 1] = run;
    }
  }
  __syncthreads();
  const int total = prefix[a.batch];
  const int per_cta = (total + gridDim.x - 1) / gridDim.x;
  const int start = blockIdx.x * per_cta;
  const int end = min(total, start + per_cta);
  if (start >= end) return;

  const int b_first = find_request(prefix, a.batch, start);
  const int b_last = find_request(prefix, a.batch, end - 1);
  int seg = 0;
  for (int b = b_first; b <= b_last; ++b) {
    const int lo = max(start, prefix[b]), hi = min(end, prefix[b + 1]);  // flattened ids
    if (lo >= hi) continue;
    // ---- P and N of request b into buffer seg & 1. The group is cut into
    // `slices` runs of query heads so that every thread has a few independent
    // loads in flight; slice partials are then added in slice order (fixed
    // order: the result does not depend on timing). The other buffer may still
    // be read by nobody: each lane copies its multipliers into registers right
    // after the barrier below.
    float* buf = pn + (seg & 1) * H * 2 * D;
    const uint16_t* qb = a.q + (size_t)b * H * a.group * D;
    const int items = H * D / 8;
    const int slices = pn_slices(items, a.group);
    for (int task = threadIdx.x; task < items * slices; task += kThreads) {
      const int it = task % items, sl = task / items;
      const int h = it / (D / 8), c0 = (it % (D / 8)) * 8;
      const int g0 = sl * a.group / slices, g1 = (sl + 1) * a.group / slices;
      float P[8], N[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) P[e] = N[e] = 0.f;
      const uint16_t* qh = qb + (size_t)h * a.group * D + c0;
      int g = g0;
      for (; g + 4 <= g1; g += 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const uint4*>(qh + (size_t)(g + u) * D);
#pragma unroll
        for (int u = 0; u < 4; ++u) add_pos_neg(v[u], P, N);
      }
      for (; g < g1; ++g) add_pos_neg(*reinterpret_cast<const uint4*>(qh + (size_t)g * D), P, N);
      float* part = slice_part + (size_t)sl * H * 2 * D;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        part[(h * 2 + 0) * D + c0 + e] = N[e];  // multiplies the min row
        part[(h * 2 + 1) * D + c0 + e] = P[e];  // multiplies the max row
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < H * 2 * D; i += kThreads) {
      float acc = slice_part[i];
      for (int sl = 1; sl < slices; ++sl) acc += slice_part[(size_t)sl * H * 2 * D + i];
      buf[i] = acc;
    }
    __syncthreads();
    float mult[T][8];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int j = lane + 32 * t;
      const bool in = j < chunks;
      const int h = in ? j / (D / 4) : 0;
      const int row = in ? (j % (D / 4)) / (D / 8) : 0;
      const int c0 = in ? (j % (D / 8)) * 8 : 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) mult[t][e] = in ? buf[(h * 2 + row) * D + c0 + e] : 0.f;
    }
    ++seg;

    // ---- this warp's pages of the segment: lo + warp, lo + warp + 8, ...
    const int first = lo + warp;
    const int npages = first < hi ? (hi - first + kWarps - 1) / kWarps : 0;
    const int32_t* bt_row = a.block_table + (size_t)b * a.bt_stride;
    const int p_first = first - prefix[b];  // page id of this warp's first page
    float* out_b = a.scores + (size_t)b * H * a.score_stride;
    // Block-table entries for 32 of this warp's pages at a time; the next 32 prefetched.
    int phys_cur = lane < npages ? bt_row[p_first + kWarps * lane] : -1;
    int phys_nxt = lane + 32 < npages ? bt_row[p_first + kWarps * (lane + 32)] : -1;
    for (int k0 = 0; k0 < npages; k0 += U) {
      if (k0 > 0 && (k0 & 31) == 0) {
        phys_cur = phys_nxt;
        phys_nxt = k0 + 32 + lane < npages ? bt_row[p_first + kWarps * (k0 + 32 + lane)] : -1;
      }
      uint4 v[U][T];
      int ph[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        ph[u] = __shfl_sync(0xffffffffu, phys_cur, (k0 + u) & 31);
        const bool live = k0 + u < npages && ph[u] >= 0 && ph[u] < a.kv.num_pages;
        const uint4* blk = reinterpret_cast<const uint4*>(a.kv.summary + (size_t)(live ? ph[u] : 0) * H * 2 * D);
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const int j = lane + 32 * t;
          v[u][t] = (live && j < chunks) ? ld_stream_v4(blk + j) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (k0 + u < npages) {
          const bool good = ph[u] >= 0 && ph[u] < a.kv.num_pages;
          if (!good && lane == 0) raise_error(a.err, SE_DEVERR_PAGE_RANGE);
          float acc[T];
#pragma unroll
          for (int t = 0; t < T; ++t) acc[t] = 0.f;
#pragma unroll
          for (int t = 0; t < T; ++t) {
            if (HEAD_PER_CHUNK) acc[t] = dot8(v[u][t], mult[t], acc[t]);
            else acc[0] = dot8(v[u][t], mult[t], acc[0]);
          }
          float* out = out_b + p_first + kWarps * (k0 + u);
          if (HEAD_PER_CHUNK) {
            reduce_and_store<T>(acc, lane, out, a.score_stride, good);
          } else {
            float r[1] = {acc[0]};
            reduce_and_store<1>(r, lane, out, a.score_stride, good);
          }
        }
      }
    }
  }
}

template <int D, int T, int U, int MIN_BLOCKS>
cudaError_t launch_t(const ScoreArgs& a, int sm_count, cudaStream_t stream) {
  const int H = a.kv.num_kv_heads;
  const size_t smem = (size_t)(2 + pn_slices(H * D / 8, a.group)) * H * 2 * D * 4 + (size_t)(a.batch + 1) * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(score_pages_kernel<D, T, U, MIN_BLOCKS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  score_pages_kernel<D, T, U, MIN_BLOCKS><<<sm_count * MIN_BLOCKS, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool score_pages_supported(int num_kv_heads, int head_dim) {
  return (head_dim == 128 && num_kv_heads >= 1 && num_kv_heads <= 8) || (head_dim == 576 && num_kv_heads == 1);
}

cudaError_t launch_score_pages(const KvView& kv, const uint16_t* q, int32_t num_q_heads,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                               int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                               int sm_count, unsigned* err, cudaStream_t stream) {
  const int max_cand = (max_seq_len + kPageSize - 1) / kPageSize - 1;
  if (batch == 0 || max_cand <= 0) return cudaSuccess;
  ScoreArgs a;
  a.kv = kv;
  a.q = q;
  a.group = num_q_heads / kv.num_kv_heads;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq_len = max_seq_len;
  a.scores = scores;
  a.score_stride = score_stride;
  a.err = err;
  // U pages in flight per warp keep about 16 16-byte loads per lane outstanding.
  if (kv.head_dim == 576) return launch_t<576, 5, 4, 1>(a, sm_count, stream);
  switch (kv.num_kv_heads) {
    case 1: return launch_t<128, 1, 16, 2>(a, sm_count, stream);
    case 2: return launch_t<128, 2, 8, 2>(a, sm_count, stream);
    case 3: return launch_t<128, 3, 4, 2>(a, sm_count, stream);
    case 4: return launch_t<128, 4, 4, 2>(a, sm_count, stream);
    case 5: return launch_t<128, 5, 4, 1>(a, sm_count, stream);
    case 6: return launch_t<128, 6, 4, 1>(a, sm_count, stream);
    case 7: return launch_t<128, 7, 2, 1>(a, sm_count, stream);
    default: return launch_t<128, 8, 2, 1>(a, sm_count, stream);
  }
}

}  // namespace se
