// Quest page selection, per (request, KV head) (SparseEngine: Sparse-First
// Inference Engine, Table 10 caption: selected budgets exclude separately kept
// tokens; Table 10, Quest (Vortex) row: 2,048 selected tokens are 128 pages).
//
// Exact top-k over the fp32 page scores: the keys are order-preserving 32-bit
// integers of the scores; a radix select of 4 passes x 8 bits finds the k-th
// largest key T and how many keys equal to T are still needed; the output is
// every key above T plus the lowest-index keys equal to T (ties go to the lower
// page id), written in ascending page order, followed by the always-kept last
// page. All integer work: the result is exact for the given fp32 scores.
//
//  * topk_pages_reg_kernel (up to 8192 candidates): 1024 threads, each holding
//    8 consecutive scores in registers; a 1024-bucket histogram between the
//    scores' min and max finds the bucket of the k-th largest, whose members
//    are then ranked exactly (a radix select restricted to that bucket when it
//    is crowded), and two block scans write the ordered output.
//  * topk_pages_smem_kernel (longer contexts): keys in dynamic shared memory.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kKeysPerThread = 8;
constexpr int kRegMaxCand = kTopkThreads * kKeysPerThread;

__device__ __forceinline__ int clamp_len(int L, int max_len, unsigned* err) {
  if (L < 0 || L > max_len) {
    raise_error(err, SE_DEVERR_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  return L;
}

// Candidate pages [c0, c1) of a request of L tokens in n pages: the pages that
// hold none of the first `sink` tokens and none of the last `recent` tokens;
// the last page (the newest token) is always kept, so c1 <= n - 1.
__device__ __forceinline__ void candidate_window(int L, int n, int sink, int recent, int& c0, int& c1) {
  const int rf = L > recent ? (L - recent) / kPageSize : 0;
  c1 = max(0, min(rf, n - 1));
  c0 = min((min(sink, L) + kPageSize - 1) / kPageSize, c1);
}

// Writes the kept pages outside the window: 0 .. c0 - 1 first, c1 .. n - 1
// after the k selected ones.
__device__ __forceinline__ void write_kept_windows(int32_t* out, int c0, int c1, int n, int k, int tid) {
  for (int i = tid; i < c0; i += kTopkThreads) out[i] = i;
  for (int j = tid; j < n - c1; j += kTopkThreads) out[c0 + k + j] = c1 + j;
}

// Larger float -> larger key (IEEE order; -0 sorts just below +0).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The digit of the k-th largest key in a 256-bin histogram (counts of keys that
// match the prefix so far), and the number of keys in higher bins. Every lane
// of the calling warp gets the answer.
__device__ __forceinline__ void find_digit(const int* hist, int remaining, int lane, int& digit, int& above) {
  int g[8], gsum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    g[j] = hist[lane * 8 + j];
    gsum += g[j];
  }
  int incl = gsum;  // keys in bins >= lane * 8
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += t;
  }
  const int up = incl - gsum;
  const bool mine = up < remaining && remaining <= incl;
  int d = 0, a = 0;
  if (mine) {
    int cum = up;
    for (int j = 7; j >= 0; --j) {
      if (cum + g[j] >= remaining) {
        d = lane * 8 + j;
        a = cum;
        break;
      }
      cum += g[j];
    }
  }
  const unsigned who = __ballot_sync(0xffffffffu, mine);
  const int src = who ? __ffs(who) - 1 : 0;
  digit = __shfl_sync(0xffffffffu, d, src);
  above = __shfl_sync(0xffffffffu, a, src);
}

constexpr int kBuckets = 1024;
constexpr int kMaxMembers = 1024;

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums over the per-warp values wtot[0..31] (one per warp of the block, in
// shared memory): lane l of every warp reads wtot[l] and the warp adds them up
// with shuffles, instead of every thread reading all 32. Returns the sum over
// the warps before `warp`; `total` gets the sum over all of them.
__device__ __forceinline__ int warps_before(const int* wtot, int warp, int lane, int& total) {
  const int x = wtot[lane];
  total = warp_sum(x);
  return warp_sum(lane < warp ? x : 0);
}

// Block-wide exclusive prefix of one int per thread, in thread order (two barriers).
__device__ __forceinline__ int block_exclusive_scan(int v, int* wtot, int warp, int lane, int& total) {
  static_assert(kTopkWarps == 32, "one warp total per lane");
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  const int before = incl - v + warps_before(wtot, warp, lane, total);
  __syncthreads();
  return before;
}

// Up to 8192 candidates, 8 consecutive scores per thread in registers.
//  1. min and max of the finite scores; 1024 linear buckets between them (the
//     bucket index is monotone in the score, so the order is kept);
//  2. histogram, and the bucket B holding the k-th largest score: every score
//     in a higher bucket is selected;
//  3. the members of bucket B are ranked exactly (score, then lower page id)
//     by brute force; if B holds more than 1024 members (near-identical scores)
//     a 4-pass radix select restricted to B finds the exact threshold instead;
//  4. the selected page ids are written in ascending order (block scan).
__global__ void __launch_bounds__(kTopkThreads) topk_pages_reg_kernel(
    const float* __restrict__ scores, int32_t score_stride, const int32_t* __restrict__ seq_lens, int32_t H,
    int32_t max_seq_len, int32_t k, int32_t sink, int32_t recent, int32_t* __restrict__ out_pages,
    int32_t* __restrict__ out_counts, int32_t sel_stride, unsigned* err) {
  pdl_enter();
  __shared__ int hist[kBuckets];
  __shared__ float s_min[kTopkWarps], s_max[kTopkWarps];
  __shared__ int wtot[kTopkWarps];
  __shared__ float mem_val[kMaxMembers];
  __shared__ int mem_idx[kMaxMembers];
  __shared__ unsigned selbits[kRegMaxCand / 32];
  __shared__ int rhist[3][257];
  __shared__ int s_info[4];  // bucket B, keys above B, members collected
  const int bh = blockIdx.x, b = bh / H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The scores are loaded from the first candidate of a request of at least
  // `sink` tokens before the length arrives, so that the two loads overlap;
  // a shorter request (another first candidate) loads them again below.
  const int c0_guess = min((sink + kPageSize - 1) / kPageSize, score_stride);
  const int guess_lim = min(kRegMaxCand, score_stride - c0_guess);
  float x[kKeysPerThread];
  {
    const float* sg = scores + (size_t)bh * score_stride + c0_guess;
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) {
      const int i = tid * kKeysPerThread + e;
      x[e] = i < guess_lim ? sg[i] : -INFINITY;
    }
  }
  const int L = clamp_len(seq_lens[b], max_seq_len, err);
  const int n = (L + kPageSize - 1) / kPageSize;
  int c0, c1;
  candidate_window(L, n, sink, recent, c0, c1);
  const int C = min(c1 - c0, kRegMaxCand);  // candidate i is page c0 + i
  int32_t* out = out_pages + (size_t)bh * sel_stride;
  if (C <= k) {
    for (int i = tid; i < n; i += kTopkThreads) out[i] = i;
    if (tid == 0) out_counts[bh] = n;
    return;
  }
  write_kept_windows(out, c0, c1, n, k, tid);
  if (c0 != c0_guess) {
    const float* sc = scores + (size_t)bh * score_stride + c0;
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) {
      const int i = tid * kKeysPerThread + e;
      x[e] = i < C ? sc[i] : -INFINITY;
    }
  }
  float lmin = INFINITY, lmax = -INFINITY;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    const int i = tid * kKeysPerThread + e;
    if (i >= C) x[e] = -INFINITY;
    if (i < C && isfinite(x[e])) {
      lmin = fminf(lmin, x[e]);
      lmax = fmaxf(lmax, x[e]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lmin = fminf(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
    lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  }
  if (lane == 0) {
    s_min[warp] = lmin;
    s_max[warp] = lmax;
  }
  hist[tid] = 0;
  if (tid < kRegMaxCand / 32) selbits[tid] = 0u;
  if (tid < 2 * 257) (&rhist[0][0])[tid] = 0;
  if (tid == 0) s_info[2] = 0;
  __syncthreads();
  float mn = s_min[lane], mx = s_max[lane];  // min and max over the warps, by shuffles
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float scale = (mx > mn) ? (float)kBuckets / (mx - mn) : 0.f;
  int bk[kKeysPerThread];
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    int bb = 0;
    if (isfinite(x[e])) bb = min(kBuckets - 1, max(0, (int)((x[e] - mn) * scale)));
    else if (x[e] > 0.f) bb = kBuckets - 1;  // +inf; -inf and NaN stay in bucket 0
    bk[e] = bb;
    if (tid * kKeysPerThread + e < C) atomicAdd(&hist[bb], 1);
  }
  __syncthreads();
  // Suffix counts over the buckets (thread i owns bucket i): keys in buckets >= i.
  const int hc = hist[tid];
  int incl = hc;  // within the warp, from the top: lanes above hold higher buckets
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += t;
  }
  if (lane == 0) wtot[warp] = incl;
  __syncthreads();
  {
    const int x = wtot[lane];
    incl += warp_sum(lane > warp ? x : 0);  // keys in the buckets of the warps above
  }
  if (incl - hc < k && k <= incl) {
    s_info[0] = tid;
    s_info[1] = incl - hc;
  }
  __syncthreads();
  const int B = s_info[0];
  const int need = k - s_info[1];  // members of bucket B to take, >= 1
  const int m = hist[B];
  if (m <= kMaxMembers) {
    // Exact ranking of the members of bucket B.
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) {
      const int i = tid * kKeysPerThread + e;
      if (i < C && bk[e] == B) {
        const int slot = atomicAdd(&s_info[2], 1);
        mem_val[slot] = x[e];
        mem_idx[slot] = i;
      }
    }
    __syncthreads();
    if (tid < m) {
      const float v = mem_val[tid];
      const int id = mem_idx[tid];
      const uint32_t kv = order_key(v);
      int rank = 0;
      for (int j = 0; j < m; ++j) {
        const uint32_t kj = order_key(mem_val[j]);
        rank += (kj > kv || (kj == kv && mem_idx[j] < id)) ? 1 : 0;
      }
      if (rank < need) atomicOr(&selbits[id >> 5], 1u << (id & 31));
    }
    __syncthreads();
  } else {
    // Radix select among the members of bucket B (4 passes x 8 bits).
    uint32_t key[kKeysPerThread];
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) key[e] = order_key(x[e]);
    uint32_t prefix = 0, mask = 0;
    int remaining = need;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int* hh = rhist[pass % 3];
      if (pass >= 1)
        for (int i = tid; i < 257; i += kTopkThreads) rhist[(pass + 1) % 3][i] = 0;
#pragma unroll
      for (int e = 0; e < kKeysPerThread; ++e) {
        const int i = tid * kKeysPerThread + e;
        if (i < C && bk[e] == B && (key[e] & mask) == prefix) atomicAdd(&hh[(key[e] >> shift) & 255u], 1);
      }
      __syncthreads();
      int d, above;
      find_digit(hh, remaining, lane, d, above);
      remaining -= above;
      prefix |= (uint32_t)d << shift;
      mask |= 255u << shift;
    }
    // Members above the threshold key, then the first `remaining` equal to it.
    int n_eq = 0;
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e)
      n_eq += (tid * kKeysPerThread + e < C && bk[e] == B && key[e] == prefix) ? 1 : 0;
    int tot;
    int r = block_exclusive_scan(n_eq, wtot, warp, lane, tot);
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) {
      const int i = tid * kKeysPerThread + e;
      if (i < C && bk[e] == B) {
        bool take = key[e] > prefix;
        if (key[e] == prefix) {
          take = r < remaining;
          ++r;
        }
        if (take) atomicOr(&selbits[i >> 5], 1u << (i & 31));
      }
    }
    __syncthreads();
  }
  // Output in ascending page order.
  bool selv[kKeysPerThread];
  int n_sel = 0;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    const int i = tid * kKeysPerThread + e;
    selv[e] = i < C && (bk[e] > B || (bk[e] == B && ((selbits[i >> 5] >> (i & 31)) & 1u)));
    n_sel += selv[e] ? 1 : 0;
  }
  int tot;
  int pos = block_exclusive_scan(n_sel, wtot, warp, lane, tot);
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    if (selv[e]) {
      if (pos < k) out[c0 + pos] = c0 + tid * kKeysPerThread + e;
      ++pos;
    }
  }
  if (tid == 0) out_counts[bh] = c0 + k + (n - c1);
}

__global__ void __launch_bounds__(kTopkThreads) topk_pages_smem_kernel(
    const float* __restrict__ scores, int32_t score_stride, const int32_t* __restrict__ seq_lens, int32_t H,
    int32_t max_seq_len, int32_t k, int32_t sink, int32_t recent, int32_t* __restrict__ out_pages,
    int32_t* __restrict__ out_counts, int32_t sel_stride, unsigned* err) {
  pdl_enter();
  extern __shared__ uint32_t keys[];
  __shared__ int hist[257];
  __shared__ int warp_tot[kTopkWarps];
  __shared__ int s_digit, s_above;
  const int bh = blockIdx.x, b = bh / H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = clamp_len(seq_lens[b], max_seq_len, err);
  const int n = (L + kPageSize - 1) / kPageSize;
  int c0, c1;
  candidate_window(L, n, sink, recent, c0, c1);
  const int C = c1 - c0;  // candidate i is page c0 + i
  int32_t* out = out_pages + (size_t)bh * sel_stride;
  if (C <= k) {
    for (int i = tid; i < n; i += kTopkThreads) out[i] = i;
    if (tid == 0) out_counts[bh] = n;
    return;
  }
  write_kept_windows(out, c0, c1, n, k, tid);
  const float* sc = scores + (size_t)bh * score_stride + c0;
  for (int i = tid; i < C; i += kTopkThreads) keys[i] = order_key(sc[i]);

  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 257; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < C; i0 += kTopkThreads) {
      const int i = i0 + tid;
      int digit = 256;
      if (i < C) {
        const uint32_t u = keys[i];
        if ((u & mask) == prefix) digit = (int)((u >> shift) & 255u);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (digit < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      int g[8], gsum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        g[j] = hist[lane * 8 + j];
        gsum += g[j];
      }
      int incl = gsum;  // count in bins >= lane*8
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += t;
      }
      const int above = incl - gsum;
      if (above < remaining && remaining <= incl) {
        int cum = above;
        for (int j = 7; j >= 0; --j) {
          if (cum + g[j] >= remaining) {
            s_digit = lane * 8 + j;
            s_above = cum;
            break;
          }
          cum += g[j];
        }
      }
    }
    __syncthreads();
    remaining -= s_above;
    prefix |= (uint32_t)s_digit << shift;
    mask |= 255u << shift;
    __syncthreads();
  }

  // Keys above the threshold, then the lowest-index keys equal to it.
  const uint32_t T = prefix;
  const int need_eq = remaining;
  const unsigned lt_mask = (1u << lane) - 1u;
  int base_out = 0, eq_seen = 0;
  for (int i0 = 0; i0 < C; i0 += kTopkThreads) {
    const int i = i0 + tid;
    const uint32_t u = i < C ? keys[i] : 0u;
    const bool gt = i < C && u > T;
    const bool eq = i < C && u == T;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_tot[warp] = __popc(beq);
    __syncthreads();
    int eq_total;
    const int eq_before = warps_before(warp_tot, warp, lane, eq_total);
    __syncthreads();
    const int eq_rank = eq_seen + eq_before + __popc(beq & lt_mask);
    const bool sel = gt || (eq && eq_rank < need_eq);
    const unsigned bsel = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) warp_tot[warp] = __popc(bsel);
    __syncthreads();
    int sel_total;
    const int sel_before = warps_before(warp_tot, warp, lane, sel_total);
    const int pos = base_out + sel_before + __popc(bsel & lt_mask);
    if (sel && pos < k) out[c0 + pos] = c0 + i;
    base_out += sel_total;
    eq_seen += eq_total;
    __syncthreads();
  }
  if (tid == 0) out_counts[bh] = c0 + k + (n - c1);
}

}  // namespace

size_t topk_smem_bytes(int32_t max_seq_len) {
  const int max_cand = (max_seq_len + kPageSize - 1) / kPageSize - 1;
  return max_cand <= kRegMaxCand ? 0 : (size_t)max_cand * 4;
}

cudaError_t launch_topk_pages(const float* scores, int32_t score_stride, const int32_t* seq_lens, int32_t batch,
                              int32_t num_kv_heads, int32_t max_seq_len, int32_t topk, int32_t sink_tokens,
                              int32_t recent_tokens, int32_t* out_pages, int32_t* out_counts, int32_t sel_stride,
                              unsigned* err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const int max_cand = (max_seq_len + kPageSize - 1) / kPageSize - 1;
  if (max_cand <= kRegMaxCand) {
    {
      const cudaError_t le = launch_pdl(topk_pages_reg_kernel, dim3(batch * num_kv_heads), dim3(kTopkThreads), 0,
                                        stream, scores, score_stride, seq_lens, num_kv_heads, max_seq_len, topk,
                                        sink_tokens, recent_tokens, out_pages, out_counts, sel_stride, err);
      if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
  }
  const size_t smem = topk_smem_bytes(max_seq_len);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_pages_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  {
    const cudaError_t le = launch_pdl(topk_pages_smem_kernel, dim3(batch * num_kv_heads), dim3(kTopkThreads), smem,
                                      stream, scores, score_stride, seq_lens, num_kv_heads, max_seq_len, topk,
                                      sink_tokens, recent_tokens, out_pages, out_counts, sel_stride, err);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace se
