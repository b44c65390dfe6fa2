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
//    8 consecutive keys in registers; one barrier per radix pass (three
//    rotating histograms, the digit search done redundantly by every warp) and
//    two block scans for the ordered output.
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

__global__ void __launch_bounds__(kTopkThreads) topk_pages_reg_kernel(
    const float* __restrict__ scores, int32_t score_stride, const int32_t* __restrict__ seq_lens, int32_t H,
    int32_t max_seq_len, int32_t k, int32_t* __restrict__ out_pages, int32_t* __restrict__ out_counts,
    int32_t sel_stride, unsigned* err) {
  __shared__ int hist[3][257];
  __shared__ int wtot_eq[kTopkWarps], wtot_sel[kTopkWarps];
  const int bh = blockIdx.x, b = bh / H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = clamp_len(seq_lens[b], max_seq_len, err);
  const int n = (L + kPageSize - 1) / kPageSize;
  const int C = min(max(n - 1, 0), kRegMaxCand);
  int32_t* out = out_pages + (size_t)bh * sel_stride;
  if (C <= k) {
    for (int i = tid; i < n; i += kTopkThreads) out[i] = i;
    if (tid == 0) out_counts[bh] = n;
    return;
  }
  const float* sc = scores + (size_t)bh * score_stride;
  uint32_t key[kKeysPerThread];
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    const int i = tid * kKeysPerThread + e;
    key[e] = i < C ? order_key(sc[i]) : 0u;
  }
  for (int i = tid; i < 2 * 257; i += kTopkThreads) (&hist[0][0])[i] = 0;
  __syncthreads();

  uint32_t prefix = 0, mask = 0;
  int remaining = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int* h = hist[pass % 3];
    if (pass >= 1)  // buffer of the next pass; its last readers passed the previous barrier
      for (int i = tid; i < 257; i += kTopkThreads) hist[(pass + 1) % 3][i] = 0;
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) {
      const int i = tid * kKeysPerThread + e;
      const bool in = i < C && (key[e] & mask) == prefix;
      const int digit = in ? (int)((key[e] >> shift) & 255u) : 256;
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&h[digit], __popc(peers));
    }
    __syncthreads();
    int d, above;
    find_digit(h, remaining, lane, d, above);
    remaining -= above;
    prefix |= (uint32_t)d << shift;
    mask |= 255u << shift;
  }

  // Output in ascending index order: every key above T, then the first
  // `need_eq` keys equal to T.
  const uint32_t T = prefix;
  const int need_eq = remaining;
  int n_eq = 0;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) n_eq += (tid * kKeysPerThread + e < C && key[e] == T) ? 1 : 0;
  int incl = n_eq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wtot_eq[warp] = incl;
  __syncthreads();
  int eq_rank = incl - n_eq;
  for (int w = 0; w < warp; ++w) eq_rank += wtot_eq[w];
  int n_sel = 0;
  {
    int r = eq_rank;
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) {
      const bool in = tid * kKeysPerThread + e < C;
      if (in && key[e] > T) ++n_sel;
      if (in && key[e] == T) {
        if (r < need_eq) ++n_sel;
        ++r;
      }
    }
  }
  incl = n_sel;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wtot_sel[warp] = incl;
  __syncthreads();
  int pos = incl - n_sel;
  for (int w = 0; w < warp; ++w) pos += wtot_sel[w];
  {
    int r = eq_rank;
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e) {
      const int i = tid * kKeysPerThread + e;
      const bool in = i < C;
      bool take = in && key[e] > T;
      if (in && key[e] == T) {
        take = r < need_eq;
        ++r;
      }
      if (take) {
        if (pos < k) out[pos] = i;
        ++pos;
      }
    }
  }
  if (tid == 0) {
    out[k] = n - 1;
    out_counts[bh] = k + 1;
  }
}


__global__ void __launch_bounds__(kTopkThreads) topk_pages_smem_kernel(
    const float* __restrict__ scores, int32_t score_stride, const int32_t* __restrict__ seq_lens, int32_t H,
    int32_t max_seq_len, int32_t k, int32_t* __restrict__ out_pages, int32_t* __restrict__ out_counts,
    int32_t sel_stride, unsigned* err) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[257];
  __shared__ int warp_tot[kTopkWarps];
  __shared__ int s_digit, s_above;
  const int bh = blockIdx.x, b = bh / H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = clamp_len(seq_lens[b], max_seq_len, err);
  const int n = (L + kPageSize - 1) / kPageSize;
  const int C = max(n - 1, 0);
  int32_t* out = out_pages + (size_t)bh * sel_stride;
  if (C <= k) {
    for (int i = tid; i < n; i += kTopkThreads) out[i] = i;
    if (tid == 0) out_counts[bh] = n;
    return;
  }
  const float* sc = scores + (size_t)bh * score_stride;
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
    int eq_before = 0, eq_total = 0;
    for (int w = 0; w < kTopkWarps; ++w) {
      const int v = warp_tot[w];
      eq_before += (w < warp) ? v : 0;
      eq_total += v;
    }
    __syncthreads();
    const int eq_rank = eq_seen + eq_before + __popc(beq & lt_mask);
    const bool sel = gt || (eq && eq_rank < need_eq);
    const unsigned bsel = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) warp_tot[warp] = __popc(bsel);
    __syncthreads();
    int sel_before = 0, sel_total = 0;
    for (int w = 0; w < kTopkWarps; ++w) {
      const int v = warp_tot[w];
      sel_before += (w < warp) ? v : 0;
      sel_total += v;
    }
    const int pos = base_out + sel_before + __popc(bsel & lt_mask);
    if (sel && pos < k) out[pos] = i;
    base_out += sel_total;
    eq_seen += eq_total;
    __syncthreads();
  }
  if (tid == 0) {
    out[k] = n - 1;
    out_counts[bh] = k + 1;
  }
}

}  // namespace

size_t topk_smem_bytes(int32_t max_seq_len) {
  const int max_cand = (max_seq_len + kPageSize - 1) / kPageSize - 1;
  return max_cand <= kRegMaxCand ? 0 : (size_t)max_cand * 4;
}

cudaError_t launch_topk_pages(const float* scores, int32_t score_stride, const int32_t* seq_lens, int32_t batch,
                              int32_t num_kv_heads, int32_t max_seq_len, int32_t topk, int32_t* out_pages,
                              int32_t* out_counts, int32_t sel_stride, unsigned* err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const int max_cand = (max_seq_len + kPageSize - 1) / kPageSize - 1;
  if (max_cand <= kRegMaxCand) {
    topk_pages_reg_kernel<<<batch * num_kv_heads, kTopkThreads, 0, stream>>>(
        scores, score_stride, seq_lens, num_kv_heads, max_seq_len, topk, out_pages, out_counts, sel_stride, err);
    return cudaGetLastError();
  }
  const size_t smem = topk_smem_bytes(max_seq_len);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_pages_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  topk_pages_smem_kernel<<<batch * num_kv_heads, kTopkThreads, smem, stream>>>(
      scores, score_stride, seq_lens, num_kv_heads, max_seq_len, topk, out_pages, out_counts, sel_stride, err);
  return cudaGetLastError();
}

}  // namespace se
