// Quest page selection (SparseEngine: Sparse-First Inference Engine, Figure 2
// caption and Table 14: Quest is the query-dependent retrieval method; Table 10:
// a selected-token budget of 2,048 is 128 pages, kept tokens beyond the budget
// are listed separately).
//
//  * score_pages_kernel: the Quest upper bound of every candidate page, for all
//    KV heads of a request at once. The per-channel bound of one query head,
//    max(q*min, q*max), summed over the heads of a GQA group equals
//    max*P + min*N with P (N) the sum of the group's positive (negative) query
//    parts, so the kernel pre-reduces the group's query once and then streams
//    the summaries: 1 multiply-add per 2 bytes, memory-bound. A producer warp
//    moves each page's contiguous summary block (all KV heads) into a shared
//    ring with bulk TMA copies; consumer warps reduce it.
//  * topk_pages_kernel: per (request, KV head), an exact radix select (4 passes
//    of 8 bits) over order-preserving integer keys of the fp32 scores, ties to
//    the lower page id, output in ascending page order, plus the always-kept
//    last page.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kScoreConsumerWarps = 4;
constexpr int kScoreThreads = (kScoreConsumerWarps + 1) * 32;
constexpr int kScoreRingBytes = 32 * 1024;
constexpr int kMaxScoreStages = 32;

__device__ __forceinline__ int clamp_len(int L, int max_len, unsigned* err) {
  if (L < 0 || L > max_len) {
    raise_error(err, SE_DEVERR_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  return L;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Shared-memory layout of the scoring CTA:
//   [ring: nstage x stage_bytes][PN: H x 2 x D fp32][full: nstage][empty: nstage][meta: nstage]
__global__ void __launch_bounds__(kScoreThreads) score_pages_kernel(
    KvView kv, const uint16_t* __restrict__ q, int32_t group, const int32_t* __restrict__ block_table,
    int32_t bt_stride, const int32_t* __restrict__ seq_lens, int32_t max_seq_len, float* __restrict__ scores,
    int32_t score_stride, int32_t pages_per_cta, int32_t nstage, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int H = kv.num_kv_heads, D = kv.head_dim;
  const int stage_bytes = H * 2 * D * 2;
  float* PN = reinterpret_cast<float*>(smem + (size_t)nstage * stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(PN + H * 2 * D);
  uint64_t* empty = full + nstage;
  int* meta = reinterpret_cast<int*>(empty + nstage);

  const int b = blockIdx.y;
  const int L = clamp_len(seq_lens[b], max_seq_len, err);
  const int n_cand = max((L + kPageSize - 1) / kPageSize - 1, 0);
  const int p0 = blockIdx.x * pages_per_cta;
  if (p0 >= n_cand) return;
  const int cnt = min(pages_per_cta, n_cand - p0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_fence_init();
  }
  // Group pre-reduction: P = sum of positive parts, N = sum of negative parts.
  const uint16_t* qb = q + (size_t)b * H * group * D;
  for (int i = threadIdx.x; i < H * D; i += kScoreThreads) {
    const int h = i / D, c = i % D;
    float pos = 0.f, neg = 0.f;
    for (int g = 0; g < group; ++g) {
      const float x = __uint_as_float((uint32_t)qb[(size_t)(h * group + g) * D + c] << 16);
      pos += fmaxf(x, 0.f);
      neg += fminf(x, 0.f);
    }
    PN[(h * 2 + 0) * D + c] = pos;
    PN[(h * 2 + 1) * D + c] = neg;
  }
  __syncthreads();

  if (warp == kScoreConsumerWarps) {
    // ---------------- producer warp
    const uint64_t policy = l2_evict_first_policy();
    const int32_t* bt = block_table + (size_t)b * bt_stride + p0;
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < cnt && ok; base += 32) {
      const int my_phys = (base + lane < cnt) ? bt[base + lane] : 0;
      const int m = min(32, cnt - base);
      for (int j = 0; j < m; ++j) {
        const int phys = __shfl_sync(0xffffffffu, my_phys, j);
        const int i = base + j, s = i % nstage;
        if (lane == 0) {
          if (i >= nstage && !mbar_wait(&empty[s], ((i / nstage) - 1) & 1)) {
            raise_error(err, SE_DEVERR_WAIT_TIMEOUT);
            ok = false;
          } else if (phys < 0 || phys >= kv.num_pages) {
            raise_error(err, SE_DEVERR_PAGE_RANGE);
            meta[s] = 0;
            mbar_arrive(&full[s]);
            ++issued;
          } else {
            meta[s] = 1;
            mbar_arrive_expect_tx(&full[s], stage_bytes);
            tma_load_bulk(smem + (size_t)s * stage_bytes, kv.summary + (size_t)phys * H * 2 * D, stage_bytes,
                          &full[s], policy);
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        if (!ok) break;
      }
    }
    // Drain: the copies this CTA issued have landed before the producer leaves.
    if (lane == 0) {
      for (int i = max(0, issued - nstage); i < issued; ++i) {
        if (!mbar_wait(&full[i % nstage], (i / nstage) & 1)) raise_error(err, SE_DEVERR_WAIT_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- consumer warps
  float* out = scores + (size_t)b * H * score_stride + p0;
  for (int i = warp; i < cnt; i += kScoreConsumerWarps) {
    const int s = i % nstage;
    if (!mbar_wait(&full[s], (i / nstage) & 1)) {
      if (lane == 0) raise_error(err, SE_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(smem + (size_t)s * stage_bytes);
    const bool good = meta[s] != 0;
    for (int h = 0; h < H; ++h) {
      float acc = 0.f;
      if (good) {
        const uint16_t* mn = blk + h * 2 * D;
        const float* P = PN + (h * 2 + 0) * D;
        const float* N = PN + (h * 2 + 1) * D;
        for (int c = 2 * lane; c < D; c += 64) {
          const uint32_t lo = *reinterpret_cast<const uint32_t*>(mn + c);
          const uint32_t hi = *reinterpret_cast<const uint32_t*>(mn + D + c);
          const float2 pp = *reinterpret_cast<const float2*>(P + c);
          const float2 nn = *reinterpret_cast<const float2*>(N + c);
          acc = fmaf(bf16_lo(hi), pp.x, acc);
          acc = fmaf(bf16_hi(hi), pp.y, acc);
          acc = fmaf(bf16_lo(lo), nn.x, acc);
          acc = fmaf(bf16_hi(lo), nn.y, acc);
        }
        acc = warp_sum(acc);
      }
      if (lane == 0) out[(size_t)h * score_stride + i] = good ? acc : -INFINITY;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// ------------------------------------------------------------------ top-k
constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkThreads) topk_pages_kernel(
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

cudaError_t launch_score_pages(const KvView& kv, const uint16_t* q, int32_t num_q_heads,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                               int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                               int sm_count, unsigned* err, cudaStream_t stream) {
  const int max_cand = (max_seq_len + kPageSize - 1) / kPageSize - 1;
  if (batch == 0 || max_cand <= 0) return cudaSuccess;
  const int H = kv.num_kv_heads, D = kv.head_dim;
  const int stage_bytes = H * 2 * D * 2;
  int nstage = kScoreRingBytes / stage_bytes;
  nstage = nstage < 4 ? 4 : (nstage > kMaxScoreStages ? kMaxScoreStages : nstage);
  // About 8 waves of 4 CTAs per SM over the upper bound of candidate pages.
  const long long total = (long long)batch * max_cand;
  long long per = total / ((long long)sm_count * 32);
  per = ((per + 31) / 32) * 32;
  const int pages_per_cta = (int)(per < 32 ? 32 : (per > 512 ? 512 : per));
  const size_t smem = (size_t)nstage * stage_bytes + (size_t)H * 2 * D * 4 + (size_t)nstage * 16 + nstage * 4;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(score_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         96 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((max_cand + pages_per_cta - 1) / pages_per_cta, batch);
  score_pages_kernel<<<grid, kScoreThreads, smem, stream>>>(kv, q, num_q_heads / H, block_table, bt_stride,
                                                             seq_lens, max_seq_len, scores, score_stride,
                                                             pages_per_cta, nstage, err);
  return cudaGetLastError();
}

size_t topk_smem_bytes(int32_t max_seq_len) {
  const int max_cand = (max_seq_len + kPageSize - 1) / kPageSize - 1;
  return (size_t)(max_cand > 0 ? max_cand : 1) * 4;
}

cudaError_t launch_topk_pages(const float* scores, int32_t score_stride, const int32_t* seq_lens, int32_t batch,
                              int32_t num_kv_heads, int32_t max_seq_len, int32_t topk, int32_t* out_pages,
                              int32_t* out_counts, int32_t sel_stride, unsigned* err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const size_t smem = topk_smem_bytes(max_seq_len);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  topk_pages_kernel<<<batch * num_kv_heads, kTopkThreads, smem, stream>>>(
      scores, score_stride, seq_lens, num_kv_heads, max_seq_len, topk, out_pages, out_counts, sel_stride, err);
  return cudaGetLastError();
}

}  // namespace se
