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
// (request-major). Each CTA takes an equal slice of it, so ragged lengths are
// balanced, and streams its slice through a shared-memory ring:
//  * a producer warp looks up the block table and issues one bulk TMA copy per
//    page of the page's whole summary block (all KV heads, contiguous);
//  * four consumer warps take every fourth page. At each request boundary they
//    compute P and N for the new request together (double-buffered in shared
//    memory), then every lane keeps the multipliers of its own 16-byte chunks
//    in registers. A page costs one 16-byte shared load, 8 multiply-adds per
//    chunk and a butterfly reduce-scatter across the KV heads.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRingBytes = 32 * 1024;
constexpr int kCtasPerSm = 4;

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
  int32_t nstage;
  unsigned* err;
};

// Largest b in [0, n - 1] with prefix[b] <= x (prefix non-decreasing, prefix[0] = 0): the
// request whose candidate range holds x (empty requests are skipped).
__device__ __forceinline__ int find_request(const int* prefix, int n, int x) {
  int lo = 0, hi = n;  // prefix[lo] <= x
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void named_barrier_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
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

// D: head dim; T: 16-byte chunks per lane per page (= KV heads for D = 128).
template <int D, int T>
__global__ void __launch_bounds__(kThreads) score_pages_kernel(const ScoreArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.kv.num_kv_heads;
  const int stage_bytes = H * 2 * D * 2;
  const int chunks = H * D / 4;  // 16-byte chunks per page block
  uint8_t* ring = smem;
  float* pn = reinterpret_cast<float*>(smem + (size_t)a.nstage * stage_bytes);  // [2][H][2][D]
  int* prefix = reinterpret_cast<int*>(pn + 2 * H * 2 * D);                      // [batch + 1]
  uint64_t* full = reinterpret_cast<uint64_t*>(prefix + ((a.batch + 2) & ~1));
  uint64_t* empty = full + a.nstage;
  int2* meta = reinterpret_cast<int2*>(empty + a.nstage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_fence_init();
  }
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
  const int cnt = end - start;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    const uint64_t policy = l2_evict_first_policy();
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < cnt && ok; base += 32) {
      int b = 0, p = -1, phys = -1;
      if (base + lane < cnt) {
        const int idx = start + base + lane;
        b = find_request(prefix, a.batch, idx);
        p = idx - prefix[b];
        phys = a.block_table[(size_t)b * a.bt_stride + p];
      }
      const int m = min(32, cnt - base);
      for (int j = 0; j < m; ++j) {
        const int bj = __shfl_sync(0xffffffffu, b, j);
        const int pj = __shfl_sync(0xffffffffu, p, j);
        const int ph = __shfl_sync(0xffffffffu, phys, j);
        const int i = base + j, s = i % a.nstage;
        if (lane == 0) {
          if (i >= a.nstage && !mbar_wait(&empty[s], ((i / a.nstage) - 1) & 1)) {
            raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            ok = false;
          } else if (ph < 0 || ph >= a.kv.num_pages) {
            raise_error(a.err, SE_DEVERR_PAGE_RANGE);
            meta[s] = make_int2(bj, -1 - pj);  // negative: skip the page, write -inf
            mbar_arrive(&full[s]);
            ++issued;
          } else {
            meta[s] = make_int2(bj, pj);
            mbar_arrive_expect_tx(&full[s], stage_bytes);
            tma_load_bulk(ring + (size_t)s * stage_bytes, a.kv.summary + (size_t)ph * H * 2 * D, stage_bytes,
                          &full[s], policy);
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        if (!ok) break;
      }
    }
    if (lane == 0) {  // drain: every copy issued by this CTA has landed
      for (int i = max(0, issued - a.nstage); i < issued; ++i)
        if (!mbar_wait(&full[i % a.nstage], (i / a.nstage) & 1)) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int ctid = threadIdx.x;  // 0 .. 127
  const int b_first = find_request(prefix, a.batch, start);
  const int b_last = find_request(prefix, a.batch, end - 1);
  int seg = 0;
  bool dead = false;  // after a timed-out wait: keep passing the barriers, skip the pages
  for (int b = b_first; b <= b_last; ++b) {
    const int lo = max(start, prefix[b]) - start, hi = min(end, prefix[b + 1]) - start;
    if (lo >= hi) continue;
    // P and N of request b into buffer seg & 1 (all consumer threads).
    float* buf = pn + (seg & 1) * H * 2 * D;
    const uint16_t* qb = a.q + (size_t)b * H * a.group * D;
    for (int task = ctid; task < H * D / 8; task += kConsumerWarps * 32) {
      const int h = task / (D / 8), c0 = (task % (D / 8)) * 8;
      float P[8], N[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) P[e] = N[e] = 0.f;
      for (int g = 0; g < a.group; ++g) {
        const uint4 v = *reinterpret_cast<const uint4*>(qb + (size_t)(h * a.group + g) * D + c0);
        const float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                            bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          P[e] += fmaxf(x[e], 0.f);
          N[e] += fminf(x[e], 0.f);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        buf[(h * 2 + 0) * D + c0 + e] = N[e];  // multiplies the min row
        buf[(h * 2 + 1) * D + c0 + e] = P[e];  // multiplies the max row
      }
    }
    named_barrier_consumers();
    // This lane's chunk j = lane + 32 t: head j / (D/4), row (min/max) and 8 channels.
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
    // Pages lo..hi-1 of this request that belong to this warp.
    int i = lo + ((warp - lo % kConsumerWarps) + kConsumerWarps) % kConsumerWarps;
    for (; i < hi && !dead; i += kConsumerWarps) {
      const int s = i % a.nstage;
      if (!mbar_wait(&full[s], (i / a.nstage) & 1)) {
        if (lane == 0) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
        dead = true;
        break;
      }
      const int2 md = meta[s];
      const bool good = md.y >= 0;
      const int p = good ? md.y : -1 - md.y;
      float acc[T];
#pragma unroll
      for (int t = 0; t < T; ++t) acc[t] = 0.f;
      if (good) {
        const uint4* blk = reinterpret_cast<const uint4*>(ring + (size_t)s * stage_bytes);
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const int j = lane + 32 * t;
          if (j < chunks) {
            const uint4 v = blk[j];
            if (D == 128) acc[t] = dot8(v, mult[t], acc[t]);
            else acc[0] = dot8(v, mult[t], acc[0]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      float* out = a.scores + (size_t)b * H * a.score_stride + p;
      if (D == 128 && (T & (T - 1)) == 0) {
        // Butterfly reduce-scatter: after log2(T) exchanges lane l holds head l >> (5 - log2 T).
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
            const float keep = upper ? hi_v : lo_v;
            acc[e] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
        }
#pragma unroll
        for (int off = 16 >> LOG_T; off > 0; off >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], off);
        if ((lane & ((32 >> LOG_T) - 1)) == 0) {
          const int h = lane >> (5 - LOG_T);
          out[(size_t)h * a.score_stride] = good ? acc[0] : -INFINITY;
        }
      } else if (D == 128) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
          float v = acc[t];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == 0) out[(size_t)t * a.score_stride] = good ? v : -INFINITY;
        }
      } else {
        float v = acc[0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) out[0] = good ? v : -INFINITY;
      }
    }
  }
}

template <int D, int T>
cudaError_t launch_t(const ScoreArgs& a, int sm_count, cudaStream_t stream) {
  const int H = a.kv.num_kv_heads;
  const size_t smem = (size_t)a.nstage * H * 2 * D * 2 + (size_t)2 * H * 2 * D * 4 +
                      (size_t)((a.batch + 2) & ~1) * 4 + (size_t)a.nstage * 16 + (size_t)a.nstage * 8;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(score_pages_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  score_pages_kernel<D, T><<<sm_count * kCtasPerSm, kThreads, smem, stream>>>(a);
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
  const int H = kv.num_kv_heads, D = kv.head_dim;
  const int stage_bytes = H * 2 * D * 2;
  int nstage = kRingBytes / stage_bytes;
  nstage = nstage < 4 ? 4 : (nstage > 32 ? 32 : nstage);
  ScoreArgs a;
  a.kv = kv;
  a.q = q;
  a.group = num_q_heads / H;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq_len = max_seq_len;
  a.scores = scores;
  a.score_stride = score_stride;
  a.nstage = nstage;
  a.err = err;
  if (D == 576) return launch_t<576, 5>(a, sm_count, stream);
  switch (H) {
    case 1: return launch_t<128, 1>(a, sm_count, stream);
    case 2: return launch_t<128, 2>(a, sm_count, stream);
    case 3: return launch_t<128, 3>(a, sm_count, stream);
    case 4: return launch_t<128, 4>(a, sm_count, stream);
    case 5: return launch_t<128, 5>(a, sm_count, stream);
    case 6: return launch_t<128, 6>(a, sm_count, stream);
    case 7: return launch_t<128, 7>(a, sm_count, stream);
    default: return launch_t<128, 8>(a, sm_count, stream);
  }
}

}  // namespace se
