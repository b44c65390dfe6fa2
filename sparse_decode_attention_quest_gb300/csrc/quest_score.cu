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
// The slice is cut at request boundaries into segments. Each of the 8 warps
// takes every eighth page of a segment and streams the pages' summary blocks
// (all KV heads of a page, contiguous) through its own ring of R stages in
// shared memory with 16-byte cp.async copies, R - 1 blocks in flight; the
// physical page ids sit in lanes, two 32-page windows per warp. The first
// copies of a segment go out before the CTA computes P and N of the request
// (all threads; double-buffered in shared memory); every lane then keeps its
// share of the multipliers in registers as MMA operands. The dot product of a
// page block with the multipliers runs on the m16n8k16 bf16 MMA: for each KV
// head, B holds the 2 D summary channels as 8 x (2 D / 8) blocks, A the
// matching multipliers split into a bf16 high part (rows 0-7) and low part
// (rows 8-15), and the score is the sum of the diagonals of the two 8x8 halves
// of D (exact bf16 products, fp32 sums; the split keeps about 17 bits of each
// multiplier). A page of H heads costs H ldmatrix and 2 H MMAs (d 128) plus a
// butterfly reduce-scatter across the KV heads. On GB300, random 2 KB blocks gathered by
// every warp through its own ring reach close to the copy bandwidth; loads
// batched into registers do not, because a warp drains its batch before it
// issues the next one.
//
// With a workspace (se_quest_score_pages_ws) pn_kernel first writes P and N of
// every request, and the scoring kernel reads them (an L2 hit) instead of
// reducing the group's queries in every CTA that scores part of a request.
// That in-CTA reduction waits on query loads that queue behind the summary
// reads of the other CTAs: measured on GB300, 12.7 us at the start of the
// latent kernel (64 query heads x 576 channels per request) and 15 us again in
// the CTAs whose slice reaches a second request, which then finish last.
// With the workspace the equal slices hold only kStaticPct percent of the
// pages: the SMs of a GB300 gather at different speeds (steadily, from launch
// to launch), so the rest is a pool of kUnit-page units that each warp takes
// from, one atomic ticket per unit, once its own pages are scored. A unit is
// streamed by one warp through the same ring (a unit that crosses a request
// boundary is two runs). The scores do not depend on which warp computes them.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStaticPct = 75;  // share of the pages in the equal static slices (with precomputed multipliers)
constexpr int kUnit = 8;        // pages per unit of the pool that follows them
constexpr int kPoolMinPages = 128;  // fair share per CTA below which every page is in the static slices

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
  const float* pn_pre;  // P and N per request, [batch][H][2][D], from pn_kernel (or null)
  unsigned* units;      // units of the pool taken so far (zeroed by pn_kernel; null without pn_pre)
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

// Two 8x8 bf16 matrices from shared memory (lanes 0-15 give the row addresses).
__device__ __forceinline__ void ldmatrix_x2(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// An fp32 multiplier as the sum of two bf16 values (high part, then the
// rounded remainder): the pair carries about 17 bits of the mantissa.
__device__ __forceinline__ void split_bf16(float x, float& hi, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(x));
  lo = x - hi;
}

// Channel of a head's 2 D summary channels (min row, then max row) that the
// MMA below pairs with k-index k of row n: 8-channel runs, n-major inside each
// block of 64, so the eight rows of one 8x8 operand matrix are 128 contiguous
// bytes (conflict-free ldmatrix).
__device__ __forceinline__ int chan(int k, int n) { return (k >> 3) * 64 + n * 8 + (k & 7); }

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

// cp.async of 16 bytes into shared memory, and its group bookkeeping.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Lanes per (KV head, 8 channels) item in the P/N pre-reduction: the group's
// query heads are cut into S runs summed by S adjacent lanes.
__host__ __device__ __forceinline__ int pn_lanes(int group) { return group >= 8 ? 8 : group >= 4 ? 4 : group >= 2 ? 2 : 1; }

// D: head dim; T: 16-byte chunks per lane per page block (= KV heads at d 128);
// R: ring stages per warp.
// For D = 128 chunk t of every lane belongs to KV head t; for the latent cache
// (D = 576, one KV head) every chunk belongs to the one head.
// kPre: the multipliers of every request were written by pn_kernel before
// this kernel; a segment reads them from global memory (an L2 hit) instead of
// reducing the group's queries itself, and no CTA barrier is needed.
template <int D, int T, int R, bool kPre>
__global__ void __launch_bounds__(kThreads, 2) score_pages_kernel(const ScoreArgs a) {
  // With the multipliers from pn_kernel (kPre), the launch before this one, the
  // lengths, block table and summaries were complete when it started: the
  // copies start at once and a thread waits for pn_kernel only before it first
  // reads the multipliers or takes a unit of the pool, and before it exits.
  if (!kPre) pdl_wait();
  pdl_launch_dependents();
  // Page i + R - 1 is looked up while page i is consumed, inside the two
  // 32-page block-table windows [base, base + 64) a warp holds.
  static_assert(R >= 2 && R <= 17, "ring depth");
  constexpr int kHeads = D == 128 ? T : 1;      // KV heads in a page's summary block
  constexpr int kKsPerHead = 2 * D / 128;        // MMA k-steps over a head's 2 D channels
  constexpr int kBlk = kHeads * 2 * D * 2;       // bytes of one page's summary block
  constexpr int kChunks = kBlk / 16;
  extern __shared__ __align__(16) uint8_t smem[];
  const int H = a.kv.num_kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + (size_t)warp * R * kBlk;                            // [warp][R][kBlk]
  float* pn = reinterpret_cast<float*>(smem + (size_t)kWarps * R * kBlk);    // [2][H][2][D] (not with kPre)
  int* prefix = reinterpret_cast<int*>(pn + (kPre ? 0 : 2 * H * 2 * D));   // [batch + 1]
  const uint32_t ring_addr = smem_addr(ring);

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
  // With the precomputed multipliers (kPre) the kernel balances its end: each
  // CTA takes an equal static slice of kStaticPct percent of the pages, and a
  // warp that has finished its part takes units of kUnit consecutive pages
  // from the rest, one atomic ticket per unit (pn_kernel zeroes the counter).
  // The SMs of a GB300 stream at different speeds, steadily so from launch to
  // launch; with equal slices the last CTA ended 11 us after the mean one.
  // Small launches (under kPoolMinPages per CTA) keep equal slices: there the
  // units' ticket and block-table round trips cost more than the balance wins.
  const bool pool = kPre && a.units != nullptr && total >= kPoolMinPages * (int)gridDim.x;
  const int per_cta = pool ? (int)((long long)total * kStaticPct / 100 / gridDim.x)
                           : (int)((total + gridDim.x - 1) / gridDim.x);
  const int start = min(total, (int)blockIdx.x * per_cta);
  const int end = min(total, start + per_cta);

  // A fragments of the m16n8k16 MMA: row n < 8 holds the high parts and row
  // n + 8 the low parts of the multipliers of channels chan(k, n); k-step s
  // of head h covers the head's channels 128 s .. 128 s + 127.
  uint32_t afrag[kHeads * kKsPerHead][4];
  int afrag_b = -1;  // request whose multipliers afrag holds (kPre)
  auto multipliers_from = [&](const float* buf) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int h = 0; h < kHeads; ++h)
#pragma unroll
      for (int s = 0; s < kKsPerHead; ++s) {
        const float* mh = buf + h * 2 * D;
        float hi[4], lo[4];
        const int k0 = 16 * s + 2 * t;
        split_bf16(mh[chan(k0, g)], hi[0], lo[0]);
        split_bf16(mh[chan(k0 + 1, g)], hi[1], lo[1]);
        split_bf16(mh[chan(k0 + 8, g)], hi[2], lo[2]);
        split_bf16(mh[chan(k0 + 9, g)], hi[3], lo[3]);
        uint32_t* f = afrag[h * kKsPerHead + s];
        f[0] = pack_bf16x2(hi[0], hi[1]);
        f[1] = pack_bf16x2(lo[0], lo[1]);
        f[2] = pack_bf16x2(hi[2], hi[3]);
        f[3] = pack_bf16x2(lo[2], lo[3]);
      }
  };
  auto precomputed = [&](int b) {
    if (b != afrag_b) {
      if (afrag_b < 0) pdl_wait();  // pn_kernel's multipliers
      multipliers_from(a.pn_pre + (size_t)b * H * 2 * D);
      afrag_b = b;
    }
  };

  // This warp's pages first, first + stride, ... (npages of them, all of
  // request b): their physical ids sit in lanes, two windows of 32 pages; the
  // blocks stream through the warp's ring and the scores are stored.
  // `prepare` runs once the first R - 1 copies are out and sets up afrag.
  auto stream_pages = [&](int b, int first, int npages, int stride, auto&& prepare) {
    const int32_t* bt_row = a.block_table + (size_t)b * a.bt_stride;
    const int p_first = first - prefix[b];  // page id of this warp's first page
    auto phys_of = [&](int i) { return i < npages ? bt_row[p_first + stride * i] : -1; };
    int base = 0;
    int ph_cur = phys_of(lane), ph_nxt = phys_of(lane + 32);
    auto lookup = [&](int i) {
      const int c = __shfl_sync(0xffffffffu, ph_cur, i & 31), n = __shfl_sync(0xffffffffu, ph_nxt, i & 31);
      return i < base + 32 ? c : n;
    };
    // Copies of page i into stage i % R; a page id outside the pool is not read.
    auto issue = [&](int i) {
      const int ph = lookup(i);
      if (ph >= 0 && ph < a.kv.num_pages) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.kv.summary) + (size_t)ph * kBlk;
        const uint32_t dst = ring_addr + (i % R) * kBlk;
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const int j = lane + 32 * t;
          if (j < kChunks) cp_async16(dst + j * 16, src + j * 16);
        }
      }
    };
#pragma unroll 1
    for (int i = 0; i < R - 1; ++i) {
      if (i < npages) issue(i);
      cp_async_commit();
    }
    prepare();

    float* out_b = a.scores + (size_t)b * H * a.score_stride;
    for (int i = 0; i < npages; ++i) {
      // Page i has left the first window: rotate; the new window is first
      // looked up about 32 - R pages later.
      if (i == base + 32) {
        base += 32;
        ph_cur = ph_nxt;
        ph_nxt = phys_of(base + 32 + lane);
      }
      if (i + R - 1 < npages) issue(i + R - 1);
      cp_async_commit();
      cp_async_wait<R - 1>();  // page i has landed (this lane's copies)
      __syncwarp();            // ... and every lane's
      const int ph = lookup(i);
      const bool good = ph >= 0 && ph < a.kv.num_pages;
      if (!good && lane == 0) raise_error(a.err, SE_DEVERR_PAGE_RANGE);
      // Per head: D = A B with B[k][n] = summary channel chan(k, n); the head's
      // score is the sum of the diagonal of D's two 8x8 halves (high and low).
      const uint32_t st = ring_addr + (i % R) * kBlk;
      float acc[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t hb = st + h * 4 * D;
#pragma unroll
        for (int s = 0; s + 1 < kKsPerHead; s += 2) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(b0, b1, b2, b3, hb + s * 256 + (lane >> 3) * 128 + (lane & 7) * 16);
          const uint32_t* f0 = afrag[h * kKsPerHead + s];
          const uint32_t* f1 = afrag[h * kKsPerHead + s + 1];
          mma_bf16_16816(d, f0[0], f0[1], f0[2], f0[3], b0, b1);
          mma_bf16_16816(d, f1[0], f1[1], f1[2], f1[3], b2, b3);
        }
        if (kKsPerHead & 1) {  // the last, unpaired k-step
          constexpr int s = kKsPerHead - 1;
          uint32_t b0, b1;
          ldmatrix_x2(b0, b1, hb + s * 256 + ((lane >> 3) & 1) * 128 + (lane & 7) * 16);
          const uint32_t* f = afrag[h * kKsPerHead + s];
          mma_bf16_16816(d, f[0], f[1], f[2], f[3], b0, b1);
        }
        const int g = lane >> 2, t = lane & 3;
        acc[h] = (2 * t == g ? d[0] + d[2] : 0.f) + (2 * t + 1 == g ? d[1] + d[3] : 0.f);
      }
      __syncwarp();  // every lane has read stage i % R before it is refilled
      float* out = out_b + p_first + stride * i;
      reduce_and_store<kHeads>(acc, lane, out, a.score_stride, good);
    }
    cp_async_wait<0>();  // nothing of these pages is in flight when the ring is reused
    __syncwarp();
  };

  // ---- the static slice, cut at request boundaries into segments; each of
  // the 8 warps takes every eighth page of a segment.
  if (start < end) {
    const int b_first = find_request(prefix, a.batch, start);
    const int b_last = find_request(prefix, a.batch, end - 1);
    int seg = 0;
    for (int b = b_first; b <= b_last; ++b) {
      const int lo = max(start, prefix[b]), hi = min(end, prefix[b + 1]);  // flattened ids
      if (lo >= hi) continue;
      const int first = lo + warp;
      const int npages = first < hi ? (hi - first + kWarps - 1) / kWarps : 0;
      stream_pages(b, first, npages, kWarps, [&]() {
        if (kPre) {
          precomputed(b);
        } else {
          // P and N of request b reduced here into buffer seg & 1. Each
          // (KV head, 8 channels) item is summed by S adjacent lanes over S
          // runs of the group's query heads and the runs are added with a
          // fixed butterfly (the result does not depend on timing). The other
          // buffer may still be read by nobody: each lane copies its
          // multipliers into registers right after the barrier below.
          float* wbuf = pn + (seg & 1) * H * 2 * D;
          const uint16_t* qb = a.q + (size_t)b * H * a.group * D;
          const int S = pn_lanes(a.group);
          const int tasks = H * (D / 8) * S;
          for (int t0 = warp * 32; t0 < tasks; t0 += kThreads) {  // warp-uniform
            const int task = t0 + lane;
            const bool live = task < tasks;
            const int it = task / S, sl = task % S;
            const int h = it / (D / 8), c0 = (it % (D / 8)) * 8;
            float P[8], N[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) P[e] = N[e] = 0.f;
            if (live) {
              const int g0 = sl * a.group / S, g1 = (sl + 1) * a.group / S;
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
            }
            for (int o = 1; o < S; o <<= 1) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                P[e] += __shfl_xor_sync(0xffffffffu, P[e], o);
                N[e] += __shfl_xor_sync(0xffffffffu, N[e], o);
              }
            }
            if (live && sl == 0) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                wbuf[(h * 2 + 0) * D + c0 + e] = N[e];  // multiplies the min row
                wbuf[(h * 2 + 1) * D + c0 + e] = P[e];  // multiplies the max row
              }
            }
          }
          __syncthreads();
          multipliers_from(wbuf);
        }
      });
      ++seg;
    }
  }

  // ---- the pool: units of kUnit consecutive pages, taken by whichever warp
  // is free (a unit that crosses a request boundary is two runs).
  if (pool) {
    pdl_wait();  // pn_kernel zeroes the unit counter
    const int dyn0 = per_cta * (int)gridDim.x;
    while (true) {
      unsigned u = 0;
      if (lane == 0) u = atomicAdd(a.units, 1u);
      u = __shfl_sync(0xffffffffu, u, 0);
      const long long u_lo = (long long)dyn0 + (long long)u * kUnit;
      if (u_lo >= total) break;
      const int p_hi = min(total, (int)u_lo + kUnit);
      for (int p = (int)u_lo; p < p_hi;) {
        const int b = find_request(prefix, a.batch, p);
        const int r_hi = min(p_hi, prefix[b + 1]);
        stream_pages(b, p, r_hi - p, 1, [&]() { precomputed(b); });
        p = r_hi;
      }
    }
  }
  pdl_wait();  // completes after pn_kernel, like every other launch
}

constexpr int kPnThreads = 640;  // up to 640 tasks in one round (d 128 with 5 KV heads; the latent 576)

// P and N of every request into pn_out [batch][H][2][D]: one CTA per request,
// the same tasks, lanes and summation order as the pre-reduction inside
// score_pages_kernel, so both give bit-identical multipliers. All loads of a
// task's run are issued before the first is summed.
template <int D>
__global__ void __launch_bounds__(kPnThreads) pn_kernel(const uint16_t* __restrict__ q, int32_t H, int32_t group,
                                                  float* __restrict__ pn_out, unsigned* __restrict__ units) {
  pdl_enter();
  const int b = blockIdx.x;
  if (b == 0 && threadIdx.x == 0) *units = 0u;  // the scoring kernel's pool starts empty
  const int lane = threadIdx.x & 31;
  const int S = pn_lanes(group);
  const int tasks = H * (D / 8) * S;
  const uint16_t* qb = q + (size_t)b * H * group * D;
  float* dst = pn_out + (size_t)b * H * 2 * D;
  for (int t0 = threadIdx.x - lane; t0 < tasks; t0 += blockDim.x) {  // warp-uniform
    const int task = t0 + lane;
    const bool live = task < tasks;
    const int it = task / S, sl = task % S;
    const int h = it / (D / 8), c0 = (it % (D / 8)) * 8;
    float P[8], N[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) P[e] = N[e] = 0.f;
    if (live) {
      const int g0 = sl * group / S, g1 = (sl + 1) * group / S;
      const uint16_t* qh = qb + (size_t)h * group * D + c0;
      for (int g = g0; g < g1; g += 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (g + u < g1) v[u] = *reinterpret_cast<const uint4*>(qh + (size_t)(g + u) * D);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (g + u < g1) add_pos_neg(v[u], P, N);
      }
    }
    for (int o = 1; o < S; o <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        P[e] += __shfl_xor_sync(0xffffffffu, P[e], o);
        N[e] += __shfl_xor_sync(0xffffffffu, N[e], o);
      }
    }
    if (live && sl == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dst[(h * 2 + 0) * D + c0 + e] = N[e];
        dst[(h * 2 + 1) * D + c0 + e] = P[e];
      }
    }
  }
}

template <int D, int T, int R, bool kPre>
cudaError_t launch_score(const ScoreArgs& a, int sm_count, cudaStream_t stream) {
  const int H = a.kv.num_kv_heads;
  constexpr int kBlk = D == 128 ? T * 512 : 2 * D * 2;
  const size_t smem =
      (size_t)kWarps * R * kBlk + (kPre ? 0 : (size_t)2 * H * 2 * D * 4) + (size_t)(a.batch + 1) * 4;
  cudaError_t e = cudaFuncSetAttribute(score_pages_kernel<D, T, R, kPre>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  {
    const cudaError_t le = launch_pdl(score_pages_kernel<D, T, R, kPre>, dim3(sm_count * 2), dim3(kThreads), smem,
                                      stream, a);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

template <int D, int T, int R>
cudaError_t launch_t(const ScoreArgs& a, int sm_count, cudaStream_t stream) {
  if (!a.pn_pre) return launch_score<D, T, R, false>(a, sm_count, stream);
  const int H = a.kv.num_kv_heads;
  const int tasks = H * (D / 8) * pn_lanes(a.group);
  const int threads = min(kPnThreads, (tasks + 31) / 32 * 32);
  {
    const cudaError_t le = launch_pdl(pn_kernel<D>, dim3(a.batch), dim3(threads), 0, stream, a.q, H, a.group,
                                      const_cast<float*>(a.pn_pre), a.units);
    if (le != cudaSuccess) return le;
  }
  return launch_score<D, T, R, true>(a, sm_count, stream);
}

}  // namespace

size_t score_pn_bytes(int32_t batch, int32_t num_kv_heads, int32_t head_dim) {
  // P and N, then the pool's unit counter (16 bytes)
  return (size_t)batch * num_kv_heads * 2 * head_dim * sizeof(float) + 16;
}

bool score_pages_supported(int num_kv_heads, int head_dim) {
  return (head_dim == 128 && num_kv_heads >= 1 && num_kv_heads <= 8) || (head_dim == 576 && num_kv_heads == 1);
}

cudaError_t launch_score_pages(const KvView& kv, const uint16_t* q, int32_t num_q_heads,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                               int32_t batch, int32_t max_seq_len, float* scores, int32_t score_stride,
                               float* pn_ws, int sm_count, unsigned* err, cudaStream_t stream) {
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
  a.pn_pre = pn_ws;
  a.units = pn_ws ? reinterpret_cast<unsigned*>(pn_ws + (size_t)batch * kv.num_kv_heads * 2 * kv.head_dim) : nullptr;
  a.err = err;
  // Ring depth per head count: about 96 KB of summary blocks in flight per CTA,
  // two CTAs per SM.
  if (kv.head_dim == 576) return launch_t<576, 5, 5>(a, sm_count, stream);
  switch (kv.num_kv_heads) {
    case 1: return launch_t<128, 1, 16>(a, sm_count, stream);
    case 2: return launch_t<128, 2, 12>(a, sm_count, stream);
    case 3: return launch_t<128, 3, 8>(a, sm_count, stream);
    case 4: return launch_t<128, 4, 6>(a, sm_count, stream);
    case 5: return launch_t<128, 5, 4>(a, sm_count, stream);
    case 6: return launch_t<128, 6, 4>(a, sm_count, stream);
    case 7: return launch_t<128, 7, 3>(a, sm_count, stream);
    default: return launch_t<128, 8, 3>(a, sm_count, stream);
  }
}

}  // namespace se
