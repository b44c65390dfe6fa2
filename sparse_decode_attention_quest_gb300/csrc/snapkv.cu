// SnapKV-style eviction at the end of prefill (SparseEngine: Sparse-First
// Inference Engine, Table 8: 32-query scoring window, pooling kernel 7, 2,016
// selected + 32 recent tokens; Table 10: probability-based prefill scores;
// Table 15 note: eviction releases storage, so kept tokens are compacted).
//
// Per (request b, KV head h) with prompt length n and window W, the R = W * G
// window query rows r = (w, g) (query head g of h's group at position
// n - W + w) attend causally to keys j <= n - W + w:
//   pass 1   LSE_r = log sum_j exp(z_rj),         z_rj = sm_scale q_r . k_j
//   pass 2   s_j   = sum_r exp(z_rj - LSE_r)      for candidates j < n - W
//   select   s'_j  = max of s over [j - p/2, j + p/2] clipped to the candidates;
//            keep the top k of s' (ties: lower j) ascending, then n - W .. n - 1
//   compact  kept token t -> page t / 16, slot t % 16 of the destination table
//
// The logits are the one dense contraction of the path: 128 query rows x 128
// keys x 128 dims per tile, on the 5th-generation tensor cores. Warp roles:
//   warp 0      TMA producer: the 8 pages of a 128-key tile, two 64-column
//               boxes each with 128-byte swizzle, into a 4-stage ring;
//   warp 1      allocates 256 TMEM columns (two fp32 128x128 accumulators)
//               and issues the tcgen05.mma (M 128, N 128, K 16) x 8 per tile;
//   warps 2-9   epilogue, two warps per TMEM lane quarter: a thread owns query
//               row r (TMEM lane r) and 64 of the tile's 128 columns; it applies
//               the causal mask (boundary tiles only) and the online max/sum
//               (pass 1) or exp(z - LSE) (pass 2). Pass 2 sums the columns with
//               a warp transpose-reduce and a fixed-order merge of the four lane
//               quarters through shared memory (deterministic).
// The tiles of all (request, KV head) pairs form one flattened range; every
// CTA takes an equal slice. Pass 1 writes per-slice partial (max, sum) per row
// that pass 2 merges.
#include <cooperative_groups.h>

#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kD = 128;
constexpr int kTileN = 128;                   // keys per tile
constexpr int kPagesPerTile = kTileN / kPageSize;
constexpr int kHalfBytes = kTileN * 128;      // 128 rows x 128 bytes (64 dims)
constexpr int kTileBytes = 2 * kHalfBytes;    // 32 KB
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kMinTilesPerCta = 4;
constexpr int kTmemCols = 256;
constexpr float kLn2 = 0.6931471805599453f;

// Dynamic shared memory: [K ring 4 x 32 KB][Q 2 x 32 KB][colsum 2 x 4 x 128 fp32][prefix][barriers]
constexpr int kRingOff = 0;
constexpr int kQOff = kStages * kTileBytes;
constexpr int kColOff = kQOff + 2 * kTileBytes;
constexpr int kStatOff = kColOff + 2 * 4 * 128 * 4;   // pass 1: [128 rows][2] (max, sum) of column half 1
constexpr int kPrefixOff = kStatOff + 128 * 2 * 4;

struct SnapArgs {
  const uint16_t* qwin;  // [B][W][Hq][D]
  int32_t W, G, H, B;
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* lens;
  int32_t max_len;
  int32_t num_pages;
  float scale_log2;
  float* part;         // pass 1: [pairs][max_slices][128] x (max, sum), log2 domain
  int32_t* pair_ns;    // pass 1: slices per pair
  int32_t max_slices;
  float* row_lse;      // pass 2, optional: [pairs][R] natural log
  float* scores;       // pass 2: [pairs][score_stride]
  int32_t score_stride;
  unsigned* err;
};

__device__ __forceinline__ int find_pair(const int* prefix, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void named_barrier_epi() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Row r's log2-domain log-sum-exp of pair p from pass 1's per-slice (max, sum); +inf when the row saw no key.
__device__ __forceinline__ float merged_lse2(const SnapArgs& a, int p, int r) {
  const int ns = min(a.pair_ns[p], a.max_slices);
  const float* pr = a.part + ((size_t)p * a.max_slices * 128 + r) * 2;
  float M = -INFINITY;
  for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, pr[(size_t)s2 * 256]);
  float L = 0.f;
  for (int s2 = 0; s2 < ns; ++s2) {
    const float mm = pr[(size_t)s2 * 256];
    if (mm != -INFINITY) L += pr[(size_t)s2 * 256 + 1] * exp2f(mm - M);
  }
  return (L > 0.f) ? M + log2f(L) : INFINITY;
}

// Tiles of pair (b, h) for the pass: all keys (pass 1) or the candidates only (pass 2).
__device__ __forceinline__ int pair_tiles(int n, int W, int pass) {
  const int cols = pass == 1 ? n : max(n - W, 0);
  return (cols + kTileN - 1) / kTileN;
}

template <int PASS>
__global__ void __launch_bounds__(kThreads, 1) snapkv_scores_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                   const SnapArgs a) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int pairs = a.B * a.H;
  int* prefix = reinterpret_cast<int*>(smem + kPrefixOff);  // [pairs + 1]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPrefixOff + ((pairs + 2) & ~1) * 4);
  uint64_t* full = bars;                 // [4]
  uint64_t* empty = full + kStages;      // [4]
  uint64_t* acc_full = empty + kStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* q_full = acc_empty + 2;      // [2]
  uint64_t* q_empty = q_full + 2;        // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_empty + 2);
  float* colsum = reinterpret_cast<float*>(smem + kColOff);  // [2][4][128]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = a.W * a.G;

  // Tiles per pair and their exclusive prefix.
  for (int p = threadIdx.x; p < pairs; p += kThreads) {
    int n = a.lens[p / a.H];
    if (n < a.W || n > a.max_len) {
      raise_error(a.err, SE_DEVERR_LENGTH);
      n = n < a.W ? 0 : a.max_len;
    }
    prefix[p + 1] = pair_tiles(n, a.W, PASS);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiThreads);
      mbar_init(&q_full[i], kEpiThreads);
      mbar_init(&q_empty[i], 1);
    }
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  __syncthreads();
  if (warp == 0) {
    const int per = (pairs + 31) / 32;
    const int lo = min(pairs, lane * per), hi = min(pairs, lo + per);
    int sum = 0;
    for (int p = lo; p < hi; ++p) sum += prefix[p + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - sum;
    if (lane == 0) prefix[0] = 0;
    for (int p = lo; p < hi; ++p) {
      run += prefix[p + 1];
      prefix[p + 1] = run;
    }
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = prefix[pairs];
  const int per_cta = max(kMinTilesPerCta, (total + (int)gridDim.x - 1) / (int)gridDim.x);
  if (PASS == 1 && blockIdx.x == 0) {
    for (int p = threadIdx.x; p < pairs; p += kThreads) {
      const int p0 = prefix[p], cnt = prefix[p + 1] - p0;
      a.pair_ns[p] = cnt == 0 ? 0 : (p0 + cnt - 1) / per_cta - p0 / per_cta + 1;
    }
  }
  const int start = blockIdx.x * per_cta;
  const int end = min(total, start + per_cta);
  bool dead = false;  // a bounded wait gave up: finish without further waits

  if (start < end) {
    const int p_first = find_pair(prefix, pairs, start);
    const int p_last = find_pair(prefix, pairs, end - 1);
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t policy = l2_evict_first_policy();
      int it = 0;
      for (int p = p_first; p <= p_last; ++p) {
        const int t0 = max(start, prefix[p]) - prefix[p], t1 = min(end, prefix[p + 1]) - prefix[p];
        const int b = p / a.H, h = p % a.H;
        const int n = min(a.lens[b], a.max_len);
        const int npages = (n + kPageSize - 1) / kPageSize;
        // Block-table entries of 4 tiles per window (lane l: page l % 8 of tile
        // wb + l / 8); the next window is read 4 tiles before it is needed, so no
        // tile waits on a table lookup.
        const int32_t* bt_row = a.bt + (size_t)b * a.bt_stride;
        auto load_window = [&](int wt) {
          const int tt = wt + (lane >> 3), page = tt * kPagesPerTile + (lane & 7);
          int ph = -1;
          if (tt < t1 && page < npages) {
            ph = bt_row[page];
            if (ph < 0 || ph >= a.num_pages) {
              raise_error(a.err, SE_DEVERR_PAGE_RANGE);
              ph = -1;
            }
          }
          return ph;
        };
        int wb = t0, win_cur = load_window(t0), win_nxt = load_window(t0 + 4);
        for (int t = t0; t < t1; ++t, ++it) {
          const int s = it % kStages;
          if (t == wb + 4) {
            wb += 4;
            win_cur = win_nxt;
            win_nxt = load_window(wb + 4);
          }
          int phys = __shfl_sync(0xffffffffu, win_cur, (t - wb) * kPagesPerTile + (lane & 7));
          if (lane >= kPagesPerTile) phys = -1;
          if (it >= kStages && !dead && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1)) {
            if (lane == 0) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            dead = true;
          }
          const unsigned live = __ballot_sync(0xffffffffu, phys >= 0);
          if (lane == 0) mbar_arrive_expect_tx(&full[s], __popc(live) * 2 * kPageSize * 128);
          __syncwarp();
          if (phys >= 0 && !dead) {
            uint8_t* st = smem + kRingOff + s * kTileBytes + lane * kPageSize * 128;
            const int y = (phys * a.H + h) * kPageSize;
            tma_load_2d(st, &kmap, 0, y, &full[s], policy);
            tma_load_2d(st + kHalfBytes, &kmap, 64, y, &full[s], policy);
          }
        }
      }
      // Drain: every copy issued by this CTA has landed.
      if (lane == 0)
        for (int i = max(0, it - kStages); i < it && !dead; ++i)
          if (!mbar_wait(&full[i % kStages], (i / kStages) & 1)) dead = true;
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // Lane 0 alone: descriptors built once per Q buffer and stage, advanced by
      // constant offsets ((bytes >> 4) in the address field, no carry: every
      // shared address is below 256 KB).
      if (lane == 0) {
        const uint32_t idesc = umma_idesc_bf16(128, kTileN);
        int it = 0, acc_it = 0, seg = 0;
        // After a failed wait the loop goes on without MMAs but keeps committing,
        // so that the other roles' waits still complete.
        for (int p = p_first; p <= p_last; ++p) {
          const int t0 = max(start, prefix[p]) - prefix[p], t1 = min(end, prefix[p + 1]) - prefix[p];
          if (t0 >= t1) continue;
          const int qb = seg & 1;
          if (!dead && !mbar_wait(&q_full[qb], (seg >> 1) & 1)) {
            raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            dead = true;
          }
          tc05_fence_after();
          const uint64_t dq = umma_desc_sw128(smem_addr(smem + kQOff + qb * kTileBytes));
          for (int t = t0; t < t1; ++t, ++it, ++acc_it) {
            const int s = it % kStages, ab = acc_it & 1;
            if (!dead && (!mbar_wait(&full[s], (it / kStages) & 1) ||
                          (acc_it >= 2 && !mbar_wait(&acc_empty[ab], ((acc_it >> 1) - 1) & 1)))) {
              raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
              dead = true;
            }
            tc05_fence_after();
            if (!dead) {
              const uint64_t dk = umma_desc_sw128(smem_addr(smem + kRingOff + s * kTileBytes));
              const uint32_t d = tmem + ab * kTileN;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                constexpr uint64_t kHalfDesc = kHalfBytes >> 4;
                const uint64_t off = (uint64_t)(kk >> 2) * kHalfDesc + (uint64_t)(kk & 3) * 2;  // 32 bytes = 2
                tc05_mma_bf16(d, dq + off, dk + off, idesc, kk > 0 ? 1u : 0u);
              }
            }
            tc05_commit(&empty[s]);
            tc05_commit(&acc_full[ab]);
            if (t == t1 - 1) tc05_commit(&q_empty[qb]);
          }
          ++seg;
        }
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ epilogue
      const int wg = warp & 3;              // TMEM lane quarter of this warp
      const int chalf = (warp - 2) >> 2;    // which 64 of the tile's 128 columns
      const int r = wg * 32 + lane;         // query row = TMEM lane
      const int w_pos = r / a.G, g = r % a.G;
      const bool row_live = r < R;
      float* stat = reinterpret_cast<float*>(smem + kStatOff);
      int acc_it = 0, seg = 0, tile_ctr = 0;
      for (int p = p_first; p <= p_last; ++p) {
        const int t0 = max(start, prefix[p]) - prefix[p], t1 = min(end, prefix[p + 1]) - prefix[p];
        if (t0 >= t1) continue;
        const int b = p / a.H, h = p % a.H;
        const int n = min(a.lens[b], a.max_len);
        const int qb = seg & 1;
        // Query row r, dims [64 chalf, 64 chalf + 64), into Q buffer qb (swizzled, zero past R).
        if (seg >= 2 && !dead && !mbar_wait(&q_empty[qb], ((seg >> 1) - 1) & 1)) {
          raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
          dead = true;
        }
        {
          uint8_t* qt = smem + kQOff + qb * kTileBytes + chalf * kHalfBytes;
          const uint16_t* qrow = a.qwin + (((size_t)b * a.W + w_pos) * (a.H * a.G) + h * a.G + g) * kD + chalf * 64;
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {
            const uint4 v = row_live ? *reinterpret_cast<const uint4*>(qrow + q8 * 8) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(qt + swz128(r, q8)) = v;
          }
          fence_proxy_async_smem();
          mbar_arrive(&q_full[qb]);
        }
        float m_run = -INFINITY, l_run = 0.f, lse2 = INFINITY;
        if (PASS == 2) {
          lse2 = merged_lse2(a, p, r);  // +inf: the row contributes nothing
          if (a.row_lse && t0 == 0 && row_live && chalf == 0)
            a.row_lse[(size_t)p * R + r] = lse2 != INFINITY ? lse2 * kLn2 : -INFINITY;
        }
        const int limit = n - a.W + w_pos;  // last key this row sees
        for (int t = t0; t < t1; ++t, ++acc_it, ++tile_ctr) {
          const int ab = acc_it & 1;
          if (!dead && !mbar_wait(&acc_full[ab], (acc_it >> 1) & 1)) {
            raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            dead = true;
          }
          tc05_fence_after();
          const int jc = t * kTileN + chalf * 64;  // first column of this thread's half
          uint32_t raw[2][32];
          {
            const uint32_t row_addr = tmem + ((uint32_t)(wg * 32) << 16) + ab * kTileN + chalf * 64;
            tmem_ld32(row_addr, raw[0]);
            tmem_ld32(row_addr + 32, raw[1]);
            tmem_ld_wait();
          }
          tc05_fence_before();
          mbar_arrive(&acc_empty[ab]);  // the accumulator can take the next tile's MMA
          if (PASS == 1) {
            const bool interior = row_live && jc + 63 <= limit;  // every column visible
            float x[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const float z = __uint_as_float(raw[c >> 5][c & 31]) * a.scale_log2;
              x[c] = (interior || (row_live && jc + c <= limit)) ? z : -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) mx = fmaxf(mx, x[c]);
            const float mn = fmaxf(m_run, mx);
            if (mn != -INFINITY) {
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int c = 0; c < 64; c += 2) {
                s0 += fast_exp2(x[c] - mn);
                s1 += fast_exp2(x[c + 1] - mn);
              }
              l_run = l_run * fast_exp2(m_run - mn) + (s0 + s1);
              m_run = mn;
            }
          } else {
            float* cs = colsum + (tile_ctr & 1) * 4 * 128 + wg * 128 + chalf * 64;
            const bool interior = jc + 63 < n - a.W;  // every column a candidate
#pragma unroll
            for (int chk = 0; chk < 2; ++chk) {
              float e[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const float v = fast_exp2(__uint_as_float(raw[chk][c]) * a.scale_log2 - lse2);
                e[c] = (interior || jc + chk * 32 + c < n - a.W) ? v : 0.f;
              }
              // Warp transpose-reduce: afterwards lane l holds column (32 chk + l) summed over the warp's rows.
#pragma unroll
              for (int k = 0; k < 5; ++k) {
                const int off = 16 >> k, half = 16 >> k;
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                  const float lo_v = e[i], hi_v = e[i + half];
                  const float send = upper ? lo_v : hi_v;
                  e[i] = (upper ? hi_v : lo_v) + __shfl_xor_sync(0xffffffffu, send, off);
                }
              }
              cs[chk * 32 + lane] = e[0];
            }
            named_barrier_epi();  // the lane quarters' column partials of this tile are in
            const int et = threadIdx.x - 64;  // 0 .. 255
            if (et < kTileN) {
              const float* cb = colsum + (tile_ctr & 1) * 4 * 128;
              const float v = ((cb[et] + cb[128 + et]) + cb[256 + et]) + cb[384 + et];
              const int j = t * kTileN + et;
              if (j < n - a.W) a.scores[(size_t)p * a.score_stride + j] = v;
            }
          }
        }
        if (PASS == 1) {
          // Merge the two column halves of each row, then write this slice's partial.
          if (chalf == 1) {
            stat[r * 2] = m_run;
            stat[r * 2 + 1] = l_run;
          }
          named_barrier_epi();
          if (chalf == 0) {
            const float m1 = stat[r * 2], l1 = stat[r * 2 + 1];
            const float M = fmaxf(m_run, m1);
            float L = 0.f;
            if (M != -INFINITY) L = l_run * fast_exp2(m_run - M) + l1 * fast_exp2(m1 - M);
            const int first_cta = prefix[p] / per_cta;
            const int slot = blockIdx.x - first_cta;
            float* dst = a.part + (((size_t)p * a.max_slices + slot) * 128 + r) * 2;
            dst[0] = M;
            dst[1] = L;
          }
          named_barrier_epi();  // stat is reused by the next segment
        }
        ++seg;
      }
    }
  }
  // Pairs whose prompt holds no candidate (n == window) have no pass-2 tile:
  // CTA 0 writes their row log-sum-exps.
  if (PASS == 2 && blockIdx.x == 0 && a.row_lse && warp >= 2 && warp < 6) {
    const int r = (warp & 3) * 32 + lane;
    for (int p = 0; p < pairs; ++p) {
      if (prefix[p + 1] != prefix[p] || r >= R) continue;
      const int n = a.lens[p / a.H];
      if (n < a.W || n > a.max_len) continue;
      const float l2 = merged_lse2(a, p, r);
      a.row_lse[(size_t)p * R + r] = l2 != INFINITY ? l2 * kLn2 : -INFINITY;
    }
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ selection
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBuckets = 1024;
constexpr int kMaxMembers = 1024;
constexpr int kSelPer = 44;                          // candidates per thread
constexpr int kPoolHalfMax = 8;                      // pooling windows up to 17 wide by shuffles
constexpr int kPoolUnroll = 4;                       // chunks of 32 positions a warp loads at once
constexpr int kSelCluster = 4;                       // CTAs per (request, KV head): the pooling is shared
constexpr int kSelMaxCand = kSelThreads * kSelPer;   // 45056

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix, in index order, of flagged candidates. Thread t owns
// candidates t + 1024 e, so index order is (e, warp, lane): per (e, warp)
// counts from ballots, one prefix over them (warp 0). Afterwards the rank of
// owned candidate e is cnt[e * 32 + warp] + popc(ballot(flag) & lanes below).
__device__ __forceinline__ int sel_warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per-candidate flags (bit e of thread t: candidate t + 1024 e) to the exclusive
// count, in candidate order, of the flagged candidates before each warp's group
// of 32: cnt[e * 32 + warp]. Every thread scans up to two of the E x 32 group
// counts, then the block adds the threads' sums with two warp-level scans.
__device__ __forceinline__ void index_order_prefix(uint64_t flags, int E, int* cnt, int* wtot, int warp,
                                                   int lane) {
  for (int e = 0; e < E; ++e) {
    const unsigned ball = __ballot_sync(0xffffffffu, (flags >> e) & 1ull);
    if (lane == 0) cnt[e * 32 + warp] = __popc(ball);
  }
  __syncthreads();
  const int N = E * 32;               // <= 2 * kSelThreads
  const int tid = warp * 32 + lane;
  const int i0 = 2 * tid;
  const int c0 = i0 < N ? cnt[i0] : 0, c1 = i0 + 1 < N ? cnt[i0 + 1] : 0;
  const int v = c0 + c1;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  const int x = wtot[lane];
  const int before = incl - v + sel_warp_sum(lane < warp ? x : 0);
  if (i0 < N) cnt[i0] = before;
  if (i0 + 1 < N) cnt[i0 + 1] = before + c0;
  __syncthreads();
}

// Max-pool of the scores, then the top `keep` candidates by pooled score (ties:
// lower position) in ascending order, then the window positions. A cluster of
// kSelCluster CTAs per (request, KV head) pools the positions into rank 0's
// shared memory, and rank 0 selects: its thread t owns candidates t + 1024 e
// (conflict-free shared-memory accesses); per-candidate flags sit in a 64-bit
// mask.
__global__ void __launch_bounds__(kSelThreads) snapkv_select_kernel(
    const float* __restrict__ scores, int32_t score_stride, const int32_t* __restrict__ lens, int32_t H, int32_t W,
    int32_t max_len, int32_t pool, int32_t keep, int32_t sink, int32_t recent, int32_t* __restrict__ kept,
    int32_t kept_stride, int32_t* __restrict__ kept_counts, unsigned* err) {
  pdl_enter();
  extern __shared__ float pooled[];  // [n - W]
  __shared__ int hist[kBuckets];
  __shared__ float s_min[kSelWarps], s_max[kSelWarps];
  __shared__ int wtot[kSelWarps];
  __shared__ float mem_val[kMaxMembers];
  __shared__ int mem_idx[kMaxMembers];
  __shared__ int cnt[kSelPer * 32];
  __shared__ int s_info[4];  // bucket B, keys above B, members collected, keys equal to the threshold
  __shared__ int rhist[3][257];
  __shared__ float cl_mm[2 * kSelCluster];  // rank 0: every rank's min and max of its pooled candidates
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int pair = blockIdx.x / kSelCluster, b = pair / H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
  const int n = lens[b];
  if (n < W || n > max_len) {  // the same decision in every rank of the cluster
    if (tid == 0 && rank == 0) {
      raise_error(err, SE_DEVERR_LENGTH);
      kept_counts[pair] = 0;
    }
    return;
  }
  // Scored positions [0, n - W); candidates [c0, c1): neither among the first
  // `sink` positions nor among the last `recent` (>= W) ones.
  const int CS = n - W;
  const int c1 = max(0, n - recent), c0 = min(sink, c1);
  const int C = c1 - c0;  // candidate j is position c0 + j
  int32_t* out = kept + (size_t)pair * kept_stride;
  if (C <= keep) {
    if (rank == 0) {
      for (int i = tid; i < n; i += kSelThreads) out[i] = i;
      if (tid == 0) kept_counts[pair] = n;
    }
    return;
  }
  // The ranks of the cluster pool the positions together, into rank 0's shared
  // memory; rank 0 alone then selects. Every rank has started before any writes
  // into rank 0's shared memory.
  cluster.sync();
  float* pooled0 = cluster.map_shared_rank(pooled, 0);
  const float* sc = scores + (size_t)pair * score_stride;
  const int half = pool / 2;
  float lmin = INFINITY, lmax = -INFINITY;  // over the finite pooled scores of the candidates
  // Max-pool over the scored positions (window clipped to them), and the min and
  // max of the candidates' pooled scores on the way. A warp takes 32
  // consecutive positions; a lane reads its own score, the `half` lanes at each
  // end also the score `half` places beyond the warp's range, and the window
  // comes from the neighbouring lanes by shuffles.
  if (half <= kPoolHalfMax) {
    // kPoolUnroll chunks of a warp are loaded before the first is pooled, so that
    // their memory latency overlaps.
    constexpr int kStride = kSelCluster * kSelThreads;  // positions the cluster's warps cover per round
    for (int base0 = (rank * kSelWarps + warp) * 32; base0 < CS; base0 += kPoolUnroll * kStride) {  // warp-uniform
      float own[kPoolUnroll], lo[kPoolUnroll], hi[kPoolUnroll];
#pragma unroll
      for (int u = 0; u < kPoolUnroll; ++u) {
        const int base = base0 + u * kStride, p = base + lane;
        const int pl = base - half + lane, ph = base + lane + half;
        own[u] = p < CS ? sc[p] : -INFINITY;
        lo[u] = (lane < half && pl >= 0 && pl < CS) ? sc[pl] : -INFINITY;     // position base - half + lane
        hi[u] = (lane >= 32 - half && ph < CS) ? sc[ph] : -INFINITY;          // position base + lane + half
      }
#pragma unroll
      for (int u = 0; u < kPoolUnroll; ++u) {
        const int base = base0 + u * kStride, p = base + lane;
        if (base < CS) {  // warp-uniform
          float m = own[u];
#pragma unroll
          for (int d = 1; d <= kPoolHalfMax; ++d) {
            if (d <= half) {
              const int dn = lane - d, up = lane + d;  // lanes holding p - d and p + d
              const float a = __shfl_sync(0xffffffffu, own[u], dn & 31);
              const float al = __shfl_sync(0xffffffffu, lo[u], (dn + half) & 31);
              const float bu = __shfl_sync(0xffffffffu, own[u], up & 31);
              const float bh = __shfl_sync(0xffffffffu, hi[u], (up - half) & 31);
              m = fmaxf(m, dn >= 0 ? a : al);
              m = fmaxf(m, up < 32 ? bu : bh);
            }
          }
          if (p < CS) pooled0[p] = m;
          if (p >= c0 && p < c1 && isfinite(m)) {
            lmin = fminf(lmin, m);
            lmax = fmaxf(lmax, m);
          }
        }
      }
    }
  } else {
    for (int i = rank * kSelThreads + tid; i < CS; i += kSelCluster * kSelThreads) {
      float m = -INFINITY;
      for (int t = max(0, i - half); t <= min(CS - 1, i + half); ++t) m = fmaxf(m, sc[t]);
      pooled0[i] = m;
      if (i >= c0 && i < c1 && isfinite(m)) {
        lmin = fminf(lmin, m);
        lmax = fmaxf(lmax, m);
      }
    }
  }
  __syncthreads();
  const float* pc = pooled + c0;  // pooled score of candidate j
  const int E = (C + kSelThreads - 1) / kSelThreads;
  hist[tid] = 0;
  if (tid < 2 * 257) (&rhist[0][0])[tid] = 0;
  if (tid == 0) s_info[2] = s_info[3] = 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lmin = fminf(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
    lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  }
  if (lane == 0) {
    s_min[warp] = lmin;
    s_max[warp] = lmax;
  }
  __syncthreads();
  float mn = s_min[lane], mx = s_max[lane];  // min and max over the warps, by shuffles
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (tid == 0) {
    float* mm0 = cluster.map_shared_rank(cl_mm, 0);
    mm0[2 * rank] = mn;
    mm0[2 * rank + 1] = mx;
  }
  cluster.sync();  // rank 0 holds every pooled score and every rank's min and max
  if (rank != 0) return;
#pragma unroll
  for (int r = 0; r < kSelCluster; ++r) {
    mn = fminf(mn, cl_mm[2 * r]);
    mx = fmaxf(mx, cl_mm[2 * r + 1]);
  }
  const float scale = (mx > mn) ? (float)kBuckets / (mx - mn) : 0.f;
  auto bucket = [&](float v) {
    if (isfinite(v)) return min(kBuckets - 1, max(0, (int)((v - mn) * scale)));
    return v > 0.f ? kBuckets - 1 : 0;
  };
  for (int e = 0; e < E; ++e) {
    const int i = tid + e * kSelThreads;
    if (i < C) atomicAdd(&hist[bucket(pc[i])], 1);
  }
  __syncthreads();
  const int hc = hist[tid];
  int incl = hc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += t;
  }
  if (lane == 0) wtot[warp] = incl;
  __syncthreads();
  {
    const int x = wtot[lane];
    incl += sel_warp_sum(lane > warp ? x : 0);  // candidates in the buckets of the warps above
  }
  if (incl - hc < keep && keep <= incl) {
    s_info[0] = tid;
    s_info[1] = incl - hc;
  }
  __syncthreads();
  const int B = s_info[0];
  const int need = keep - s_info[1];
  const int m = hist[B];
  __syncthreads();  // s_info is rewritten below
  uint32_t T;
  int need_eq;
  if (m <= kMaxMembers) {
    for (int e = 0; e < E; ++e) {
      const int i = tid + e * kSelThreads;
      if (i < C && bucket(pc[i]) == B) {
        const int slot = atomicAdd(&s_info[2], 1);
        mem_val[slot] = pc[i];
        mem_idx[slot] = i;
      }
    }
    __syncthreads();
    // The member of rank need - 1 (score desc, position asc) fixes the threshold.
    if (tid < m) {
      const uint32_t kv = order_key(mem_val[tid]);
      const int id = mem_idx[tid];
      int rank = 0, above = 0;
      for (int j = 0; j < m; ++j) {
        const uint32_t kj = order_key(mem_val[j]);
        rank += (kj > kv || (kj == kv && mem_idx[j] < id)) ? 1 : 0;
        above += kj > kv ? 1 : 0;
      }
      if (rank == need - 1) {
        s_info[0] = (int)kv;
        s_info[1] = need - above;
      }
    }
    __syncthreads();
    T = (uint32_t)s_info[0];
    need_eq = s_info[1];
  } else {
    uint32_t prefix = 0, mask = 0;
    int remaining = need;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int* hh = rhist[pass % 3];
      if (pass >= 1)
        for (int i = tid; i < 257; i += kSelThreads) rhist[(pass + 1) % 3][i] = 0;
      for (int e = 0; e < E; ++e) {
        const int i = tid + e * kSelThreads;
        if (i < C) {
          const float v = pc[i];
          const uint32_t key = order_key(v);
          if (bucket(v) == B && (key & mask) == prefix) atomicAdd(&hh[(key >> shift) & 255u], 1);
        }
      }
      __syncthreads();
      int g8[8], gsum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        g8[j] = hh[lane * 8 + j];
        gsum += g8[j];
      }
      int inc2 = gsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, inc2, o);
        if (lane + o < 32) inc2 += t;
      }
      const int up = inc2 - gsum;
      const bool mine = up < remaining && remaining <= inc2;
      int d = 0, ab = 0;
      if (mine) {
        int cum = up;
        for (int j = 7; j >= 0; --j) {
          if (cum + g8[j] >= remaining) {
            d = lane * 8 + j;
            ab = cum;
            break;
          }
          cum += g8[j];
        }
      }
      const unsigned who = __ballot_sync(0xffffffffu, mine);
      const int src = who ? __ffs(who) - 1 : 0;
      d = __shfl_sync(0xffffffffu, d, src);
      ab = __shfl_sync(0xffffffffu, ab, src);
      remaining -= ab;
      prefix |= (uint32_t)d << shift;
      mask |= 255u << shift;
    }
    T = prefix;
    need_eq = remaining;
  }
  // Selected: pooled key above T, or equal to T among the first need_eq by position.
  uint64_t self = 0, eqf = 0;
  int n_eq = 0;
  for (int e = 0; e < E; ++e) {
    const int i = tid + e * kSelThreads;
    if (i < C) {
      const uint32_t key = order_key(pc[i]);
      if (key > T) {
        self |= 1ull << e;
      } else if (key == T) {
        eqf |= 1ull << e;
        ++n_eq;
      }
    }
  }
  if (n_eq) atomicAdd(&s_info[3], n_eq);
  __syncthreads();
  if (s_info[3] <= need_eq) {  // block-uniform: every key equal to T is taken (the usual case)
    self |= eqf;
  } else {                     // more ties than places: the first need_eq by position
    index_order_prefix(eqf, E, cnt, wtot, warp, lane);
    for (int e = 0; e < E; ++e) {
      const unsigned ball = __ballot_sync(0xffffffffu, (eqf >> e) & 1ull);
      const int eq_rank = cnt[e * 32 + warp] + __popc(ball & lt);
      if (((eqf >> e) & 1ull) && eq_rank < need_eq) self |= 1ull << e;
    }
    __syncthreads();  // cnt is reused
  }
  index_order_prefix(self, E, cnt, wtot, warp, lane);
  for (int e = 0; e < E; ++e) {
    const unsigned ball = __ballot_sync(0xffffffffu, (self >> e) & 1ull);
    if ((self >> e) & 1ull) {
      const int pos = cnt[e * 32 + warp] + __popc(ball & lt);
      if (pos < keep) out[c0 + pos] = c0 + tid + e * kSelThreads;
    }
  }
  for (int i = tid; i < c0; i += kSelThreads) out[i] = i;
  for (int w = tid; w < n - c1; w += kSelThreads) out[c0 + keep + w] = c1 + w;
  if (tid == 0) kept_counts[pair] = c0 + keep + (n - c1);
}

// ------------------------------------------------------------------ compaction
// Kept token t of pair (b, h) goes to destination page dst_bt[b][t / 16], slot t % 16.
// A half-warp copies the K and V rows (256 bytes each, 16 x 16 bytes) of
// kGatherTok consecutive kept tokens of one pair: their positions and page ids
// are looked up together and their 2 kGatherTok row loads are in flight at once.
constexpr int kGatherTok = 4;
__global__ void __launch_bounds__(256) snapkv_gather_kernel(KvView src, uint16_t* __restrict__ dk,
                                                            uint16_t* __restrict__ dv, int32_t dst_num_pages,
                                                            const int32_t* __restrict__ src_bt, int32_t src_bt_stride,
                                                            const int32_t* __restrict__ dst_bt, int32_t dst_bt_stride,
                                                            const int32_t* __restrict__ lens, int32_t pairs,
                                                            const int32_t* __restrict__ kept, int32_t kept_stride,
                                                            const int32_t* __restrict__ kept_counts, unsigned* err) {
  pdl_enter();
  const long long unit = (long long)blockIdx.x * 16 + (threadIdx.x >> 4);  // (pair, group of kGatherTok tokens)
  const int sub = threadIdx.x & 15;
  const int groups = (kept_stride + kGatherTok - 1) / kGatherTok;
  if (unit >= (long long)pairs * groups) return;
  const int pair = (int)(unit / groups), t0 = (int)(unit % groups) * kGatherTok;
  const int H = src.num_kv_heads;
  const int b = pair / H, h = pair % H;
  const int cnt = kept_counts[pair];
  if (cnt > kept_stride) return;
  const int n = lens[b];
  // (page, head, slot) row of each token in the source and the destination cache; -1: not copied
  long long srow[kGatherTok], drow[kGatherTok];
#pragma unroll
  for (int u = 0; u < kGatherTok; ++u) {
    srow[u] = drow[u] = -1;
    const int t = t0 + u;
    if (t >= cnt) continue;
    const int pos = kept[(size_t)pair * kept_stride + t];
    if (pos < 0 || pos >= n || pos / kPageSize >= src_bt_stride || t / kPageSize >= dst_bt_stride) {
      if (sub == 0) raise_error(err, SE_DEVERR_LENGTH);
      continue;
    }
    const int sp = src_bt[(size_t)b * src_bt_stride + pos / kPageSize];
    const int dp = dst_bt[(size_t)b * dst_bt_stride + t / kPageSize];
    if (sp < 0 || sp >= src.num_pages || dp < 0 || dp >= dst_num_pages) {
      if (sub == 0) raise_error(err, SE_DEVERR_PAGE_RANGE);
      continue;
    }
    srow[u] = ((long long)sp * H + h) * kPageSize + pos % kPageSize;
    drow[u] = ((long long)dp * H + h) * kPageSize + t % kPageSize;
  }
  uint4 kr[kGatherTok], vr[kGatherTok];
#pragma unroll
  for (int u = 0; u < kGatherTok; ++u) {
    if (srow[u] < 0) continue;
    kr[u] = reinterpret_cast<const uint4*>(src.k + (size_t)srow[u] * src.row_stride_k)[sub];
    vr[u] = reinterpret_cast<const uint4*>(src.v + (size_t)srow[u] * src.row_stride_v)[sub];
  }
#pragma unroll
  for (int u = 0; u < kGatherTok; ++u) {
    if (drow[u] < 0) continue;
    reinterpret_cast<uint4*>(dk + (size_t)drow[u] * kD)[sub] = kr[u];
    reinterpret_cast<uint4*>(dv + (size_t)drow[u] * kD)[sub] = vr[u];
  }
}

size_t scores_smem_bytes(int pairs) {
  return 1024 + (size_t)kPrefixOff + (size_t)((pairs + 2) & ~1) * 4 + 16 * 8 + 16;
}

}  // namespace

int snapkv_max_slices(int max_len) {
  const int tiles = (max_len + kTileN - 1) / kTileN;
  return (tiles + kMinTilesPerCta - 1) / kMinTilesPerCta + 1;
}

size_t snapkv_part_bytes(int pairs, int max_len) {
  const size_t part = (size_t)pairs * snapkv_max_slices(max_len) * 128 * 2 * sizeof(float);
  return ((part + 15) & ~size_t(15)) + (((size_t)pairs * sizeof(int32_t) + 15) & ~size_t(15));
}

int snapkv_select_max_candidates() { return kSelMaxCand; }

cudaError_t launch_snapkv_scores(const CUtensorMap& kmap, const KvView& kv, const uint16_t* qwin, int32_t num_q_heads,
                                 int32_t window, const int32_t* bt, int32_t bt_stride, const int32_t* lens,
                                 int32_t batch, int32_t max_len, float sm_scale, float* scores, int32_t score_stride,
                                 float* row_lse, void* part_ws, int sm_count, unsigned* err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  SnapArgs a;
  a.qwin = qwin;
  a.W = window;
  a.H = kv.num_kv_heads;
  a.G = num_q_heads / kv.num_kv_heads;
  a.B = batch;
  a.bt = bt;
  a.bt_stride = bt_stride;
  a.lens = lens;
  a.max_len = max_len;
  a.num_pages = kv.num_pages;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  const int pairs = batch * kv.num_kv_heads;
  a.max_slices = snapkv_max_slices(max_len);
  const size_t part = (size_t)pairs * a.max_slices * 128 * 2 * sizeof(float);
  a.part = static_cast<float*>(part_ws);
  a.pair_ns = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(part_ws) + ((part + 15) & ~size_t(15)));
  a.row_lse = row_lse;
  a.scores = scores;
  a.score_stride = score_stride;
  a.err = err;
  const size_t smem = scores_smem_bytes(pairs);
  cudaError_t e = cudaFuncSetAttribute(snapkv_scores_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(snapkv_scores_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  {
    const cudaError_t le = launch_pdl(snapkv_scores_kernel<1>, dim3(sm_count), dim3(kThreads), smem, stream, kmap, a);
    if (le != cudaSuccess) return le;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    const cudaError_t le = launch_pdl(snapkv_scores_kernel<2>, dim3(sm_count), dim3(kThreads), smem, stream, kmap, a);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_snapkv_select(const float* scores, int32_t score_stride, const int32_t* lens, int32_t batch,
                                 int32_t num_kv_heads, int32_t window, int32_t max_len, int32_t pool, int32_t keep,
                                 int32_t sink, int32_t recent, int32_t* kept, int32_t kept_stride,
                                 int32_t* kept_counts, unsigned* err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const int maxc = max(max_len - window, 1);
  const size_t smem = (size_t)maxc * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(snapkv_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // A cluster of kSelCluster CTAs per (request, KV head), launched with
  // programmatic dependent launch like every other kernel of the library.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch * num_kv_heads * kSelCluster);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSelCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, snapkv_select_kernel, scores, score_stride, lens, num_kv_heads, window, max_len, pool,
                         keep, sink, recent, kept, kept_stride, kept_counts, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_snapkv_gather(const KvView& src, uint16_t* dk, uint16_t* dv, int32_t dst_num_pages,
                                 const int32_t* src_bt, int32_t src_bt_stride, const int32_t* dst_bt,
                                 int32_t dst_bt_stride, const int32_t* lens, int32_t batch, const int32_t* kept,
                                 int32_t kept_stride, const int32_t* kept_counts, unsigned* err, cudaStream_t stream) {
  const int pairs = batch * src.num_kv_heads;
  const long long units = (long long)pairs * ((kept_stride + kGatherTok - 1) / kGatherTok);
  if (units == 0) return cudaSuccess;
  {
    const cudaError_t le = launch_pdl(snapkv_gather_kernel, dim3((unsigned)((units + 15) / 16)), dim3(256), 0, stream,
                                      src, dk, dv, dst_num_pages, src_bt, src_bt_stride, dst_bt, dst_bt_stride, lens,
                                      pairs, kept, kept_stride, kept_counts, err);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace se
