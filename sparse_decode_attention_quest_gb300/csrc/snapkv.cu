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
// The logits are the one dense contraction of the path: 128 query rows x 256
// keys x 128 dims per tile, on the 5th-generation tensor cores. Warp roles:
//   warp 0      TMA producer: per segment the pair's window queries (two 4-D
//               boxes), then the 16 pages of each 256-key tile, one 3-D box
//               per page (both 64-dim halves, 4 KB, 128-byte swizzle) into a
//               2-stage ring. Streaming random 4 KB pages, 4 KB boxes reach
//               about a fifth more HBM bandwidth than two 2 KB boxes per page,
//               hence one box per page and the page-major tile;
//   warp 1      allocates all 512 TMEM columns (two tiles x two fp32 128x128
//               accumulators) and issues the tcgen05.mma (M 128, N 128, K 16):
//               rows 0-7 of the tile's 16 pages (8-row groups 4 KB apart) into
//               accumulator 0, rows 8-15 into accumulator 1, 8 K steps each;
//   warps 2-9   epilogue, two warps per TMEM lane quarter, each thread with 64
//               of each accumulator's 128 columns.
// Pass 1 computes S = Q K^T: TMEM lane = query row, so a thread keeps its
// row's running max and sum (causal mask on the last tiles only). Pass 2
// computes S^T = K Q^T: TMEM lane = key, so a thread sums exp(z - LSE) over
// its 64 query rows and the two halves meet in shared memory; no shuffles.
// Element-wise work runs on paired fp32 instructions (f32x2 fma / add).
//
// The (request, KV head) pairs are cut into chunks (at most 2,048 pairs, and
// about SE_SNAPKV_CHUNK_BYTES of keys), and the passes run chunk by chunk:
// pass 1 of chunk c, pass 2 of chunk c, pass 1 of chunk c + 1, ..., one launch
// each. A pass-1 launch after the first does not wait for the pass-2 launch
// before it (it touches nothing that launch reads or writes), so the two
// overlap; it waits for it before it exits. A pass-2 launch starts its copies
// and products as soon as its CTAs are resident, and only its epilogue waits
// for the pass-1 launch, before reading the rows' -LSE (each CTA of it waited
// about 10 us for its first accumulator when the whole launch waited at its
// start). Smaller chunks would let pass 2
// read keys that pass 1 of the chunk has just brought into L2, but on GB300 the
// fill and drain of the extra launches cost more than the re-read from HBM
// (4 x 32K prompts: 0.255 ms per eviction with 32 MiB chunks, 0.195 with 64,
// 0.182 with 96, 0.152 with one chunk), so the default keeps one chunk up to
// 256 MiB of keys. In a launch the chunk's tiles form one flattened range that
// every CTA shares equally; pass 2 walks its share backwards, so that its first
// tiles are the ones pass 1 read last, still in L2. Every pass-1 share writes its rows' (max, sum) and
// counts itself in on the pair's counter (zeroed before the first launch); the
// share that completes the count merges them into the rows' final
// log-sum-exps, which pass 2 reads.

#include <cooperative_groups.h>

#include <algorithm>

#include "se_ptx.cuh"

#ifndef SE_SNAPKV_CHUNK_BYTES
#define SE_SNAPKV_CHUNK_BYTES (256u << 20)  // keys of one chunk of pairs
#endif

namespace se {
namespace {

constexpr int kD = 128;
constexpr int kTileN = 256;                   // keys per tile: 16 pages
constexpr int kPagesPerTile = kTileN / kPageSize;
constexpr int kPageHalfBytes = kPageSize * 128;  // 16 rows x 128 bytes (64 dims)
constexpr int kPageBytes = 2 * kPageHalfBytes;   // one page of one head: 4 KB
constexpr int kTileBytes = kPagesPerTile * kPageBytes;  // 64 KB
constexpr int kQHalfBytes = 128 * 128;        // 128 query rows x 128 bytes (64 dims)
constexpr int kQBytes = 2 * kQHalfBytes;      // 32 KB
constexpr int kStages = 2;
constexpr int kThreads = 320;                 // producer, MMA issuer, 8 epilogue warps
constexpr int kEpiThreads = 256;
constexpr int kMinTilesPerCta = 4;
constexpr int kTmemCols = 512;                // two tiles x two 128 x 128 fp32 accumulators
constexpr int kMaxPairsPerChunk = 2048;
constexpr float kLn2 = 0.6931471805599453f;

// Dynamic shared memory: [K ring 2 x 64 KB][Q 2 x 32 KB][column partials 2 x 2 x 128 fp32]
// [final -LSE 2 x 128 fp32][row stats 2 x 128 x 2 fp32][flag][prefix][barriers]
constexpr int kRingOff = 0;
constexpr int kQOff = kStages * kTileBytes;
constexpr int kColOff = kQOff + 2 * kQBytes;
constexpr int kNegLseOff = kColOff + 2 * 2 * 128 * 4;
constexpr int kStatOff = kNegLseOff + 2 * 128 * 4;
constexpr int kFlagOff = kStatOff + 2 * 128 * 2 * 4;
constexpr int kPrefixOff = kFlagOff + 16;

struct SnapArgs {
  int32_t W, G, H;
  int32_t pair0;         // first pair (b * H + h) of this launch
  int32_t pairs;         // pairs of this launch
  int32_t wait_previous; // wait for the previous launch of the stream before the first access
  int32_t late_wait;     // pass 2: only the epilogue waits (for the -LSE), every thread before it exits
  const int32_t* bt;
  int32_t bt_stride;
  const int32_t* lens;
  int32_t max_len;
  int32_t num_pages;
  float scale_log2;
  float* part;           // pass 1: [pairs][max_slices][128] x (max, sum), log2 domain
  uint32_t* done;        // pass-1 shares counted in per pair (zero before the first launch)
  float* final_nlse;     // [pairs][128]: -LSE_r (log2 domain) of every row, merged by the pair's last share
  int32_t max_slices;
  uint64_t probe_limit_ns;  // 0; in a wait probe, the limit of the MMA issuer's wait on a barrier nothing arrives at
  float* row_lse;        // optional: [pairs][R] natural log
  float* scores;         // [pairs][score_stride]
  int32_t score_stride;
  unsigned* err;
};

// ---------------------------------------------------------------- paired fp32
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Sum of exp2(x_c * s + bias_c) over 64 values (two packed lanes at a time, four
// independent packed accumulators).
__device__ __forceinline__ float sum_exp2_64(const uint32_t (&raw)[2][32], uint64_t s2, const uint64_t (&bias)[32]) {
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x0, x1;
    f2_split(ffma2(f2(__uint_as_float(raw[c >> 4][(2 * c) & 31]), __uint_as_float(raw[c >> 4][(2 * c + 1) & 31])),
                   s2, bias[c]),
             x0, x1);
    acc[c & 3] = fadd2(acc[c & 3], f2(fast_exp2(x0), fast_exp2(x1)));
  }
  float a0, a1;
  f2_split(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), a0, a1);
  return a0 + a1;
}

// ---------------------------------------------------------------- schedule
__device__ __forceinline__ int find_pair(const int* prefix, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// A flattened range of T tiles is shared by min(grid, T / kMinTilesPerCta) CTAs
// (at least one), share i holding tiles [floor(i T / n), floor((i + 1) T / n)):
// every share has at least kMinTilesPerCta tiles when T does.
__device__ __forceinline__ int share_count(int T, int grid) { return max(1, min(grid, T / kMinTilesPerCta)); }
__device__ __forceinline__ int share_start(int T, int n, int i) { return (int)(((long long)i * T) / n); }
__device__ __forceinline__ int share_of_tile(int T, int n, int u) {
  return (int)(((long long)(u + 1) * n + T - 1) / T) - 1;
}

__device__ __forceinline__ void named_barrier_epi() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Tiles of a pair with n keys for the pass: all keys (pass 1) or the candidates only (pass 2).
__device__ __forceinline__ int pair_tiles(int n, int W, int pass) {
  const int cols = pass == 1 ? n : max(n - W, 0);
  return (cols + kTileN - 1) / kTileN;
}

// One pass over the tiles of one chunk of pairs (see the file comment).
template <int PASS>
__global__ void __launch_bounds__(kThreads, 1) snapkv_pass_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                 const __grid_constant__ CUtensorMap qmap,
                                                                 const SnapArgs a) {
  if (a.wait_previous && !a.late_wait) pdl_wait();
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int pairs = a.pairs;
  int* prefix = reinterpret_cast<int*>(smem + kPrefixOff);  // [pairs + 1]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPrefixOff + ((pairs + 2) & ~1) * 4);
  uint64_t* full = bars;                 // [4]
  uint64_t* empty = full + kStages;      // [4]
  uint64_t* acc_full = empty + kStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;    // [2]
  uint64_t* q_full = acc_empty + 2;      // [2]
  uint64_t* q_empty = q_full + 2;        // [2]
  uint64_t* mma_fin = q_empty + 2;       // every MMA of the CTA has completed
  uint64_t* probe = mma_fin + 1;         // wait probe: a barrier nothing arrives at
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(probe + 1);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + kFlagOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = a.W * a.G;

  // Tiles per pair and their exclusive prefix; zero query buffers (the copies
  // write rows 0 .. R - 1 only).
  for (int p = threadIdx.x; p < pairs; p += kThreads) {
    int n = a.lens[(a.pair0 + p) / a.H];
    if (n < a.W || n > a.max_len) {
      if (PASS == 1) raise_error(a.err, SE_DEVERR_LENGTH);
      n = n < a.W ? 0 : a.max_len;
    }
    prefix[p + 1] = pair_tiles(n, a.W, PASS);
  }
  for (int i = threadIdx.x; i < 2 * kQBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kQOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiThreads);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(mma_fin, 1);
    mbar_init(probe, 1);
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
  const int T = prefix[pairs];
  const int nsh = share_count(T, (int)gridDim.x);
  const int lo = (int)blockIdx.x < nsh ? share_start(T, nsh, blockIdx.x) : T;
  const int hi = (int)blockIdx.x < nsh ? share_start(T, nsh, blockIdx.x + 1) : T;
  // Calls fn(p, t0, t1) for every segment (one pair's tiles [t0, t1)) of this CTA's share.
  // Pass 2 walks its share backwards (segments and tiles): its first tiles are the
  // ones pass 1 read last, still in L2. Loops run over t in [t0, t1) either way;
  // iteration t of pass 2 reads tile t0 + t1 - 1 - t.
  constexpr bool kBackwards = PASS == 2;
  auto for_each_segment = [&](auto&& fn) {
    if (lo >= hi) return;
    const int pf = find_pair(prefix, pairs, lo), pl = find_pair(prefix, pairs, hi - 1);
    for (int i = 0; i <= pl - pf; ++i) {
      const int p = kBackwards ? pl - i : pf + i;
      const int t0 = max(lo, prefix[p]) - prefix[p], t1 = min(hi, prefix[p + 1]) - prefix[p];
      if (t0 < t1) fn(p, t0, t1);
    }
  };
  bool dead = false;  // a bounded wait gave up: finish without further waits

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per segment: the pair's window queries (two 4-D boxes: 64 dims x G heads
    // x W positions, rows r = w G + g), then its key tiles.
    const uint64_t q_policy = l2_evict_normal_policy();
    // pass 1: the keys are read again by pass 2 (its first tiles from L2); pass 2: last use
    const uint64_t policy = PASS == 1 ? l2_evict_normal_policy() : l2_evict_first_policy();
    int it = 0, seg = 0;
    for_each_segment([&](int p, int t0, int t1) {
      const int g = a.pair0 + p;
      const int b = g / a.H, h = g % a.H;
      const int n = min(a.lens[b], a.max_len);
      const int npages = (n + kPageSize - 1) / kPageSize;
      const int qb = seg & 1;
      if (lane == 0) {
        if (seg >= 2 && !dead && !mbar_wait(&q_empty[qb], ((seg >> 1) - 1) & 1)) {
          raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
          dead = true;
        }
        mbar_arrive_expect_tx(&q_full[qb], dead ? 0u : (uint32_t)(2 * R * 128));
        if (!dead) {
          uint8_t* qt = smem + kQOff + qb * kQBytes;
          tma_load_4d(qt, &qmap, 0, h * a.G, 0, b, &q_full[qb], q_policy);
          tma_load_4d(qt + kQHalfBytes, &qmap, 64, h * a.G, 0, b, &q_full[qb], q_policy);
        }
      }
      dead = __shfl_sync(0xffffffffu, (int)dead, 0) != 0;
      ++seg;
      // Block-table entries of 2 tiles per window (lane l: page l % 16 of tile
      // wb + l / 16); the next window is read 2 tiles before it is needed.
      const int32_t* bt_row = a.bt + (size_t)b * a.bt_stride;
      auto load_window = [&](int wt) {
        const int tt = wt + (lane >> 4);
        const int page = (kBackwards ? t0 + t1 - 1 - tt : tt) * kPagesPerTile + (lane & 15);
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
      int wb = t0, win_cur = load_window(t0), win_nxt = load_window(t0 + 2);
      for (int t = t0; t < t1; ++t, ++it) {
        const int s = it % kStages;
        if (t == wb + 2) {
          wb += 2;
          win_cur = win_nxt;
          win_nxt = load_window(wb + 2);
        }
        // Lane l < 16 copies page l of the tile: [64-dim half][16 rows][128 bytes].
        int phys = __shfl_sync(0xffffffffu, win_cur, (t - wb) * kPagesPerTile + (lane & 15));
        if (lane >= kPagesPerTile) phys = -1;
        if (it >= kStages && !dead && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1)) {
          if (lane == 0) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
          dead = true;
        }
        const unsigned live = __ballot_sync(0xffffffffu, phys >= 0 && !dead);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], __popc(live) * kPageBytes);
        __syncwarp();
        if (phys >= 0 && !dead)
          tma_load_3d(smem + kRingOff + s * kTileBytes + lane * kPageBytes, &kmap, 0, (phys * a.H + h) * kPageSize, 0,
                      &full[s], policy);
      }
    });
    // Drain: every copy this CTA issued has landed before it exits.
    if (lane == 0) {
      for (int i = max(0, it - kStages); i < it; ++i)
        if (!mbar_wait(&full[i % kStages], (i / kStages) & 1)) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
      for (int i = max(0, seg - 2); i < seg; ++i)
        if (!mbar_wait(&q_full[i & 1], (i >> 1) & 1)) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 alone: descriptors advanced by constant offsets ((bytes >> 4) in the
    // address field, no carry: every shared address is below 256 KB). Pass 1
    // multiplies Q (A, M = query rows) by K (B, N = keys); pass 2 swaps them.
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(128, 128);
      int it = 0, seg = 0;
      if (a.probe_limit_ns && !mbar_wait_ns(probe, 0, a.probe_limit_ns)) {
        // the probe's wait ran out, as it must: no MMA from here on
        raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
        dead = true;
      }
      // After a failed wait the loop goes on without MMAs but keeps committing,
      // so that the other roles' waits still complete.
      for_each_segment([&](int p, int t0, int t1) {
        const int qb = seg & 1;
        if (!dead && !mbar_wait(&q_full[qb], (seg >> 1) & 1)) {
          raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
          dead = true;
        }
        tc05_fence_after();
        const uint64_t dq = umma_desc_sw128(smem_addr(smem + kQOff + qb * kQBytes));
        for (int t = t0; t < t1; ++t, ++it) {
          const int s = it % kStages, ab = it & 1;
          if (!dead && (!mbar_wait(&full[s], (it / kStages) & 1) ||
                        (it >= 2 && !mbar_wait(&acc_empty[ab], ((it >> 1) - 1) & 1)))) {
            raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            dead = true;
          }
          tc05_fence_after();
          if (!dead) {
            const uint32_t kt = smem_addr(smem + kRingOff + s * kTileBytes);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const uint64_t dk = umma_desc_sw128_groups(kt + q * 1024, kPageBytes);
              const uint32_t d = tmem + ab * 256 + q * 128;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                // K step kk: 64-dim half kk / 4, 32 bytes (2 in the address field) per step inside it.
                const uint64_t oq = (uint64_t)(kk >> 2) * (kQHalfBytes >> 4) + (uint64_t)(kk & 3) * 2;
                const uint64_t ok = (uint64_t)(kk >> 2) * (kPageHalfBytes >> 4) + (uint64_t)(kk & 3) * 2;
                if (PASS == 1)
                  tc05_mma_bf16(d, dq + oq, dk + ok, idesc, kk > 0 ? 1u : 0u);
                else
                  tc05_mma_bf16(d, dk + ok, dq + oq, idesc, kk > 0 ? 1u : 0u);
              }
            }
          }
          tc05_commit(&empty[s]);
          tc05_commit(&acc_full[ab]);
          if (t == t1 - 1) tc05_commit(&q_empty[qb]);
        }
        ++seg;
      });
      // Every MMA issued has completed before the CTA frees its tensor memory.
      tc05_commit(mma_fin);
      if (!mbar_wait(mma_fin, 0)) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = warp & 3;              // TMEM lane quarter of this warp
    const int chalf = (warp - 2) >> 2;    // which 64 of the tile's 128 columns
    const int lq = wg * 32 + lane;        // this thread's TMEM lane
    const int et = threadIdx.x - 64;      // 0 .. 255
    float* stat = reinterpret_cast<float*>(smem + kStatOff);        // [2][128 rows][2]
    float* colpart = reinterpret_cast<float*>(smem + kColOff);      // [2 tiles][2 halves][128 keys]
    float* neglse = reinterpret_cast<float*>(smem + kNegLseOff);    // [2 segments][128 rows]
    const uint64_t s2 = f2(a.scale_log2, a.scale_log2);
    int it = 0, seg = 0;
    for_each_segment([&](int p, int t0, int t1) {
      const int g = a.pair0 + p;
      const int b = g / a.H;
      const int n = min(a.lens[b], a.max_len);
      if (PASS == 1) {
        // ---------------------------------------------------- pass 1: row max / sum
        const int r = lq, w_pos = r / a.G;
        const bool row_live = r < R;
        const int limit = n - a.W + w_pos;  // last key this row sees
        float m_run = -INFINITY, l_run = 0.f;
        for (int t = t0; t < t1; ++t, ++it) {
          const int ab = it & 1;
          if (!dead && !mbar_wait(&acc_full[ab], (it >> 1) & 1)) {
            raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            dead = true;
          }
          tc05_fence_after();
#pragma unroll 1
          for (int q = 0; q < 2; ++q) {
            uint32_t raw[2][32];
            {
              const uint32_t addr = tmem + ((uint32_t)(wg * 32) << 16) + ab * 256 + q * 128 + chalf * 64;
              tmem_ld32(addr, raw[0]);
              tmem_ld32(addr + 32, raw[1]);
              tmem_ld_wait();
            }
            if (q == 1) {
              tc05_fence_before();
              mbar_arrive(&acc_empty[ab]);  // both accumulators read: the slot can take the next tile
            }
            if (!row_live) continue;
            // Column c of this thread's 64 holds key kb + 16 (c / 8) + c % 8 (page
            // 8 chalf + c / 8 of the tile, row 8 q + c % 8); the last is kb + 119.
            const int kb = t * kTileN + chalf * 128 + q * 8;
            if (kb + 119 <= limit) {
              // Every key visible: max of the raw logits (scale > 0), then the sum.
              float m21[22];
#pragma unroll
              for (int i = 0; i < 21; ++i)
                m21[i] = fmax3(__uint_as_float(raw[(3 * i) >> 5][(3 * i) & 31]),
                               __uint_as_float(raw[(3 * i + 1) >> 5][(3 * i + 1) & 31]),
                               __uint_as_float(raw[(3 * i + 2) >> 5][(3 * i + 2) & 31]));
              m21[21] = __uint_as_float(raw[1][31]);
              float m8[8];
#pragma unroll
              for (int i = 0; i < 7; ++i) m8[i] = fmax3(m21[3 * i], m21[3 * i + 1], m21[3 * i + 2]);
              m8[7] = m21[21];
              const float zmax = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
              const float mn = fmaxf(m_run, zmax * a.scale_log2);
              uint64_t bias[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) bias[c] = f2(-mn, -mn);
              const float sum = sum_exp2_64(raw, s2, bias);
              l_run = l_run * fast_exp2(m_run - mn) + sum;
              m_run = mn;
            } else {
              // Causal boundary: keys past `limit` (and past the prompt) are masked.
              float x[64];
#pragma unroll
              for (int c = 0; c < 64; ++c) {
                const float z = __uint_as_float(raw[c >> 5][c & 31]) * a.scale_log2;
                x[c] = kb + (c >> 3) * 16 + (c & 7) <= limit ? z : -INFINITY;
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
            }
          }
        }
        // Merge the two column halves of each row (double-buffered by segment),
        // write this share's partial and count it in on the pair's counter.
        float* st = stat + (seg & 1) * 256;
        if (chalf == 1) {
          st[lq * 2] = m_run;
          st[lq * 2 + 1] = l_run;
        }
        named_barrier_epi();
        const int Tp = prefix[p + 1] - prefix[p];  // tiles of the pair; its shares:
        const int first = share_of_tile(T, nsh, prefix[p]);
        const int ns = share_of_tile(T, nsh, prefix[p] + Tp - 1) - first + 1;
        if (chalf == 0) {
          const float m1 = st[lq * 2], l1 = st[lq * 2 + 1];
          const float M = fmaxf(m_run, m1);
          float L = 0.f;
          if (M != -INFINITY) L = l_run * fast_exp2(m_run - M) + l1 * fast_exp2(m1 - M);
          const int slot = (int)blockIdx.x - first;
          if (slot >= 0 && slot < a.max_slices) {
            float* dst = a.part + (((size_t)g * a.max_slices + slot) * 128 + lq) * 2;
            *reinterpret_cast<float2*>(dst) = make_float2(M, L);
          }
        }
        named_barrier_epi();
        if (et == 0) {
          __threadfence();
          const uint32_t before = atomicAdd(a.done + g, 1u);
          *flag = (int)before == ns - 1 ? 1 : 0;
        }
        named_barrier_epi();
        if (*flag) {
          // The pair's last share: merge every share's (max, sum) per row (two
          // threads per row over alternate shares, 8 loads in flight each), then
          // write the rows' final -LSE and log-sum-exp.
          __threadfence();
          const int r = et & 127, hs = et >> 7;
          const float* pr = a.part + ((size_t)g * a.max_slices * 128 + r) * 2;
          const int nsc = min(ns, a.max_slices);
          float m = -INFINITY, l = 0.f;
          for (int s0 = hs; s0 < nsc; s0 += 16) {
            float2 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              v[u] = s0 + 2 * u < nsc ? __ldcg(reinterpret_cast<const float2*>(pr + (size_t)(s0 + 2 * u) * 256))
                                      : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float mn = fmaxf(m, v[u].x);
              if (mn != -INFINITY) {
                l = l * fast_exp2(m - mn) + v[u].y * fast_exp2(v[u].x - mn);
                m = mn;
              }
            }
          }
          float* mrg = colpart;  // [2 halves][128 rows][2]
          mrg[(hs * 128 + r) * 2] = m;
          mrg[(hs * 128 + r) * 2 + 1] = l;
          named_barrier_epi();
          if (hs == 0) {
            const float m1 = mrg[(128 + r) * 2], l1 = mrg[(128 + r) * 2 + 1];
            const float M = fmaxf(m, m1);
            float L = 0.f;
            if (M != -INFINITY) L = l * fast_exp2(m - M) + l1 * fast_exp2(m1 - M);
            const float lse2 = L > 0.f ? M + log2f(L) : INFINITY;  // +inf: the row saw no key
            a.final_nlse[(size_t)g * 128 + r] = -lse2;
            if (a.row_lse && r < R) a.row_lse[(size_t)g * R + r] = lse2 != INFINITY ? lse2 * kLn2 : -INFINITY;
          }
          named_barrier_epi();  // the merge scratch is free again
        }
      } else {
        // ---------------------------------------------------- pass 2: column sums
        // The rows' final -LSE of this pair (written by the pass-1 launch: with
        // a late wait, the copies and products of this launch have started
        // before it completed).
        float* nl = neglse + (seg & 1) * 128;
        if (a.late_wait) pdl_wait();
        if (et < 128) nl[et] = __ldcg(a.final_nlse + (size_t)g * 128 + et);
        named_barrier_epi();
        uint64_t bias[32];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float4 v = *reinterpret_cast<const float4*>(nl + chalf * 64 + 2 * c);
          bias[c] = f2(v.x, v.y);
          bias[c + 1] = f2(v.z, v.w);
        }
        const bool half_live = chalf * 64 < R;  // rows past R contribute nothing
        for (int t = t0; t < t1; ++t, ++it) {
          const int ab = it & 1;
          if (!dead && !mbar_wait(&acc_full[ab], (it >> 1) & 1)) {
            raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            dead = true;
          }
          tc05_fence_after();
#pragma unroll 1
          for (int q = 0; q < 2; ++q) {
            uint32_t raw[2][32];
            {
              const uint32_t addr = tmem + ((uint32_t)(wg * 32) << 16) + ab * 256 + q * 128 + chalf * 64;
              tmem_ld32(addr, raw[0]);
              tmem_ld32(addr + 32, raw[1]);
              tmem_ld_wait();
            }
            if (q == 1) {
              tc05_fence_before();
              mbar_arrive(&acc_empty[ab]);
            }
            const float part = (half_live && !dead) ? sum_exp2_64(raw, s2, bias) : 0.f;
            float* cp = colpart + q * 256;
            cp[chalf * 128 + lq] = part;
            named_bar_sync(2 + wg, 64);  // the other half of these 32 keys is in (warps w and w + 4)
            if (chalf == 0) {
              // TMEM lane m holds key 16 (m / 8) + 8 q + m % 8 of the tile.
              const int j = (kBackwards ? t0 + t1 - 1 - t : t) * kTileN + (lq >> 3) * 16 + q * 8 + (lq & 7);
              if (j < n - a.W) a.scores[(size_t)g * a.score_stride + j] = cp[lq] + cp[128 + lq];
            }
          }
        }
      }
      ++seg;
    });
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  // A launch that did not wait at its start completes only after the launch
  // before it, so that a later kernel that waits for this one sees both.
  if (!a.wait_previous || a.late_wait) pdl_wait();
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
constexpr int kSelWords = kSelMaxCand / 32;          // one bit per candidate

// Monotone map of a float to an unsigned key (a < b <=> key(a) < key(b)).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int sel_warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Exclusive prefix over the block's threads (in thread order) of v; `wtot`
// holds kSelWarps ints. Every thread of the block calls it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* wtot, int warp, int lane) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  int x = wtot[lane], xs = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, xs, o);
    if (lane >= o) xs += t;
  }
  const int base = __shfl_sync(0xffffffffu, xs - x, warp);  // totals of the warps before this one
  __syncthreads();                                          // wtot is free again
  return base + incl - v;
}

// Max-pool of the scores, then the top `keep` candidates by pooled score (ties:
// lower position) in ascending order, then the window positions. A cluster of
// kSelCluster CTAs per (request, KV head) pools the positions into rank 0's
// shared memory, and rank 0 alone selects. Its thread t owns candidates
// t + 1024 e, so that a warp's ballot over its e-th candidates is bit word
// e * 32 + warp of the candidate bitmap, which covers candidates 32 w .. 32 w + 31
// (index order = word order).
//   1. pool into rank 0's shared memory, with the range [kmin, kmax] of the
//      candidates' order keys;
//   2. histogram of the keys in 1,024 log-linear buckets (key - kmin) >> shift,
//      shift the smallest that fits the range: a bucket spans a fixed fraction
//      of an octave, so heavy-tailed scores spread over many buckets;
//   3. the bucket B that holds the keep-th largest; one pass sets the bitmap
//      bits of every candidate above B and lists B's members;
//   4. each member's rank (key descending, position ascending) among them
//      decides it: the first keep - (candidates above B) are kept. A bucket with
//      more than kMaxMembers members is settled by an 8-bit radix select of
//      its keys instead (threshold key T, then the first equal keys by
//      position);
//   5. the kept positions leave in index order from a prefix over the bitmap.
__global__ void __launch_bounds__(kSelThreads) snapkv_select_kernel(
    const float* __restrict__ scores, int32_t score_stride, const int32_t* __restrict__ lens, int32_t H, int32_t W,
    int32_t max_len, int32_t pool, int32_t keep, int32_t sink, int32_t recent, int32_t* __restrict__ kept,
    int32_t kept_stride, int32_t* __restrict__ kept_counts, unsigned* err) {
  // The scores are the previous kernel's output: everything before the first
  // score load (lengths, the cluster's start, zeroing its shared memory) runs
  // before that kernel has completed; every thread waits for it before it reads
  // a score or exits.
  extern __shared__ float pooled[];  // [n - W]
  __shared__ int hist[kBuckets];
  __shared__ uint32_t s_kmin[kSelWarps], s_kmax[kSelWarps];
  __shared__ int wtot[kSelWarps];
  __shared__ uint32_t mem_key[kMaxMembers];
  __shared__ int mem_idx[kMaxMembers];
  __shared__ uint32_t selw[kSelWords];  // bit j % 32 of word j / 32: candidate j is kept
  __shared__ uint32_t eqw[kSelWords];   // radix path: candidate j has the threshold key
  __shared__ int s_info[4];             // bucket B, candidates above B, members listed, -
  __shared__ int rhist[3][257];
  __shared__ uint32_t cl_range[2 * kSelCluster];  // rank 0: every rank's key range
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int pair = blockIdx.x / kSelCluster, b = pair / H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = lens[b];
  if (n < W || n > max_len) {  // the same decision in every rank of the cluster
    pdl_wait();
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
    pdl_wait();
    if (rank == 0) {
      for (int i = tid; i < n; i += kSelThreads) out[i] = i;
      if (tid == 0) kept_counts[pair] = n;
    }
    return;
  }
  hist[tid] = 0;  // this rank's histogram; rank 0's is the pair's
  for (int i = tid; i < kSelWords; i += kSelThreads) selw[i] = 0u;
  if (tid < 2 * 257) (&rhist[0][0])[tid] = 0;
  if (tid == 0) s_info[2] = 0;
  // Every rank has started and zeroed its shared memory before any rank writes
  // into another's.
  cluster.sync();
  pdl_enter();
  const float* sc = scores + (size_t)pair * score_stride;
  const int half = pool / 2;
  uint32_t kmin = 0xffffffffu, kmax = 0u;  // over the candidates' pooled order keys
  // Max-pool over the scored positions (window clipped to them). A warp takes 32
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
          if (p < CS) pooled[p] = m;
          if (p >= c0 && p < c1) {
            const uint32_t k = order_key(m);
            kmin = min(kmin, k);
            kmax = max(kmax, k);
          }
        }
      }
    }
  } else {
    for (int i = rank * kSelThreads + tid; i < CS; i += kSelCluster * kSelThreads) {
      float m = -INFINITY;
      for (int t = max(0, i - half); t <= min(CS - 1, i + half); ++t) m = fmaxf(m, sc[t]);
      pooled[i] = m;
      if (i >= c0 && i < c1) {
        const uint32_t k = order_key(m);
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    s_kmin[warp] = kmin;
    s_kmax[warp] = kmax;
  }
  __syncthreads();
  kmin = s_kmin[lane];
  kmax = s_kmax[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (tid < kSelCluster) {  // this rank's key range to every rank
    uint32_t* r = cluster.map_shared_rank(cl_range, tid);
    r[2 * rank] = kmin;
    r[2 * rank + 1] = kmax;
  }
  cluster.sync();  // every rank holds every rank's key range; rank 0's histogram and bitmap are zero
#pragma unroll
  for (int r = 0; r < kSelCluster; ++r) {
    kmin = min(kmin, cl_range[2 * r]);
    kmax = max(kmax, cl_range[2 * r + 1]);
  }
  int shift = 0;  // block-uniform
  while (((kmax - kmin) >> shift) >= (uint32_t)kBuckets) ++shift;
  // This rank's positions come in chunks of 32: chunk k (positions 32 k ..
  // 32 k + 31) belongs to rank (k mod 128) / 32 and its warp k mod 32, in both
  // pooling loops above.
  constexpr int kChunkStep = kSelCluster * kSelWarps;
  for (int k = rank * kSelWarps + warp; 32 * k < CS; k += kChunkStep) {
    const int p = 32 * k + lane;
    if (p >= c0 && p < c1) atomicAdd(&hist[(order_key(pooled[p]) - kmin) >> shift], 1);
  }
  __syncthreads();
  int* hist0 = cluster.map_shared_rank(hist, 0);
  if (rank != 0) {
    const int h = hist[tid];
    if (h) atomicAdd(hist0 + tid, h);
  }
  cluster.sync();  // rank 0's histogram is the pair's
  // The bucket B holding the keep-th largest (every rank finds the same):
  // thread t sums the buckets >= t.
  {
    const int hc = hist0[tid];
    int incl = hc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += t;
    }
    if (lane == 0) wtot[warp] = incl;
    __syncthreads();
    const int x = wtot[lane];
    incl += sel_warp_sum(lane > warp ? x : 0);  // candidates in the buckets of the warps above
    if (incl - hc < keep && keep <= incl) {
      s_info[0] = tid;
      s_info[1] = incl - hc;
    }
    __syncthreads();
  }
  const int B = s_info[0];
  const int need = keep - s_info[1];  // members of B to keep, >= 1
  const int m = hist0[B];
  // Every rank: its candidates above B set their bits of rank 0's bitmap (by
  // position: chunk k is word k, one ballot), and B's members are listed in rank 0.
  {
    uint32_t* selw0 = cluster.map_shared_rank(selw, 0);
    int* info0 = cluster.map_shared_rank(s_info, 0);
    uint32_t* key0 = cluster.map_shared_rank(mem_key, 0);
    int* idx0 = cluster.map_shared_rank(mem_idx, 0);
    for (int k = rank * kSelWarps + warp; 32 * k < CS; k += kChunkStep) {
      const int p = 32 * k + lane;
      const bool cand = p >= c0 && p < c1;
      const uint32_t key = cand ? order_key(pooled[p]) : 0u;
      const int bb = cand ? (int)((key - kmin) >> shift) : -1;
      const unsigned above = __ballot_sync(0xffffffffu, bb > B);
      if (lane == 0 && above) selw0[k] = above;
      if (bb == B && m <= kMaxMembers) {
        const int slot = atomicAdd(info0 + 2, 1);
        key0[slot] = key;
        idx0[slot] = p;
      }
    }
  }
  cluster.sync();  // rank 0 holds the bitmap of the candidates above B and B's members
  if (rank != 0) {
    if (m > kMaxMembers) cluster.sync();  // rank 0's radix select reads this rank's pooled scores
    return;
  }
  if (m <= kMaxMembers) {
    // A member is kept when fewer than `need` members rank before it (key
    // descending, then position).
    for (int s = tid; s < m; s += kSelThreads) {
      const uint32_t k = mem_key[s];
      const int id = mem_idx[s];
      int r = 0;
      for (int j = 0; j < m; ++j) {
        const uint32_t kj = mem_key[j];
        r += (kj > k || (kj == k && mem_idx[j] < id)) ? 1 : 0;
      }
      if (r < need) atomicOr(&selw[id >> 5], 1u << (id & 31));
    }
  } else {
    // Radix select of the need-th largest key in B, 8 bits at a time, over
    // every rank's pooled scores (read across the cluster): the threshold key
    // T and how many of the keys equal to T are kept.
    auto key_at = [&](int p) {
      const int owner = ((p >> 5) & (kChunkStep - 1)) / kSelWarps;
      const float v = owner == 0 ? pooled[p] : cluster.map_shared_rank(pooled, owner)[p];
      return order_key(v);
    };
    uint32_t prefix = 0, mask = 0;
    int remaining = need;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift8 = 24 - 8 * pass;
      int* hh = rhist[pass % 3];
      if (pass >= 1)
        for (int i = tid; i < 257; i += kSelThreads) rhist[(pass + 1) % 3][i] = 0;
      for (int p = c0 + tid; p < c1; p += kSelThreads) {
        const uint32_t key = key_at(p);
        if ((int)((key - kmin) >> shift) == B && (key & mask) == prefix) atomicAdd(&hh[(key >> shift8) & 255u], 1);
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
      prefix |= (uint32_t)d << shift8;
      mask |= 255u << shift8;
    }
    const uint32_t T = prefix;
    const int need_eq = remaining;  // keys equal to T to keep, the first by position
    for (int k = warp; 32 * k < CS; k += kSelWarps) {
      const int p = 32 * k + lane;
      const bool cand = p >= c0 && p < c1;
      const uint32_t key = cand ? key_at(p) : 0u;
      const bool inb = cand && (int)((key - kmin) >> shift) == B;
      const unsigned gt = __ballot_sync(0xffffffffu, inb && key > T);
      const unsigned eq = __ballot_sync(0xffffffffu, inb && key == T);
      if (lane == 0) {
        selw[k] |= gt;
        eqw[k] = eq;
      }
    }
    __syncthreads();
    cluster.sync();  // the other ranks' pooled scores are no longer read
    // Thread t: equal-key words 2t, 2t + 1 (position order).
    const int nw = (CS + 31) / 32;
    const uint32_t e0 = 2 * tid < nw ? eqw[2 * tid] : 0u, e1 = 2 * tid + 1 < nw ? eqw[2 * tid + 1] : 0u;
    int before = block_exclusive_scan(__popc(e0) + __popc(e1), wtot, warp, lane);
    uint32_t take0 = 0, take1 = 0;
    for (uint32_t v = e0; v && before < need_eq; v &= v - 1, ++before) take0 |= v & (~v + 1u);
    for (uint32_t v = e1; v && before < need_eq; v &= v - 1, ++before) take1 |= v & (~v + 1u);
    if (take0) selw[2 * tid] |= take0;
    if (take1) selw[2 * tid + 1] |= take1;
  }
  __syncthreads();
  // Kept candidates in position order: thread t holds bitmap words 2t, 2t + 1.
  {
    const int nw = (CS + 31) / 32;
    const uint32_t w0 = 2 * tid < nw ? selw[2 * tid] : 0u, w1 = 2 * tid + 1 < nw ? selw[2 * tid + 1] : 0u;
    int pos = block_exclusive_scan(__popc(w0) + __popc(w1), wtot, warp, lane);
    for (uint32_t v = w0; v; v &= v - 1) out[c0 + pos++] = 64 * tid + __ffs(v) - 1;
    for (uint32_t v = w1; v; v &= v - 1) out[c0 + pos++] = 64 * tid + 32 + __ffs(v) - 1;
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
  // The lengths and the destination pages of these slots do not depend on the
  // selection (the previous kernel): they are read before it has completed.
  const long long unit = (long long)blockIdx.x * 16 + (threadIdx.x >> 4);  // (pair, group of kGatherTok tokens)
  const int sub = threadIdx.x & 15;
  const int groups = (kept_stride + kGatherTok - 1) / kGatherTok;
  if (unit >= (long long)pairs * groups) {
    pdl_wait();
    return;
  }
  const int pair = (int)(unit / groups), t0 = (int)(unit % groups) * kGatherTok;
  const int H = src.num_kv_heads;
  const int b = pair / H, h = pair % H;
  const int n = lens[b];
  int dpg[kGatherTok];
#pragma unroll
  for (int u = 0; u < kGatherTok; ++u) {
    const int t = t0 + u;
    dpg[u] = (t < kept_stride && t / kPageSize < dst_bt_stride) ? dst_bt[(size_t)b * dst_bt_stride + t / kPageSize] : -1;
  }
  pdl_enter();
  const int cnt = kept_counts[pair];
  if (cnt > kept_stride) return;
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
    const int dp = dpg[u];
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

size_t pass_smem_bytes(int pairs) {
  return 1024 + (size_t)kPrefixOff + (size_t)((pairs + 2) & ~1) * 4 + 18 * 8 + 16;
}

}  // namespace

int snapkv_max_slices(int max_len) {
  const int tiles = (max_len + kTileN - 1) / kTileN;
  return (tiles + kMinTilesPerCta - 1) / kMinTilesPerCta + 1;
}

size_t snapkv_part_bytes(int pairs, int max_len) {
  // per-share (max, sum) of every row, the pair counters, the rows' final -LSE
  const size_t part = (size_t)pairs * snapkv_max_slices(max_len) * 128 * 2 * sizeof(float);
  return ((part + 15) & ~size_t(15)) + (((size_t)pairs * sizeof(int32_t) + 15) & ~size_t(15)) +
         (size_t)pairs * 128 * sizeof(float);
}

int snapkv_select_max_candidates() { return kSelMaxCand; }

namespace {
// One-shot wait probe of this host thread (se_debug_snapkv_wait_probe): 0 = none.
thread_local uint32_t t_wait_probe_us = 0;
}  // namespace

void set_snapkv_wait_probe(uint32_t limit_us) { t_wait_probe_us = limit_us; }

cudaError_t launch_snapkv_scores(const CUtensorMap& kmap, const CUtensorMap& qmap, const KvView& kv, const uint16_t* qwin,
                                 int32_t num_q_heads, int32_t window, const int32_t* bt, int32_t bt_stride,
                                 const int32_t* lens, int32_t batch, int32_t max_len, float sm_scale, float* scores,
                                 int32_t score_stride, float* row_lse, void* part_ws, int sm_count, unsigned* err,
                                 cudaStream_t stream) {
  (void)qwin;
  if (batch == 0) return cudaSuccess;
  SnapArgs a;
  a.W = window;
  a.H = kv.num_kv_heads;
  a.G = num_q_heads / kv.num_kv_heads;
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
  a.done = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(part_ws) + ((part + 15) & ~size_t(15)));
  a.final_nlse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a.done) +
                                          (((size_t)pairs * sizeof(uint32_t) + 15) & ~size_t(15)));
  a.row_lse = row_lse;
  a.scores = scores;
  a.score_stride = score_stride;
  a.err = err;
  const uint64_t probe_ns = (uint64_t)t_wait_probe_us * 1000u;
  t_wait_probe_us = 0;
  // Pairs per chunk: their keys take about SE_SNAPKV_CHUNK_BYTES (at most
  // kMaxPairsPerChunk pairs: their prefix lives in shared memory).
  const size_t pair_bytes = (size_t)std::max(max_len, 1) * kD * 2;
  const int chunk = (int)std::min<size_t>(kMaxPairsPerChunk, std::max<size_t>(1, (size_t)SE_SNAPKV_CHUNK_BYTES / pair_bytes));
  cudaError_t e = cudaMemsetAsync(a.done, 0, (size_t)pairs * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const size_t smem = pass_smem_bytes(std::min(chunk, pairs));
  e = cudaFuncSetAttribute(snapkv_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(snapkv_pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  for (int p0 = 0; p0 < pairs; p0 += chunk) {
    a.pair0 = p0;
    a.pairs = std::min(chunk, pairs - p0);
    // Pass 1 of a later chunk touches nothing the pass 2 before it reads or
    // writes: it starts at once and waits for that launch only before it exits.
    a.wait_previous = p0 == 0 ? 1 : 0;
    a.late_wait = 0;
    a.probe_limit_ns = p0 == 0 ? probe_ns : 0;
    e = launch_pdl(snapkv_pass_kernel<1>, dim3(sm_count), dim3(kThreads), smem, stream, kmap, qmap, a);
    if (e != cudaSuccess) return e;
    // Pass 2 reads keys and queries (the inputs, complete once pass 1 has
    // started) and pass 1's -LSE: its copies and products start at once, its
    // epilogue waits for pass 1 before reading the -LSE.
    a.wait_previous = 1;
    a.late_wait = 1;
    a.probe_limit_ns = 0;
    e = launch_pdl(snapkv_pass_kernel<2>, dim3(sm_count), dim3(kThreads), smem, stream, kmap, qmap, a);
    if (e != cudaSuccess) return e;
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
