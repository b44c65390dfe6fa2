// One Quest decode step in a single launch (SparseEngine: Sparse-First Inference
// Engine, Figure 2 caption: Quest as the query-dependent retrieval method;
// Figure 3 caption: the summaries kept beside the KV blocks; Tables 9-12: the
// sink / recent keep windows beside the selected budget; Table 7: logit z and
// weight alpha, the history includes the current token).
//
// A thread-block cluster of C CTAs (C = 1, 2, 4 or 8) serves one (request, KV
// head) item; the scores never leave the cluster's shared memory:
//   0. append (optional): rank 0 writes the new token's K/V rows and updates the
//      summary of its page (the last page, which is never a scoring candidate);
//   1. score: P/N of the item's query group (all threads); rank r scores the
//      candidate pages c0 + r, c0 + r + C, ... of the keep window; each warp
//      scores 4 pages per iteration (8 lanes per 512 B summary block of the KV
//      head), streamed through an 8-stage cp.async ring, and stores the scores'
//      order keys straight into rank 0's shared memory;
//   2. select (rank 0): bucket-selects the topk best (1,024 linear score
//      buckets, the threshold bucket's members ranked exactly, ties to the
//      lower page; a radix select when that bucket is crowded) and writes the kept
//      pages, ascending (sink window, selected, recent window), to its shared
//      memory and to the caller's selection arrays;
//   3. decode: rank r takes the kept pages r, r + C, ...; its 8 warps stream
//      them through 3-stage cp.async rings (128-byte swizzle, rows past the
//      length zero-filled) with the m16n8k16 bf16 MMA and an online softmax in
//      log2; the warps merge in shared memory, every rank pushes its partial
//      into rank 0's shared memory, and rank 0 merges the C partials and writes
//      out and lse.
// Cluster barriers separate the phases; every thread of the cluster reaches
// each of them.
#include <cooperative_groups.h>

#include "se_ptx.cuh"

namespace cg = cooperative_groups;

namespace se {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBlk = 2 * kD * 2;                      // one KV head's summary block (min, max rows)
constexpr int kPagesPerIter = 4;                      // summary blocks a warp scores per iteration
constexpr int kScoreStages = 8;                       // ring stages of kPagesPerIter blocks
constexpr int kHalfBytes = 16 * 64 * 2;               // one 64-column half of a (page, head) block
constexpr int kTileBytes = 2 * kHalfBytes;            // K or V block of one page
constexpr int kPageBytes = 2 * kTileBytes;            // K then V
constexpr int kDecStages = 3;
constexpr int kMaxCand = 8192;                        // candidate pages per request
constexpr int kMaxKept = 2048;                        // kept pages per (request, KV head)
constexpr int kSelBuckets = 1024;                     // linear score buckets of the selection
constexpr int kSelMaxMembers = 512;                   // members of the threshold bucket ranked one by one
constexpr int kRegionA = kWarps * kDecStages * kPageBytes;  // 192 KB, reused phase by phase
constexpr float kLn2 = 0.6931471805599453f;

// Phase-1/2 layout inside region A.
constexpr int kScoreRingOff = 0;                                                    // [8][8][4][512]
constexpr int kKeysOff = kScoreRingOff + kWarps * kScoreStages * kPagesPerIter * kBlk;  // uint32 [kMaxCand]
static_assert(kKeysOff + kMaxCand * 4 <= kRegionA, "phase-1/2 storage fits region A");
static_assert(kSelBuckets * 4 + kSelMaxMembers * 8 + kMaxCand / 8 + 2 * kWarps * 4 + 16 <= kKeysOff,
              "the selection's scratch fits the idle score ring");
static_assert(kWarps * 16 * kD * 4 <= kRegionA, "warp states fit region A");

struct FusedArgs {
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* k_mut;
  uint16_t* v_mut;
  uint16_t* summary;
  int32_t num_pages;
  int32_t H;
  int32_t row_stride_k;
  int32_t row_stride_v;
  const uint16_t* k_new;  // [B][H][128] or null
  const uint16_t* v_new;
  const uint16_t* q;      // [B][Hq][128]
  int32_t group;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;  // tokens after the append
  int32_t max_seq_len;
  int32_t topk;
  int32_t sink;
  int32_t recent;
  float scale_log2;
  uint16_t* out;
  float* out_lse;
  int32_t* sel;
  int32_t* sel_counts;
  int32_t sel_stride;
  unsigned* err;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The score whose order key is u (order_key's inverse).
__device__ __forceinline__ float key_value(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Candidate pages [c0, c1): none of the first `sink` tokens, none of the last
// `recent` tokens; the last page is always kept.
__device__ __forceinline__ void candidate_window(int L, int n, int sink, int recent, int& c0, int& c1) {
  const int rf = L > recent ? (L - recent) / kPageSize : 0;
  c1 = max(0, min(rf, n - 1));
  c0 = min((min(sink, L) + kPageSize - 1) / kPageSize, c1);
}

// Block-wide exclusive prefix of one int per thread, in thread order.
__device__ __forceinline__ int block_scan(int v, int* wtot, int warp, int lane, int& total) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  int before = incl - v;
  total = 0;
  for (int w = 0; w < kWarps; ++w) {
    const int x = wtot[w];
    before += (w < warp) ? x : 0;
    total += x;
  }
  __syncthreads();
  return before;
}

template <bool kHiRows>
__global__ void __launch_bounds__(kThreads, 1) quest_fused_kernel(const FusedArgs a) {
  pdl_enter();
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int item = blockIdx.x / C;
  const int H = a.H, G = a.group, Hq = H * G;
  const int b = item / H, h = item % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* regA = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* pn = reinterpret_cast<float*>(regA + kRegionA);  // [2][128]: N (min row), P (max row)
  int* sel_s = reinterpret_cast<int*>(pn + 2 * kD);       // [kMaxKept]
  float* part_o = reinterpret_cast<float*>(sel_s + kMaxKept);  // [16][128]: this CTA's merged rows
  float* part_ml = part_o + 16 * kD;                            // [2][16]
  float* red_ml = part_ml + 32;                                 // [2][kWarps][16]
  int* misc = reinterpret_cast<int*>(red_ml + 2 * kWarps * 16);  // [0] kept count, [1..3] scratch, [8..15] scan
  int* hist = misc + 16;                                          // [256]
  uint32_t* keys = reinterpret_cast<uint32_t*>(regA + kKeysOff);  // rank 0: order keys of every candidate
  uint32_t* keys0 = cluster.map_shared_rank(keys, 0);
  const uint32_t regA_addr = smem_addr(regA);
  cluster.sync();  // every rank has started before any rank writes into rank 0's shared memory

  int L = a.seq_lens[b];
  if (L < 0 || L > a.max_seq_len) {
    if (tid == 0 && rank == 0) raise_error(a.err, SE_DEVERR_LENGTH);
    L = L < 0 ? 0 : a.max_seq_len;
  }
  const int n = (L + kPageSize - 1) / kPageSize;
  const int32_t* bt_row = a.block_table + (size_t)b * a.bt_stride;

  // ---- 0. append the new token (rank 0, warp 0)
  if (a.k_new != nullptr && rank == 0 && warp == 0 && L > 0) {
    const int pos = L - 1, page = pos / kPageSize, slot = pos % kPageSize;
    const int phys = bt_row[page];
    if (phys < 0 || phys >= a.num_pages) {
      if (lane == 0) raise_error(a.err, SE_DEVERR_PAGE_RANGE);
    } else {
      const size_t blk = (size_t)phys * H + h;
      const uint32_t* ks = reinterpret_cast<const uint32_t*>(a.k_new + (size_t)item * kD);
      const uint32_t* vs = reinterpret_cast<const uint32_t*>(a.v_new + (size_t)item * kD);
      uint32_t* kd = reinterpret_cast<uint32_t*>(a.k_mut + (blk * kPageSize + slot) * a.row_stride_k);
      uint32_t* vd = reinterpret_cast<uint32_t*>(a.v_mut + (blk * kPageSize + slot) * a.row_stride_v);
      uint32_t* smin = reinterpret_cast<uint32_t*>(a.summary + blk * 2 * kD);
      uint32_t* smax = smin + kD / 2;
      for (int c = lane; c < kD / 2; c += 32) {
        const uint32_t x = ks[c];
        kd[c] = x;
        vd[c] = vs[c];
        if (slot == 0) {
          smin[c] = x;
          smax[c] = x;
        } else {
          const uint32_t lo = smin[c], hi = smax[c];
          smin[c] = pack_bf16x2(fminf(bf16_lo(lo), bf16_lo(x)), fminf(bf16_hi(lo), bf16_hi(x)));
          smax[c] = pack_bf16x2(fmaxf(bf16_lo(hi), bf16_lo(x)), fmaxf(bf16_hi(hi), bf16_hi(x)));
        }
      }
      // the rows are read by the decode copies of every CTA of the cluster
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }

  // ---- 1. score the candidate pages of this rank
  int c0, c1;
  candidate_window(L, n, a.sink, a.recent, c0, c1);
  const int Cn = c1 - c0;
  const int mine = Cn > rank ? (Cn - rank + C - 1) / C : 0;  // candidates j = rank + C i, i < mine
  for (int c = tid; c < kD; c += kThreads) {
    float P = 0.f, N = 0.f;
    const uint16_t* qc = a.q + ((size_t)b * Hq + h * G) * kD + c;
    for (int g = 0; g < G; ++g) {
      const float x = __uint_as_float((uint32_t)qc[(size_t)g * kD] << 16);
      P += fmaxf(x, 0.f);
      N += fminf(x, 0.f);
    }
    pn[c] = N;
    pn[kD + c] = P;
  }
  __syncthreads();
  // Lane group q = lane / 8 scores page 4 s + q of the warp's pages at iteration s;
  // lane gl = lane % 8 holds chunks gl + 8 e (e = 0..3) of the 32 16-byte chunks of
  // a summary block: chunk c is row c / 16 (0: min, times N; 1: max, times P),
  // channels (c % 16) * 8 .. + 7.
  const int gq = lane >> 3, gl = lane & 7;
  float mult[4][8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int c = gl + 8 * e;
#pragma unroll
    for (int x = 0; x < 8; ++x) mult[e][x] = pn[(c >> 4) * kD + (c & 15) * 8 + x];
  }
  {
    // this warp: local candidates i = warp + kWarps t, t < np1
    const int np1 = mine > warp ? (mine - warp + kWarps - 1) / kWarps : 0;
    const int iters = (np1 + kPagesPerIter - 1) / kPagesPerIter;
    const uint32_t ring = regA_addr + kScoreRingOff + warp * kScoreStages * kPagesPerIter * kBlk;
    auto phys_of = [&](int t) {
      if (t >= np1) return -1;
      const int page = c0 + rank + C * (warp + kWarps * t);
      return bt_row[page];
    };
    // Physical pages of t = base .. base + 127, lane l holding base + l + 32 k in w[k].
    int base = 0, w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = phys_of(base + 32 * k + lane);
    auto lookup = [&](int t) {
      const int d = t - base;
      const int v0 = __shfl_sync(0xffffffffu, w[0], d & 31), v1 = __shfl_sync(0xffffffffu, w[1], d & 31);
      const int v2 = __shfl_sync(0xffffffffu, w[2], d & 31), v3 = __shfl_sync(0xffffffffu, w[3], d & 31);
      const int k = d >> 5;
      return k == 0 ? v0 : k == 1 ? v1 : k == 2 ? v2 : v3;
    };
    auto issue = [&](int s) {
      const int t = s * kPagesPerIter + gq;
      const int ph = lookup(t);
      if (t < np1 && ph >= 0 && ph < a.num_pages) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.summary) + ((size_t)ph * H + h) * kBlk;
        const uint32_t dst = ring + ((s % kScoreStages) * kPagesPerIter + gq) * kBlk;
#pragma unroll
        for (int e = 0; e < 4; ++e) cp_async16(dst + (gl + 8 * e) * 16, src + (gl + 8 * e) * 16, 16u);
      }
    };
#pragma unroll 1
    for (int s0 = 0; s0 < kScoreStages - 1; ++s0) {
      if (s0 < iters) issue(s0);
      cp_async_commit();
    }
    for (int s0 = 0; s0 < iters; ++s0) {
      // The pages of this iteration have left the first half of the windows: rotate
      // by 64 pages; the new windows are first looked up 9 iterations later.
      if (s0 * kPagesPerIter == base + 64) {
        base += 64;
        w[0] = w[2];
        w[1] = w[3];
        w[2] = phys_of(base + 64 + lane);
        w[3] = phys_of(base + 96 + lane);
      }
      if (s0 + kScoreStages - 1 < iters) issue(s0 + kScoreStages - 1);
      cp_async_commit();
      cp_async_wait<kScoreStages - 1>();
      __syncwarp();
      const int t = s0 * kPagesPerIter + gq;
      const int ph = lookup(t);
      const bool good = ph >= 0 && ph < a.num_pages;
      const uint8_t* blk = regA + kScoreRingOff +
                           ((size_t)(warp * kScoreStages + s0 % kScoreStages) * kPagesPerIter + gq) * kBlk;
      float pe[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint4 v = *reinterpret_cast<const uint4*>(blk + (gl + 8 * e) * 16);
        float x = bf16_lo(v.x) * mult[e][0];
        x = fmaf(bf16_hi(v.x), mult[e][1], x);
        x = fmaf(bf16_lo(v.y), mult[e][2], x);
        x = fmaf(bf16_hi(v.y), mult[e][3], x);
        x = fmaf(bf16_lo(v.z), mult[e][4], x);
        x = fmaf(bf16_hi(v.z), mult[e][5], x);
        x = fmaf(bf16_lo(v.w), mult[e][6], x);
        pe[e] = fmaf(bf16_hi(v.w), mult[e][7], x);
      }
      float acc = (pe[0] + pe[1]) + (pe[2] + pe[3]);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      __syncwarp();  // every lane has read the stage before it is refilled
      if (gl == 0 && t < np1) {
        if (!good) raise_error(a.err, SE_DEVERR_PAGE_RANGE);
        keys0[rank + C * (warp + kWarps * t)] = order_key(good ? acc : -INFINITY);  // candidate j, in rank 0
      }
    }
    cp_async_wait<0>();
  }
  cluster.sync();  // every rank's scores are in its shared memory

  // ---- 2. select (rank 0)
  if (rank == 0) {
    int* wtot = misc + 8;
    int cnt;
    if (Cn <= a.topk) {
      cnt = n;
      for (int i = tid; i < n; i += kThreads) sel_s[i] = i;
    } else {
      // Bucket select (one pass over the keys): the scores' min and max over
      // the finite ones, kSelBuckets linear buckets between them (monotone in
      // the score), the bucket B that holds the topk-th largest (every key in a
      // higher bucket is selected), and an exact ranking of B's members by
      // order key, then lower index. Warp w owns the contiguous candidates
      // [32 E w, 32 E (w + 1)), its lane l the candidates 32 E w + 32 i + l
      // (conflict-free reads); the kept ones are bits of a candidate bitmap set
      // by warp ballots, whose words leave in order behind a popcount prefix. A
      // crowded B (near-identical scores) falls back to a radix select over all
      // keys.
      // Scratch: the score ring of region A, idle once the scores are in.
      int* bhist = reinterpret_cast<int*>(regA + kScoreRingOff);                  // [kSelBuckets]
      uint32_t* mkey = reinterpret_cast<uint32_t*>(bhist + kSelBuckets);          // [kSelMaxMembers]
      int* midx = reinterpret_cast<int*>(mkey + kSelMaxMembers);                  // [kSelMaxMembers]
      uint32_t* selbits = reinterpret_cast<uint32_t*>(midx + kSelMaxMembers);     // [kMaxCand / 32]
      float* wmm = reinterpret_cast<float*>(selbits + kMaxCand / 32);             // [2][kWarps]
      int* sinfo = reinterpret_cast<int*>(wmm + 2 * kWarps);                      // [4]
      const int E = (Cn + kThreads - 1) / kThreads;  // candidates per lane
      const int wbase = warp * 32 * E;
      float lmin = INFINITY, lmax = -INFINITY;
      for (int i = 0; i < E; ++i) {
        const int j = wbase + 32 * i + lane;
        if (j >= Cn) break;
        const float v = key_value(keys[j]);
        if (isfinite(v)) {
          lmin = fminf(lmin, v);
          lmax = fmaxf(lmax, v);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lmin = fminf(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
        lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
      }
      if (lane == 0) {
        wmm[warp] = lmin;
        wmm[kWarps + warp] = lmax;
      }
      for (int i = tid; i < kSelBuckets; i += kThreads) bhist[i] = 0;
      for (int i = tid; i < kMaxCand / 32; i += kThreads) selbits[i] = 0u;
      if (tid == 0) sinfo[2] = 0;
      __syncthreads();
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        mn = fminf(mn, wmm[w]);
        mx = fmaxf(mx, wmm[kWarps + w]);
      }
      const float scale = (mx > mn) ? (float)kSelBuckets / (mx - mn) : 0.f;
      auto bucket_of = [&](float v) {
        if (isfinite(v)) return min(kSelBuckets - 1, max(0, (int)((v - mn) * scale)));
        return v > 0.f ? kSelBuckets - 1 : 0;  // +inf on top; -inf and NaN in bucket 0
      };
      for (int i = 0; i < E; ++i) {
        const int j = wbase + 32 * i + lane;
        if (j >= Cn) break;
        atomicAdd(&bhist[bucket_of(key_value(keys[j]))], 1);
      }
      __syncthreads();
      {
        // thread t owns buckets [4 t, 4 t + 4); the bucket of the topk-th largest
        static_assert(kSelBuckets == 4 * kThreads, "four buckets per thread");
        int hc[4], sum = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hc[q] = bhist[4 * tid + q];
          sum += hc[q];
        }
        int tot;
        const int below = block_scan(sum, wtot, warp, lane, tot);
        int cum = tot - below - sum;  // keys in the buckets above this thread's
#pragma unroll
        for (int q = 3; q >= 0; --q) {
          if (cum < a.topk && a.topk <= cum + hc[q]) {
            sinfo[0] = 4 * tid + q;
            sinfo[1] = cum;
          }
          cum += hc[q];
        }
      }
      __syncthreads();
      const int B = sinfo[0];
      const int need = a.topk - sinfo[1];  // members of bucket B to take, >= 1
      const int m = bhist[B];
      if (m <= kSelMaxMembers) {
        // One pass: every candidate above B sets its bit of the candidate bitmap
        // (a warp's ballot over its i-th candidates is word 32 E w / 32 + i, as the
        // warp owns candidates [32 E w, 32 E (w + 1))), and B's members are listed.
        for (int i = 0; i < E; ++i) {
          const int j = wbase + 32 * i + lane;
          const bool in = j < Cn;
          const uint32_t u = in ? keys[j] : 0u;
          const int bk = in ? bucket_of(key_value(u)) : -1;
          const unsigned above = __ballot_sync(0xffffffffu, bk > B);
          if (lane == 0) selbits[(wbase >> 5) + i] = above;
          if (bk == B) {
            const int slot = atomicAdd(&sinfo[2], 1);
            mkey[slot] = u;
            midx[slot] = j;
          }
        }
        __syncthreads();
        // A member is kept when fewer than `need` members rank before it (key
        // descending, then lower index).
        for (int i = tid; i < m; i += kThreads) {
          const uint32_t ku = mkey[i];
          const int ji = midx[i];
          int rank = 0;
          for (int x = 0; x < m; ++x) {
            const uint32_t kx = mkey[x];
            rank += (kx > ku || (kx == ku && midx[x] < ji)) ? 1 : 0;
          }
          if (rank < need) atomicOr(&selbits[ji >> 5], 1u << (ji & 31));
        }
        __syncthreads();
        // Output in candidate order: thread t holds bitmap word t.
        static_assert(kMaxCand / 32 == kThreads, "one bitmap word per thread");
        const uint32_t wv = tid < (Cn + 31) / 32 ? selbits[tid] : 0u;
        int tot;
        int pos = block_scan(__popc(wv), wtot, warp, lane, tot);
        for (uint32_t v = wv; v; v &= v - 1, ++pos)
          if (pos < a.topk) sel_s[c0 + pos] = c0 + 32 * tid + __ffs(v) - 1;
      } else {
        // radix select of the topk-th largest key T (4 passes of 8 bits)
        uint32_t prefix = 0, mask = 0;
        int remaining = a.topk;
        for (int shift = 24; shift >= 0; shift -= 8) {
          for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
          __syncthreads();
          for (int j0 = 0; j0 < Cn; j0 += kThreads) {  // warp-uniform: one atomic per distinct digit and warp
            const int j = j0 + tid;
            int digit = 256;
            if (j < Cn) {
              const uint32_t u = keys[j];
              if ((u & mask) == prefix) digit = (int)((u >> shift) & 255u);
            }
            const unsigned peers = __match_any_sync(0xffffffffu, digit);
            if (digit < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
          }
          __syncthreads();
          if (warp == 0) {
            int g8[8], gsum = 0;
  #pragma unroll
            for (int q = 0; q < 8; ++q) {
              g8[q] = hist[lane * 8 + q];
              gsum += g8[q];
            }
            int incl = gsum;  // keys in bins >= lane * 8
  #pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int t = __shfl_down_sync(0xffffffffu, incl, o);
              if (lane + o < 32) incl += t;
            }
            const int above = incl - gsum;
            if (above < remaining && remaining <= incl) {
              int cum = above;
              for (int q = 7; q >= 0; --q) {
                if (cum + g8[q] >= remaining) {
                  misc[1] = lane * 8 + q;
                  misc[2] = cum;
                  break;
                }
                cum += g8[q];
              }
            }
          }
          __syncthreads();
          remaining -= misc[2];
          prefix |= (uint32_t)misc[1] << shift;
          mask |= 255u << shift;
          __syncthreads();
        }
        // selected: keys above T, then the lowest-index keys equal to T; thread t owns
        // the contiguous candidates [t E, t E + E) so the output comes out ascending
        const int E = (Cn + kThreads - 1) / kThreads;
        const int j0 = min(Cn, tid * E), j1 = min(Cn, j0 + E);
        int n_eq = 0;
        for (int j = j0; j < j1; ++j) n_eq += keys[j] == prefix ? 1 : 0;
        int tot;
        int eq_rank = block_scan(n_eq, wtot, warp, lane, tot);
        int n_sel = 0;
        for (int j = j0; j < j1; ++j) {
          const uint32_t u = keys[j];
          if (u > prefix || (u == prefix && eq_rank++ < remaining)) ++n_sel;
        }
        int pos = block_scan(n_sel, wtot, warp, lane, tot);
        eq_rank -= n_eq;  // back to this thread's first equal key
        for (int j = j0; j < j1; ++j) {
          const uint32_t u = keys[j];
          if (u > prefix || (u == prefix && eq_rank++ < remaining)) {
            if (pos < a.topk) sel_s[c0 + pos] = c0 + j;
            ++pos;
          }
        }
      }
      for (int i = tid; i < c0; i += kThreads) sel_s[i] = i;
      for (int i = tid; i < n - c1; i += kThreads) sel_s[c0 + a.topk + i] = c1 + i;
      cnt = c0 + a.topk + (n - c1);
    }
    if (tid == 0) misc[0] = cnt;
    __syncthreads();
    int32_t* gsel = a.sel + (size_t)item * a.sel_stride;
    for (int i = tid; i < cnt; i += kThreads) gsel[i] = sel_s[i];
    if (tid == 0) a.sel_counts[item] = cnt;
  }
  cluster.sync();  // the kept list is in rank 0's shared memory

  // ---- 3. decode the kept pages of this rank
  const int* sel0 = cluster.map_shared_rank(sel_s, 0);
  const int kept = *cluster.map_shared_rank(misc, 0);
  const int mine3 = kept > rank ? (kept - rank + C - 1) / C : 0;  // kept index rank + C i
  const int np = mine3 > warp ? (mine3 - warp + kWarps - 1) / kWarps : 0;  // i = warp + kWarps t
  const int g = lane >> 2, t4 = lane & 3;
  const uint32_t wring = regA_addr + warp * kDecStages * kPageBytes;
  auto meta = [&](int t, int& phys, int& valid) {
    phys = 0;
    valid = 0;
    if (t < np) {
      const int logical = sel0[rank + C * (warp + kWarps * t)];
      if (logical >= 0 && logical < n) {
        const int ph = bt_row[logical];
        if (ph >= 0 && ph < a.num_pages) {
          phys = ph;
          valid = min(kPageSize, L - logical * kPageSize);
        } else {
          raise_error(a.err, SE_DEVERR_PAGE_RANGE);
        }
      } else {
        raise_error(a.err, SE_DEVERR_LENGTH);
      }
    }
  };
  int base = 0, ph_cur, va_cur, ph_nxt, va_nxt;
  meta(lane, ph_cur, va_cur);
  meta(lane + 32, ph_nxt, va_nxt);
  auto lookup = [&](int t, int& phys, int& valid) {
    const int pc = __shfl_sync(0xffffffffu, ph_cur, t & 31), vc = __shfl_sync(0xffffffffu, va_cur, t & 31);
    const int pq = __shfl_sync(0xffffffffu, ph_nxt, t & 31), vq = __shfl_sync(0xffffffffu, va_nxt, t & 31);
    const bool in_cur = t < base + 32;
    phys = in_cur ? pc : pq;
    valid = in_cur ? vc : vq;
  };
  auto issue_page = [&](int t) {
    int phys, valid;
    lookup(t, phys, valid);
    const uint32_t stage = wring + (t % kDecStages) * kPageBytes;
    const size_t blk = ((size_t)phys * H + h) * kPageSize;
    const uint16_t* kp = a.k + blk * a.row_stride_k;
    const uint16_t* vp = a.v + blk * a.row_stride_v;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int c = lane + 32 * it;  // 16-byte chunk 0..255 of the 16 x 256-byte block
      const int r = c >> 4, q16 = c & 15;
      const uint32_t off = (uint32_t)(q16 >> 3) * kHalfBytes + swz128(r, q16 & 7);
      const bool in = r < valid;
      cp_async16(stage + off, kp + (size_t)(in ? r : 0) * a.row_stride_k + q16 * 8, in ? 16u : 0u);
      cp_async16(stage + kTileBytes + off, vp + (size_t)(in ? r : 0) * a.row_stride_v + q16 * 8, in ? 16u : 0u);
    }
  };
#pragma unroll
  for (int t = 0; t < kDecStages - 1; ++t) {
    if (t < np) issue_page(t);
    cp_async_commit();
  }
  uint32_t qa[8][4];
  {
    const uint16_t* qrow0 = a.q + ((size_t)b * Hq + h * G + g) * kD;
    const uint16_t* qrow1 = a.q + ((size_t)b * Hq + h * G + g + 8) * kD;
    const bool r0 = g < G, r1 = kHiRows && (g + 8 < G);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c = ks * 16 + 2 * t4;
      qa[ks][0] = r0 ? *reinterpret_cast<const uint32_t*>(qrow0 + c) : 0u;
      qa[ks][2] = r0 ? *reinterpret_cast<const uint32_t*>(qrow0 + c + 8) : 0u;
      qa[ks][1] = r1 ? *reinterpret_cast<const uint32_t*>(qrow1 + c) : 0u;
      qa[ks][3] = r1 ? *reinterpret_cast<const uint32_t*>(qrow1 + c + 8) : 0u;
    }
  }
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  for (int t = 0; t < np; ++t) {
    const int tn = t + kDecStages - 1;
    if (tn == base + 64) {  // the copy ahead needs the next window: rotate
      base += 32;
      ph_cur = ph_nxt;
      va_cur = va_nxt;
      meta(base + 32 + lane, ph_nxt, va_nxt);
    }
    if (tn < np) issue_page(tn);
    cp_async_commit();
    cp_async_wait<kDecStages - 1>();
    __syncwarp();
    int ph_t, valid;
    lookup(t, ph_t, valid);
    (void)ph_t;
    if (valid > 0) {
      const uint32_t kt = wring + (t % kDecStages) * kPageBytes;
      const uint32_t vt = kt + kTileBytes;
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int krow = (lane & 7) + ((lane >> 4) << 3);
      const int ksub = (lane >> 3) & 1;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4(r0, r1, r2, r3, kt + (ks >> 2) * kHalfBytes + swz128(krow, ((ks & 3) << 1) + ksub));
        mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r0, r1);
        mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r2, r3);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = nt * 8 + 2 * t4 + (e & 1);
          sc[nt][e] = tok < valid ? sc[nt][e] * a.scale_log2 : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float f0 = fast_exp2(m0 - n0), f1 = fast_exp2(m1 - n1);
      m0 = n0;
      m1 = n1;
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        p[nt][0] = fast_exp2(sc[nt][0] - n0);
        p[nt][1] = fast_exp2(sc[nt][1] - n0);
        p[nt][2] = fast_exp2(sc[nt][2] - n1);
        p[nt][3] = fast_exp2(sc[nt][3] - n1);
      }
      l0 = l0 * f0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
      l1 = l1 * f1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= f0;
        o[j][1] *= f0;
        o[j][2] *= f1;
        o[j][3] *= f1;
      }
      const uint32_t pa0 = pack_bf16x2(p[0][0], p[0][1]);
      const uint32_t pa1 = pack_bf16x2(p[0][2], p[0][3]);
      const uint32_t pa2 = pack_bf16x2(p[1][0], p[1][1]);
      const uint32_t pa3 = pack_bf16x2(p[1][2], p[1][3]);
      const int vtok = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int vsub = lane >> 4;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int chunk = 2 * j + vsub;
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4_trans(r0, r1, r2, r3, vt + (chunk >> 3) * kHalfBytes + swz128(vtok, chunk & 7));
        mma_bf16_16816(o[2 * j], pa0, pa1, pa2, pa3, r0, r1);
        mma_bf16_16816(o[2 * j + 1], pa0, pa1, pa2, pa3, r2, r3);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  // merge the warps (their rings are idle: the states go to region A)
  __syncthreads();
  float* red_o = reinterpret_cast<float*>(regA);  // [kWarps][16][128]
  if (t4 == 0) {
    red_ml[warp * 16 + g] = m0;
    red_ml[kWarps * 16 + warp * 16 + g] = l0;
    red_ml[warp * 16 + g + 8] = m1;
    red_ml[kWarps * 16 + warp * 16 + g + 8] = l1;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    *reinterpret_cast<float2*>(red_o + ((size_t)warp * 16 + g) * kD + j * 8 + 2 * t4) = make_float2(o[j][0], o[j][1]);
    *reinterpret_cast<float2*>(red_o + ((size_t)warp * 16 + g + 8) * kD + j * 8 + 2 * t4) =
        make_float2(o[j][2], o[j][3]);
  }
  __syncthreads();
  for (int idx = tid; idx < G * kD; idx += kThreads) {
    const int r = idx / kD, d = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[w * 16 + r]);
    float lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red_ml[w * 16 + r];
      const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
      lsum += f * red_ml[kWarps * 16 + w * 16 + r];
      acc += f * red_o[((size_t)w * 16 + r) * kD + d];
    }
    part_o[r * kD + d] = acc;  // unnormalised, relative to M
    if (d == 0) {
      part_ml[r] = M;
      part_ml[16 + r] = lsum;
    }
  }
  // push this rank's partial into rank 0's region A (idle once every rank has
  // passed the barrier below: rank 0's rings and warp states are no longer used)
  cluster.sync();
  {
    float* dst = cluster.map_shared_rank(reinterpret_cast<float*>(regA), 0) + (size_t)rank * (16 * kD + 32);
    for (int i = tid; i < G * kD; i += kThreads) dst[i] = part_o[i];
    for (int i = tid; i < 32; i += kThreads) dst[16 * kD + i] = part_ml[i];
  }
  cluster.sync();  // every rank's partial is in rank 0's shared memory

  // ---- rank 0 merges the ranks' partials and writes the output
  if (rank == 0) {
    const float* parts = reinterpret_cast<const float*>(regA);  // [C][16 * 128 + 32]
    for (int idx = tid; idx < G * kD; idx += kThreads) {
      const int r = idx / kD, d = idx % kD;
      float M = -INFINITY;
      for (int q = 0; q < C; ++q) M = fmaxf(M, parts[(size_t)q * (16 * kD + 32) + 16 * kD + r]);
      float lsum = 0.f, acc = 0.f;
      for (int q = 0; q < C; ++q) {
        const float* pq = parts + (size_t)q * (16 * kD + 32);
        const float mq = pq[16 * kD + r];
        const float f = (mq == -INFINITY) ? 0.f : fast_exp2(mq - M);
        lsum += f * pq[16 * kD + 16 + r];
        acc += f * pq[r * kD + d];
      }
      const bool empty_row = !(lsum > 0.f);
      const size_t row = (size_t)b * Hq + h * G + r;
      a.out[row * kD + d] = __bfloat16_as_ushort(__float2bfloat16_rn(empty_row ? 0.f : acc / lsum));
      if (a.out_lse && d == 0) a.out_lse[row] = empty_row ? -INFINITY : (M + log2f(lsum)) * kLn2;
    }
  }
}

size_t fused_smem_bytes() {
  return 1024 + (size_t)kRegionA + 2 * kD * 4 + kMaxKept * 4 + 16 * kD * 4 + 32 * 4 + 2 * kWarps * 16 * 4 +
         (16 + 256) * 4;
}

template <bool kHiRows>
cudaError_t launch_fused(const FusedArgs& a, int items, int C, cudaStream_t stream) {
  const size_t smem = fused_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(quest_fused_kernel<kHiRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items * C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, quest_fused_kernel<kHiRows>, a);
}

}  // namespace

int fused_max_candidates() { return kMaxCand; }
int fused_max_kept() { return kMaxKept; }

int fused_cluster_size(int items, int sm_count) {
  int C = 1;
  while (C < 8 && items * C * 2 <= sm_count) C *= 2;
  return C;
}

cudaError_t launch_quest_fused(const KvView& kv, uint16_t* k_mut, uint16_t* v_mut, const uint16_t* k_new,
                               const uint16_t* v_new, const uint16_t* q, int32_t num_q_heads,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens, int32_t batch,
                               int32_t max_seq_len, int32_t topk, int32_t sink_tokens, int32_t recent_tokens,
                               float sm_scale, uint16_t* out, float* out_lse, int32_t* sel, int32_t* sel_counts,
                               int32_t sel_stride, int sm_count, unsigned* err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  FusedArgs a;
  a.k = kv.k;
  a.v = kv.v;
  a.k_mut = k_mut;
  a.v_mut = v_mut;
  a.summary = kv.summary;
  a.num_pages = kv.num_pages;
  a.H = kv.num_kv_heads;
  a.row_stride_k = kv.row_stride_k;
  a.row_stride_v = kv.row_stride_v;
  a.k_new = k_new;
  a.v_new = v_new;
  a.q = q;
  a.group = num_q_heads / kv.num_kv_heads;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.max_seq_len = max_seq_len;
  a.topk = topk;
  a.sink = sink_tokens;
  a.recent = recent_tokens;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = out;
  a.out_lse = out_lse;
  a.sel = sel;
  a.sel_counts = sel_counts;
  a.sel_stride = sel_stride;
  a.err = err;
  const int items = batch * kv.num_kv_heads;
  const int C = fused_cluster_size(items, sm_count);
  return a.group > 8 ? launch_fused<true>(a, items, C, stream) : launch_fused<false>(a, items, C, stream);
}

}  // namespace se
