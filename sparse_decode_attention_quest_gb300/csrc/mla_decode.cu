// Sparse paged decode over a latent (MLA-style) cache (SparseEngine:
// Sparse-First Inference Engine, Figure 5 caption: GLM-4.7-Flash, an MLA model,
// decoding at 32K/128K; Table 7: logit z and weight alpha over the history).
//
// One cache row per token holds 576 dims (512 latent + 64 RoPE) and serves as
// the key; its first 512 dims are the value. All query heads (16..64) share the
// one KV head, so every selected page (16 rows x 1152 bytes) is read once and
// used by all heads: with 64 heads both products are dense contractions, and
// they run on the 5th-generation tensor cores with the scores and the output
// accumulated in tensor memory (TMEM).
//
//  * Work split as in the GQA decode: the selected pages of all requests form
//    one flattened range and every CTA takes an equal slice (>= 16 pages).
//  * A tile is 64 tokens (4 pages) in eight groups of 8 rows (group g: rows
//    8 g .. 8 g + 7, i.e. rows 0-7 or 8-15 of page g / 2), each group nine 64-dim
//    chunks of 8 rows x 128 bytes, 128-byte swizzled; two tiles are in flight.
//    One thread copies a group with one 3-D TMA box (64 dims x 8 rows x 9
//    chunks, 9 KiB): 8 boxes per tile instead of 36 of 2 KiB, since the TMA rate
//    goes with the number of boxes. A product's 8-row groups are then 9 KiB
//    apart, in token order. Pages not selected are not copied, and the value
//    dims of rows at or past the request's length are zeroed in shared memory
//    by the softmax warps before the PV MMAs read them.
//  * Two threads issue the MMAs: one the S^T MMAs of each tile chunk by chunk as
//    the chunks land, the other the PV MMAs of each tile once its P is written.
//  * S^T = K Q^T: one M = 64 tcgen05.mma per 16 dims (36 per tile) with the tile
//    as the K-major A operand and the request's queries (64 rows x 576 dims in
//    shared memory) as B; S^T lands in TMEM, token r in lane 32 (r / 16) + r % 16,
//    as two accumulators that the softmax adds (chunks 0-4 and 5-8, issued by
//    two threads: one thread issuing all 36 small MMAs of a tile takes 1.5 us).
//  * Eight softmax warps, two per page of the tile, read S^T (each thread one
//    token x 16 heads), take per-head tile maxima, keep a running maximum per
//    head that moves only when a tile exceeds it by 2^8 (then the output
//    accumulator columns of the heads that moved are rescaled in TMEM), and
//    write P as bf16 over the tile's RoPE chunks (one per group), which S^T no
//    longer needs.
//  * O^T += V^T P^T: four M = 128 MMAs per 16 tokens (dims 128 mt ..), A = the
//    tile's first 512 dims read MN-major, B = P read MN-major; O^T of all 64
//    heads is 4 x 64 TMEM columns. The epilogue divides by the softmax sums
//    and writes the output (one slice) or a partial for the combine kernel:
//    four heads per dim, one 16-byte store each (the softmax warps serve no
//    tile meanwhile; one 4-byte store per head and dim took three times as
//    long at every segment switch).
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kChunks = kD / 64;                        // 9 chunks of 64 dims
constexpr int kMinPagesPerCta = 16;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kTileTok = 64;                            // 4 pages per tile
constexpr int kTilePages = kTileTok / kPageSize;
constexpr int kGroupRows = 8;                           // rows of a copy group (half a page)
constexpr int kChunkBytes = kGroupRows * 128;           // 8 rows x 64 dims
constexpr int kGroupBytes = kChunks * kChunkBytes;      // 9 KB: one TMA box
constexpr int kStageBytes = (kTileTok / kGroupRows) * kGroupBytes;  // 72 KB
constexpr int kStages = 2;
constexpr int kQRows = 64;
constexpr int kQBytes = kChunks * kQRows * 128;         // 64 heads x 576 dims
constexpr int kPOff = 8 * kChunkBytes;                  // P of a group: over its RoPE chunk
constexpr int kQOff = kStages * kStageBytes;
constexpr int kMiscOff = kQOff + kQBytes;
constexpr int kThreads = 384;
constexpr int kSoftThreads = 256;                       // warps 0-7: softmax + epilogue
constexpr int kMmaWarp = 8;                             // lane 0 issues the S^T MMAs (and owns TMEM)
constexpr int kLoadWarp = 9;                            // lane 0 issues the TMA copies
constexpr int kPvWarp = 10;                             // lane 0 issues the PV MMAs
constexpr int kMmaWarp2 = 11;                           // lane 0 issues the S^T MMAs of chunks 5-8
constexpr int kTmemCols = 512;
// S^T of tile parity s is the sum of two accumulators (chunks 0-4 and 5-8, from
// two issuing threads): columns 128 s + 64 h, h = 0, 1.
constexpr int kSCol = 0;
constexpr int kOCol = 256;                              // O^T M-tile mt: columns 256 + 64 mt
constexpr float kRescaleLog2 = 8.f;                     // running max moves when exceeded by 2^8
constexpr uint32_t kSoftBar = 1;                        // named barrier of the softmax warps

// Shared memory after the Q buffer.
constexpr int kBarOff = 0;        // 32 mbarriers
constexpr int kTmemSlotOff = 256;
constexpr int kValidOff = 272;    // [2 stages][4 pages] valid rows
constexpr int kXmaxOff = 512;     // [2 tile parities][4 pages][64 heads] tile maxima
constexpr int kLsumOff = 2560;    // [4 pages][64] softmax sums
constexpr int kMrowOff = 3584;    // [64] running maxima
constexpr int kLinvOff = 3840;    // [64] 1 / sum
constexpr int kLseOff = 4096;     // [64] log2-sum-exp2
constexpr int kPrefixOff = 4352;  // [batch + 1]

struct MlaArgs {
  const uint16_t* kv;
  int32_t row_stride;
  const uint16_t* q;  // [B][Hq][576]
  int32_t Hq;
  int32_t batch;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* sel_counts;
  int32_t sel_stride;
  int32_t max_splits;
  int32_t num_pages;
  float scale_log2;
  uint16_t* out;     // [B][Hq][512]
  float* out_lse;
  float* o_part;     // [B * Hq / 4][max_splits][512][4]: four heads' partials per dim
  float* lse_part;   // [B * Hq][max_splits], log2 domain
  int32_t* item_ns;  // [B]
  unsigned* err;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ int find_item(const int* prefix, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Reduction of 16 values over the 16 lanes of a half-warp by halving exchanges
// (xor 1, 2, 4, 8: 15 shuffles). Afterwards v[0] holds the result for the value
// with index reduced_index(lane).
template <bool kMax>
__device__ __forceinline__ void half_warp_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int b = 1 << st, w = 8 >> st;
    const bool up = (lane & b) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, b);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
}
__device__ __forceinline__ int reduced_index(int lane) {
  return 8 * (lane & 1) + 4 * ((lane >> 1) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 3) & 1);
}

// Walks the tiles of a CTA's slice in order: request segments (the part of a
// request's selected pages inside the slice), each cut into tiles of 4 pages.
struct TileCursor {
  const int* prefix;
  int start, end, i_last;
  int item, lo, hi, ntiles, t, seg, j;
  bool valid;
  __device__ void open(int it) {
    for (item = it; item <= i_last; ++item) {
      const int p0 = prefix[item];
      lo = max(start, p0) - p0;
      hi = min(end, prefix[item + 1]) - p0;
      if (lo < hi) {
        ntiles = (hi - lo + kTilePages - 1) / kTilePages;
        t = 0;
        valid = true;
        return;
      }
    }
    valid = false;
  }
  __device__ void init(const int* pf, int st, int en, int i_first, int il) {
    prefix = pf;
    start = st;
    end = en;
    i_last = il;
    seg = 0;
    j = 0;
    open(i_first);
  }
  __device__ bool last() const { return t == ntiles - 1; }
  __device__ void next() {
    ++j;
    if (++t == ntiles) {
      ++seg;
      open(item + 1);
    }
  }
};

__global__ void __launch_bounds__(kThreads, 1) mla_decode_kernel(const __grid_constant__ CUtensorMap kvmap,
                                                                 const __grid_constant__ CUtensorMap qmap,
                                                                 const MlaArgs a) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* misc = smem + kMiscOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + kBarOff);
  uint64_t* full = bars;          // [2 stages] a tile landed (TMA transaction count)
  uint64_t* empty = bars + 18;    // [2] the PV MMAs of the stage's tile are done
  uint64_t* s_full = bars + 20;   // [2] S^T of a tile is in TMEM
  uint64_t* s_free = bars + 22;   // [2] S^T read by the softmax threads
  uint64_t* p_full = bars + 24;   // [2] P written, V rows past the length zeroed, O^T rescaled
  uint64_t* o_done = bars + 26;   // the PV MMAs of a tile are done
  uint64_t* o_free = bars + 27;   // O^T read by the epilogue (softmax threads)
  uint64_t* q_full = bars + 28;   // the request's queries landed
  uint64_t* q_empty = bars + 29;  // the last S^T MMA of a request's segment is done
  uint64_t* fin = bars + 30;      // every MMA of the CTA is done (both issuers)
  // The PV MMAs of a segment's last tile are done (one phase per segment).
  // The epilogue cannot wait for that on o_done: the softmax threads do not
  // wait for every tile's PV, so when they finish the last tile j, o_done may
  // still be in phase j - 1; a parity wait may only name the current or the
  // preceding phase, and phase j has the parity of the completed phase j - 2.
  uint64_t* o_last = bars + 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + kTmemSlotOff);
  int* tile_valid = reinterpret_cast<int*>(misc + kValidOff);
  float* xmax = reinterpret_cast<float*>(misc + kXmaxOff);
  float* lsum = reinterpret_cast<float*>(misc + kLsumOff);
  float* mrow = reinterpret_cast<float*>(misc + kMrowOff);
  float* linv = reinterpret_cast<float*>(misc + kLinvOff);
  float* lse_s = reinterpret_cast<float*>(misc + kLseOff);
  int* prefix = reinterpret_cast<int*>(misc + kPrefixOff);
  const int items = a.batch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < items; i += kThreads) {
    int c = a.sel_counts[i];
    if (c < 0 || c > a.sel_stride) {
      raise_error(a.err, SE_DEVERR_LENGTH);
      c = c < 0 ? 0 : a.sel_stride;
    }
    prefix[i + 1] = c;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (items + 31) / 32;
    const int lo = min(items, lane * per), hi = min(items, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += prefix[i + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tt = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += tt;
    }
    int run = incl - sum;
    if (lane == 0) prefix[0] = 0;
    for (int i = lo; i < hi; ++i) {
      run += prefix[i + 1];
      prefix[i + 1] = run;
    }
  }
  __syncthreads();
  const int total = prefix[items];
  const int per_cta = max(kMinPagesPerCta, (total + (int)gridDim.x - 1) / (int)gridDim.x);
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < items; i += kThreads) {
      const int p0 = prefix[i], cnt = prefix[i + 1] - p0;
      a.item_ns[i] = cnt == 0 ? 0 : (p0 + cnt - 1) / per_cta - p0 / per_cta + 1;
    }
  }
  const int start = blockIdx.x * per_cta;
  const int end = min(total, start + per_cta);
  if (start >= end) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&empty[s], 1);
      mbar_init(&s_full[s], 2);  // both S^T issuers commit
      mbar_init(&s_free[s], kSoftThreads);
      mbar_init(&p_full[s], kSoftThreads);
    }
    mbar_init(o_done, 1);
    mbar_init(o_free, kSoftThreads);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 2);
    mbar_init(fin, 3);
    mbar_init(o_last, 1);
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem0 = smem_addr(smem);
  const int i_first = find_item(prefix, items, start);
  const int i_last = find_item(prefix, items, end - 1);
  const int Hq = a.Hq;
  bool dead = false;  // a bounded wait gave up: leave the loops, no further waits

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 issues the copies, two groups (one box each) per selected page, all
    // signalling the stage's barrier; the lanes hold the page metadata.
    const uint64_t policy = l2_evict_first_policy();
    TileCursor c;
    c.init(prefix, start, end, i_first, i_last);
    int base = 0, ph_cur = 0, va_cur = 0, ph_nxt = 0, va_nxt = 0, n_b = 0, L = 0;
    const int32_t* sel_row = nullptr;
    const int32_t* bt_row = nullptr;
    // Metadata of page k of the segment (physical page, valid rows; 0 rows: not copied).
    auto meta = [&](int k, int& phys, int& valid) {
      phys = 0;
      valid = 0;
      if (k < c.hi - c.lo) {
        const int logical = sel_row[k];
        if (logical >= 0 && logical < n_b) {
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
    for (; c.valid; c.next()) {
      const int s = c.j & 1;
      if (c.t == 0) {
        const int b = c.item;
        L = a.seq_lens[b];
        if (L < 0) {
          if (lane == 0) raise_error(a.err, SE_DEVERR_LENGTH);
          L = 0;
        }
        n_b = (L + kPageSize - 1) / kPageSize;
        if (n_b > a.bt_stride) {
          if (lane == 0) raise_error(a.err, SE_DEVERR_LENGTH);
          n_b = a.bt_stride;
          L = n_b * kPageSize;
        }
        sel_row = a.sel + (size_t)c.item * a.sel_stride + c.lo;
        bt_row = a.block_table + (size_t)b * a.bt_stride;
        base = 0;
        meta(lane, ph_cur, va_cur);
        meta(lane + 32, ph_nxt, va_nxt);
      } else if (c.t * kTilePages == base + 32) {
        // The tile has left the first window: rotate (the new one is used 8 tiles later).
        base += 32;
        ph_cur = ph_nxt;
        va_cur = va_nxt;
        meta(base + 32 + lane, ph_nxt, va_nxt);
      }
      int phys[kTilePages], valid[kTilePages], live = 0;
#pragma unroll
      for (int pg = 0; pg < kTilePages; ++pg) {
        const int k = c.t * kTilePages + pg;
        const int pc = __shfl_sync(0xffffffffu, ph_cur, k & 31), vc = __shfl_sync(0xffffffffu, va_cur, k & 31);
        const int pn = __shfl_sync(0xffffffffu, ph_nxt, k & 31), vn = __shfl_sync(0xffffffffu, va_nxt, k & 31);
        const bool in_cur = k < base + 32;
        phys[pg] = in_cur ? pc : pn;
        valid[pg] = in_cur ? vc : vn;
        live += valid[pg] > 0;
      }
      if (lane == 0) {
        if (c.j >= 2 && !mbar_wait(&empty[s], ((c.j >> 1) - 1) & 1)) dead = true;
        if (!dead) {
#pragma unroll
          for (int pg = 0; pg < kTilePages; ++pg) tile_valid[s * kTilePages + pg] = valid[pg];
          uint8_t* st = smem + s * kStageBytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)live * 2 * kGroupBytes);
#pragma unroll
          for (int pg = 0; pg < kTilePages; ++pg)
            if (valid[pg] > 0)
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                tma_load_3d(st + (2 * pg + hf) * kGroupBytes, &kvmap, 0, phys[pg] * kPageSize + hf * kGroupRows, 0,
                            &full[s], policy);
          if (c.t == 0) {
            // The request's queries, once the previous segment's S^T MMAs are done with the buffer.
            if (c.seg >= 1 && !mbar_wait(q_empty, (c.seg - 1) & 1)) dead = true;
            if (!dead) {
              mbar_arrive_expect_tx(q_full, (uint32_t)Hq * kD * 2);
#pragma unroll
              for (int ch = 0; ch < kChunks; ++ch)
                tma_load_2d(smem + kQOff + ch * kQRows * 128, &qmap, ch * 64, c.item * Hq, q_full, policy);
            }
          }
        }
      }
      if (__shfl_sync(0xffffffffu, (int)dead, 0)) {
        dead = true;
        break;
      }
    }
    if (dead && lane == 0) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
  } else if (warp == kMmaWarp || warp == kMmaWarp2) {
    // ------------------------------------------------------------ S^T issuers
    // The score MMAs of each tile once it has landed: warp kMmaWarp the 64-dim
    // chunks 0-4 into the first accumulator, warp kMmaWarp2 chunks 5-8 into the
    // second (one thread issuing all 36 back to back takes 1.5 us a tile, two
    // take 1.0; splitting the 36 K steps 18 / 18 instead was slower).
    if (lane == 0) {
      const int hf = warp == kMmaWarp2 ? 1 : 0;
      const int ch0 = hf ? 5 : 0, ch1 = hf ? kChunks : 5;
      const uint32_t idesc_s = umma_idesc_bf16(64, Hq);
      // Operand descriptors of the bases; an MMA adds a constant offset (the
      // address field is bits 0-13 of (address >> 4), and every shared address
      // here is below 256 KB, so the additions never carry out of it).
      const uint64_t desc_k0 = umma_desc_sw128_groups(smem0, kGroupBytes);
      const uint64_t desc_q = umma_desc_sw128(smem0 + kQOff);
      constexpr uint64_t kStageDesc = kStageBytes >> 4;
      TileCursor c;
      c.init(prefix, start, end, i_first, i_last);
      for (; c.valid && !dead; c.next()) {
        const int s = c.j & 1;
        if ((c.t == 0 && !mbar_wait(q_full, c.seg & 1)) || (c.j >= 2 && !mbar_wait(&s_free[s], ((c.j >> 1) - 1) & 1))) {
          dead = true;
          break;
        }
        tc05_fence_after();  // after the softmax's read of this S^T buffer
        const uint32_t d_s = tmem + kSCol + s * 128 + hf * 64;
        const uint64_t dk = desc_k0 + (s ? kStageDesc : 0);
        if (!mbar_wait(&full[s], (c.j >> 1) & 1)) {
          dead = true;
          break;
        }
#pragma unroll 1
        for (int ch = ch0; ch < ch1; ++ch) {
          // 16 dims = 32 bytes = 2 per K step; a chunk is (chunk bytes >> 4) further.
          const uint64_t da = dk + (uint64_t)(ch * (kChunkBytes >> 4));
          const uint64_t dq = desc_q + (uint64_t)(ch * ((kQRows * 128) >> 4));
          tc05_mma_bf16(d_s, da, dq, idesc_s, ch != ch0 ? 1u : 0u);
          tc05_mma_bf16(d_s, da + 2, dq + 2, idesc_s, 1u);
          tc05_mma_bf16(d_s, da + 4, dq + 4, idesc_s, 1u);
          tc05_mma_bf16(d_s, da + 6, dq + 6, idesc_s, 1u);
        }
        if (dead) break;
        tc05_commit(&s_full[s]);
        if (c.last()) tc05_commit(q_empty);
      }
      if (dead) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
      tc05_commit(fin);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // O^T += V^T P^T of each tile once its P is written.
    if (lane == 0) {
      const uint32_t idesc_o = umma_idesc_bf16_mn(128, 64);
      // V^T and P^T read MN-major: 64 elements of M (dims, or heads) per 128-byte
      // row, the next 64 dims one chunk further, the next 8 tokens one group further.
      const uint64_t desc_v0 = umma_desc_sw128_mn_groups(smem0, kChunkBytes, kGroupBytes);
      constexpr uint64_t kStageDesc = kStageBytes >> 4, kPDesc = kPOff >> 4;
      TileCursor c;
      c.init(prefix, start, end, i_first, i_last);
      for (; c.valid; c.next()) {
        const int s = c.j & 1;
        const bool first = c.t == 0;
        if (!mbar_wait(&p_full[s], (c.j >> 1) & 1) || (first && c.seg >= 1 && !mbar_wait(o_free, (c.seg - 1) & 1))) {
          dead = true;
          break;
        }
        tc05_fence_after();
        // 16 tokens = 2 groups = (2 group bytes >> 4) per K step; 128 dims = 2
        // chunks = (2 chunk bytes >> 4) per M-tile.
        constexpr uint64_t kStep = (2 * kGroupBytes) >> 4, kMt = (2 * kChunkBytes) >> 4;
        const uint64_t dv = desc_v0 + (s ? kStageDesc : 0), dp = dv + kPDesc;
        const uint32_t acc0 = first ? 0u : 1u;
        // K step outer, M-tile inner: consecutive MMAs go to different accumulators.
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
          for (int mt = 0; mt < 4; ++mt)
            tc05_mma_bf16(tmem + kOCol + mt * 64, dv + mt * kMt + ks * kStep, dp + ks * kStep, idesc_o,
                          ks > 0 ? 1u : acc0);
        tc05_commit(&empty[s]);
        tc05_commit(o_done);
        if (c.last()) tc05_commit(o_last);
      }
      if (dead) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
      tc05_commit(fin);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Warp w: page w % 4 of the tile (its TMEM lane quarter), heads 32 (w / 4) ..;
    // thread: token `tok` of the page, heads hh .. hh + 15.
    const int q4 = warp & 3;
    const int tok = lane & 15, hh = 32 * (warp >> 2) + 16 * (lane >> 4);
    const int hr = hh + reduced_index(lane);  // head of this thread's reduction results
    const int row = q4 * kPageSize + tok;     // token row of the tile
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    float m_h[16], l_h[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m_h[i] = l_h[i] = 0.f;
    TileCursor c;
    c.init(prefix, start, end, i_first, i_last);
    for (; c.valid; c.next()) {
      const int j = c.j, t = c.t, s = j & 1;
      const bool ok_s = __all_sync(0xffffffffu, mbar_wait(&s_full[s], (j >> 1) & 1));
      uint32_t r[16];
      if (ok_s) {
        tc05_fence_after();
        uint32_t r2[16];
        tmem_ld16x2_16(tmem + lane_base + kSCol + s * 128 + 32 * (warp >> 2), r);
        tmem_ld16x2_16(tmem + lane_base + kSCol + s * 128 + 64 + 32 * (warp >> 2), r2);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = 0u;
      }
      tc05_fence_before();
      mbar_arrive(&s_free[s]);
      const bool ok_f = mbar_wait(&full[s], (j >> 1) & 1);  // valid rows of the tile
      dead = dead || !ok_s || !ok_f;
      const bool tok_ok = tok < tile_valid[s * kTilePages + q4];
      float x[16], v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[i] = (tok_ok && hh + i < Hq) ? __uint_as_float(r[i]) * a.scale_log2 : -INFINITY;
        v[i] = x[i];
      }
      if (!tok_ok && (warp >> 2) == 0) {
        // Rows past the request's length (or of pages not copied) hold stale
        // data: zero their value dims so that P = 0 times them stays 0.
        const uint32_t st = smem0 + s * kStageBytes + (row / kGroupRows) * kGroupBytes;
#pragma unroll 1
        for (int ch = 4 * (lane >> 4); ch < 4 * (lane >> 4) + 4; ++ch)
#pragma unroll
          for (int k = 0; k < 8; ++k) st_shared_v4(st + ch * kChunkBytes + swz128(row % kGroupRows, k), 0u, 0u, 0u, 0u);
      }
      // Fast path: after the segment's first tile, a tile whose scores all stay
      // within 2^8 of the running maxima changes nothing but P and l. Otherwise
      // (first tile, a larger score, or a failed wait) the tile maxima are
      // exchanged and the running maxima recomputed.
      bool need = t == 0 || dead;
#pragma unroll
      for (int i = 0; i < 16; ++i) need = need || x[i] > m_h[i] + kRescaleLog2;
      if (bar_red_or(kSoftBar, kSoftThreads, need)) {
        half_warp_reduce16<true>(v, lane);
        // Two buffers by tile parity: the barriers keep every thread within one
        // tile of the others.
        float* xm = xmax + s * 256;
        xm[q4 * 64 + hr] = v[0];
        if (bar_red_or(kSoftBar, kSoftThreads, dead)) {  // also publishes xmax
          dead = true;
          break;
        }
        // Running maximum per head: set by the segment's first tile, then moved
        // only when a tile exceeds it by 2^8 (so P stays <= 256). Every warp of
        // a head half computes the same maxima from the same tile maxima.
        float f[16];
        bool moved = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 w0 = *reinterpret_cast<const float4*>(xm + hh + 4 * k);
          const float4 w1 = *reinterpret_cast<const float4*>(xm + 64 + hh + 4 * k);
          const float4 w2 = *reinterpret_cast<const float4*>(xm + 128 + hh + 4 * k);
          const float4 w3 = *reinterpret_cast<const float4*>(xm + 192 + hh + 4 * k);
          const float tm[4] = {fmaxf(fmaxf(w0.x, w1.x), fmaxf(w2.x, w3.x)), fmaxf(fmaxf(w0.y, w1.y), fmaxf(w2.y, w3.y)),
                               fmaxf(fmaxf(w0.z, w1.z), fmaxf(w2.z, w3.z)), fmaxf(fmaxf(w0.w, w1.w), fmaxf(w2.w, w3.w))};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 4 * k + e;
            const float mo = m_h[i];
            const float mn = (t == 0 || tm[e] > mo + kRescaleLog2) ? tm[e] : mo;
            const bool mv = t > 0 && mn != mo;
            f[i] = mv ? fast_exp2(mo - mn) : 1.f;
            moved = moved || mv;
            m_h[i] = mn;
            l_h[i] = t == 0 ? 0.f : l_h[i] * f[i];
          }
        }
        if (__any_sync(0xffffffffu, moved)) {
          // The O^T columns of this warp's head half (its lane quarter) to the new maxima.
          const bool ok_o = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1));
          if (ok_o) {
            float fc[32];  // factor of column c of the half: lanes 0-15 hold heads 0-15, lanes 16-31 heads 16-31
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) fc[cc] = __shfl_sync(0xffffffffu, f[cc & 15], (cc >> 4) * 16);
            tc05_fence_after();
#pragma unroll 1
            for (int mt = 0; mt < 4; ++mt) {
              const uint32_t ta = tmem + lane_base + kOCol + mt * 64 + 32 * (warp >> 2);
              uint32_t o[32];
              tmem_ld32(ta, o);
              tmem_ld_wait();
#pragma unroll
              for (int cc = 0; cc < 32; ++cc) o[cc] = __float_as_uint(__uint_as_float(o[cc]) * fc[cc]);
              tmem_st32(ta, o);
            }
            tmem_st_wait();
          } else {
            dead = true;
          }
        }
      }
      // P of this token for heads hh .. hh + 15 into its row of its group's RoPE
      // chunk (64 heads per 128-byte row).
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float ma = m_h[2 * i] == -INFINITY ? 0.f : m_h[2 * i];
        const float mb = m_h[2 * i + 1] == -INFINITY ? 0.f : m_h[2 * i + 1];
        const float pa = fast_exp2(x[2 * i] - ma), pb = fast_exp2(x[2 * i + 1] - mb);
        l_h[2 * i] += pa;
        l_h[2 * i + 1] += pb;
        pk[i] = pack_bf16x2(pa, pb);
      }
      const uint32_t prow = smem0 + s * kStageBytes + (row / kGroupRows) * kGroupBytes + kPOff;
      st_shared_v4(prow + swz128(row % kGroupRows, hh >> 3), pk[0], pk[1], pk[2], pk[3]);
      st_shared_v4(prow + swz128(row % kGroupRows, (hh >> 3) + 1), pk[4], pk[5], pk[6], pk[7]);
      fence_proxy_async_smem();
      tc05_fence_before();
      mbar_arrive(&p_full[s]);

      if (c.last()) {
        // ---- epilogue of the segment: O = O^T / l per head, or a partial
        const int b = c.item;
        const bool ok_e = __all_sync(0xffffffffu, mbar_wait(o_last, c.seg & 1));
        dead = dead || !ok_e;
        float w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = l_h[i];
        half_warp_reduce16<false>(w, lane);
        lsum[q4 * 64 + hr] = w[0];
        if (q4 == 0 && tok == 0)
#pragma unroll
          for (int i = 0; i < 16; ++i) mrow[hh + i] = m_h[i];
        named_bar_sync(kSoftBar, kSoftThreads);
        if (threadIdx.x < 64) {
          const int h = threadIdx.x;
          const float l = (lsum[h] + lsum[64 + h]) + (lsum[128 + h] + lsum[192 + h]);
          linv[h] = l > 0.f ? 1.f / l : 0.f;
          lse_s[h] = l > 0.f ? mrow[h] + log2f(l) : -INFINITY;
        }
        named_bar_sync(kSoftBar, kSoftThreads);
        const int p0 = prefix[b], cnt = prefix[b + 1] - p0;
        const int first_cta = p0 / per_cta;
        const int ns = (p0 + cnt - 1) / per_cta - first_cta + 1;
        const int slot = blockIdx.x - first_cta;
        if (ok_e) {
          tc05_fence_after();
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + kOCol + mt * 64 + 32 * (warp >> 2), o);
            tmem_ld_wait();
            const int d = mt * 128 + 32 * q4 + lane;
            if (ns == 1) {
#pragma unroll
              for (int cc = 0; cc < 32; ++cc) {
                const int h = 32 * (warp >> 2) + cc;
                if (h < Hq) {
                  const float val = __uint_as_float(o[cc]) * linv[h];
                  a.out[((size_t)b * Hq + h) * kDv + d] = (uint16_t)(pack_bf16x2(val, 0.f) & 0xffffu);
                }
              }
            } else {
              // A partial: the thread's four heads 4 k .. 4 k + 3 at its dim d in
              // one 16-byte store (four 4-byte stores per value run at a
              // fraction of the rate and hold up the softmax warps).
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int h = 32 * (warp >> 2) + 4 * k;
                if (h < Hq) {
                  const float4 val =
                      make_float4(__uint_as_float(o[4 * k]) * linv[h], __uint_as_float(o[4 * k + 1]) * linv[h + 1],
                                  __uint_as_float(o[4 * k + 2]) * linv[h + 2], __uint_as_float(o[4 * k + 3]) * linv[h + 3]);
                  const size_t blk = ((size_t)b * Hq + h) / 4;
                  *reinterpret_cast<float4*>(a.o_part + ((blk * a.max_splits + slot) * kDv + d) * 4) = val;
                }
              }
            }
          }
        }
        if (threadIdx.x < Hq) {
          const size_t orow = (size_t)b * Hq + threadIdx.x;
          if (ns == 1) {
            if (a.out_lse) a.out_lse[orow] = lse_s[threadIdx.x] * kLn2;
          } else {
            a.lse_part[orow * a.max_splits + slot] = lse_s[threadIdx.x];
          }
        }
        tc05_fence_before();
        mbar_arrive(o_free);
      }
    }
  }
  if (warp == kMmaWarp && lane == 0 && !mbar_wait(fin, 0)) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Merge the partials of the items spread over several CTAs; one warp per four
// query heads of a request (the partials hold four heads per dim). Splits come
// in chunks of 32: lane s holds the four heads' log-sum-exps of split s of the
// chunk (one round trip);
// lane l takes dims 4 l + 128 j (j = 0..3, 4 consecutive dims each) of the four
// heads, and the splits are added in split order, two at a time in flight.
// Items held by one CTA were written directly; rows of requests with no
// selected page get 0 and lse = -inf.
__global__ void __launch_bounds__(128) mla_combine_kernel(const float* __restrict__ o_part,
                                                          const float* __restrict__ lse_part,
                                                          const int32_t* __restrict__ item_ns, int32_t batch,
                                                          int32_t Hq, int32_t max_splits, uint16_t* __restrict__ out,
                                                          float* __restrict__ out_lse) {
  pdl_enter();
  const int blk = blockIdx.x * 4 + (threadIdx.x >> 5);  // four heads: rows 4 blk .. 4 blk + 3
  if (blk * 4 >= batch * Hq) return;
  const int lane = threadIdx.x & 31;
  const int ns = min(item_ns[(blk * 4) / Hq], max_splits);
  if (ns == 1) return;
  float ls[4], M[4], wsum[4];
#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    const float* lp = lse_part + (size_t)(blk * 4 + hh) * max_splits;
    ls[hh] = lane < ns ? lp[lane] : -INFINITY;  // the first chunk
    float m = ls[hh];
    for (int c0 = 32; c0 < ns; c0 += 32) m = fmaxf(m, c0 + lane < ns ? lp[c0 + lane] : -INFINITY);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    M[hh] = m;
    wsum[hh] = 0.f;
  }
  // acc[j][e]: dim 4 lane + 128 j + e, the four heads in x, y, z, w
  float4 acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* op = o_part + (size_t)blk * max_splits * kDv * 4;
  auto load = [&](int sp, float4 (&v)[4][4]) {
    const float* p = op + (size_t)sp * kDv * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[j][e] = *reinterpret_cast<const float4*>(p + (size_t)(4 * lane + 128 * j + e) * 4);
  };
  auto add = [&](int sp, const float4 (&v)[4][4]) {
    float f[4];
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const float l = __shfl_sync(0xffffffffu, ls[hh], sp & 31);
      f[hh] = l == -INFINITY ? 0.f : fast_exp2(l - M[hh]);
      wsum[hh] += f[hh];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[j][e].x += f[0] * v[j][e].x;
        acc[j][e].y += f[1] * v[j][e].y;
        acc[j][e].z += f[2] * v[j][e].z;
        acc[j][e].w += f[3] * v[j][e].w;
      }
  };
  for (int sp = 0; sp < ns; sp += 2) {  // warp-uniform
    if (sp > 0 && (sp & 31) == 0)  // the next chunk's log-sum-exps
#pragma unroll
      for (int hh = 0; hh < 4; ++hh)
        ls[hh] = sp + lane < ns ? lse_part[(size_t)(blk * 4 + hh) * max_splits + sp + lane] : -INFINITY;
    float4 v0[4][4], v1[4][4];
    load(sp, v0);
    if (sp + 1 < ns) load(sp + 1, v1);
    add(sp, v0);
    if (sp + 1 < ns) add(sp + 1, v1);
  }
  float inv[4], lse[4];
#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    const bool empty_row = !(wsum[hh] > 0.f);
    inv[hh] = empty_row ? 0.f : 1.f / wsum[hh];
    lse[hh] = empty_row ? -INFINITY : (M[hh] + log2f(wsum[hh])) * kLn2;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int d = 4 * lane + 128 * j;
    uint2 pk[4];
    pk[0].x = pack_bf16x2(acc[j][0].x * inv[0], acc[j][1].x * inv[0]);
    pk[0].y = pack_bf16x2(acc[j][2].x * inv[0], acc[j][3].x * inv[0]);
    pk[1].x = pack_bf16x2(acc[j][0].y * inv[1], acc[j][1].y * inv[1]);
    pk[1].y = pack_bf16x2(acc[j][2].y * inv[1], acc[j][3].y * inv[1]);
    pk[2].x = pack_bf16x2(acc[j][0].z * inv[2], acc[j][1].z * inv[2]);
    pk[2].y = pack_bf16x2(acc[j][2].z * inv[2], acc[j][3].z * inv[2]);
    pk[3].x = pack_bf16x2(acc[j][0].w * inv[3], acc[j][1].w * inv[3]);
    pk[3].y = pack_bf16x2(acc[j][2].w * inv[3], acc[j][3].w * inv[3]);
#pragma unroll
    for (int hh = 0; hh < 4; ++hh)
      *reinterpret_cast<uint2*>(out + (size_t)(blk * 4 + hh) * kDv + d) = pk[hh];
  }
  if (out_lse && lane < 4)
    out_lse[blk * 4 + lane] = lane == 0 ? lse[0] : lane == 1 ? lse[1] : lane == 2 ? lse[2] : lse[3];
}

size_t smem_bytes(int32_t batch) { return 1024 + (size_t)kMiscOff + kPrefixOff + (size_t)(batch + 1) * 4; }

}  // namespace

bool mla_decode_supported(int num_kv_heads, int head_dim, int head_dim_v, int num_q_heads) {
  return num_kv_heads == 1 && head_dim == kD && head_dim_v == kDv && num_q_heads % 16 == 0 && num_q_heads >= 16 &&
         num_q_heads <= 64;
}

DecodePlan plan_mla_decode(int32_t sel_stride, int sm_count) {
  DecodePlan p;
  p.pages_per_split = kMinPagesPerCta;
  p.nsplit = (sel_stride + kMinPagesPerCta - 1) / kMinPagesPerCta + 1;
  p.grid = sm_count;
  return p;
}

size_t mla_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, const DecodePlan& plan) {
  const size_t rows = (size_t)batch * num_q_heads;
  const size_t part = rows * plan.nsplit * ((size_t)kDv + 1) * sizeof(float);
  return ((part + 15) & ~size_t(15)) + (size_t)batch * sizeof(int32_t);
}

// Requests one launch takes: the per-request prefix must fit beside the two
// tiles and the queries in shared memory.
size_t mla_decode_max_items() { return (227 * 1024 - smem_bytes(0)) / 4; }

cudaError_t launch_mla_decode(const CUtensorMap& kvmap, const CUtensorMap& qmap, const KvView& kv, const uint16_t* q,
                              int32_t num_q_heads, const int32_t* block_table,
                              int32_t bt_stride, const int32_t* seq_lens, int32_t batch, const int32_t* sel_pages,
                              const int32_t* sel_counts, int32_t sel_stride, float sm_scale, uint16_t* out,
                              float* out_lse, void* workspace, const DecodePlan& plan, unsigned* err,
                              cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  MlaArgs a;
  a.kv = kv.k;
  a.row_stride = kv.row_stride_k;
  a.q = q;
  a.Hq = num_q_heads;
  a.batch = batch;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.sel = sel_pages;
  a.sel_counts = sel_counts;
  a.sel_stride = sel_stride;
  a.max_splits = plan.nsplit;
  a.num_pages = kv.num_pages;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = out;
  a.out_lse = out_lse;
  const size_t rows = (size_t)batch * num_q_heads;
  const size_t part = rows * plan.nsplit * ((size_t)kDv + 1) * sizeof(float);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o_part = reinterpret_cast<float*>(ws);
  a.lse_part = a.o_part + rows * plan.nsplit * kDv;
  a.item_ns = reinterpret_cast<int32_t*>(ws + ((part + 15) & ~size_t(15)));
  a.err = err;
  const size_t smem = smem_bytes(batch);
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mla_decode_kernel, dim3(plan.grid), dim3(kThreads), smem, stream, kvmap, qmap, a);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mla_combine_kernel, dim3((unsigned)((rows / 4 + 3) / 4)), dim3(128), 0, stream, a.o_part, a.lse_part,
                 a.item_ns, batch, num_q_heads, plan.nsplit, out, out_lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace se
