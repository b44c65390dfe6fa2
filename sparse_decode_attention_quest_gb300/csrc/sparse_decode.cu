// Sparse paged flash-decode over the Quest-selected pages (SparseEngine:
// Sparse-First Inference Engine, Figure 2 caption: attention execution reads
// the method's view of the cache; Table 7: the logit z and weight alpha, the
// history includes the current token).
//
// GQA path (head_dim = head_dim_v = 128, 1..16 query heads per KV head):
//  * the selected pages of all (request, KV head) items form one flattened
//    range; every CTA takes an equal slice (at least 16 pages), so ragged
//    selections balance. A slice is cut at item boundaries into segments;
//  * one CTA serves a whole query group, so every selected (page, head) block
//    is read from HBM once. The four warps of a CTA take every fourth page of
//    the slice; each warp streams its pages through its own ring of 4 KB
//    stages (six for groups of up to 8 heads, five above) with 16-byte
//    cp.async copies, a page's K block and V block in stages of their own, so
//    that all but one block of the ring are in flight while the warp computes.
//    The stream runs on across item boundaries: the pages of the next item
//    are already in flight while a segment's state is merged. Each lane holds
//    the metadata (physical page, valid tokens, KV head) of one page of a
//    32-page window, loaded a window ahead of the copies;
//    the copies write the 128-byte-swizzled layout that makes the ldmatrix
//    reads conflict-free, and token rows at or past the request's length are
//    zero-filled instead of read, so stale cache slots (even NaN) never reach
//    the output;
//  * per page: S = Q K^T and O += P V on the tensor cores with the m16n8k16
//    bf16 MMA (query heads are the 16 rows), an online softmax in the log2
//    domain, fp32 accumulation;
//  * at the end of a segment warps 1..3 stage their states in shared memory
//    and stream on; warp 0 merges them with its own, element by element of its
//    MMA fragments. An item held by one CTA writes its output directly; an
//    item spread over several CTAs writes normalised partials (output,
//    log-sum-exp), and the CTA that publishes the item's last partial merges
//    them: o = sum_s exp(lse_s - LSE) o_s. Each CTA counts itself in on a
//    per-item arrival counter in the workspace; the last one resets it to
//    zero, so a workspace that starts zeroed is left zeroed by every call.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kHeadDim = 128;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kHalfBytes = 16 * 64 * 2;     // one 64-column half of a (page, head) block
constexpr int kTileBytes = 2 * kHalfBytes;  // one (page, head) block of K or V: one stage
constexpr int kMinPagesPerCta = 16;
constexpr int kCtasPerSm = 2;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeArgs {
  const uint16_t* k;
  const uint16_t* v;
  int32_t row_stride_k;
  int32_t row_stride_v;
  const uint16_t* q;
  int32_t group;
  int32_t num_kv_heads;
  int32_t batch;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* sel_counts;
  int32_t sel_stride;
  int32_t max_splits;
  int32_t num_pages;
  float scale_log2;  // sm_scale * log2(e)
  uint16_t* out;
  float* out_lse;
  float* o_part;     // [B * Hq][max_splits][128]
  float* lse_part;   // [B * Hq][max_splits], log2 domain
  uint32_t* arrivals;  // [B * H]: CTAs of a split item that have published their partial (zero between calls)
  unsigned* err;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Largest i in [0, n - 1] with prefix[i] <= x: the item whose page range holds x.
__device__ __forceinline__ int find_item(const int* prefix, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Copy one (page, head) block of K or V (cache base, row stride) into a stage;
// rows >= valid are zero-filled without reading the cache.
__device__ __forceinline__ void issue_block(const uint16_t* cache, int row_stride, int num_kv_heads,
                                            uint32_t stage, int phys, int h, int valid, int lane) {
  const uint16_t* src = cache + ((size_t)phys * num_kv_heads + h) * kPageSize * row_stride;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int c = lane + 32 * it;  // 16-byte chunk 0..255 of the 16 x 256-byte block
    const int r = c >> 4, q16 = c & 15;
    const uint32_t off = (uint32_t)(q16 >> 3) * kHalfBytes + swz128(r, q16 & 7);
    const bool in = r < valid;
    cp_async16(stage + off, src + (size_t)(in ? r : 0) * row_stride + q16 * 8, in ? 16u : 0u);
  }
}

// Shared memory of a decode CTA. Query groups of up to 8 heads keep six blocks
// per warp ring; groups of 9..16 heads stage twice the rows and keep five.
template <bool kHiRows>
struct DecodeSmem {
  static constexpr int kStages = kHiRows ? 5 : 6;  // blocks per warp ring
  static constexpr int kRows = kHiRows ? 16 : 8;   // query rows of a warp's state that can be real heads
  static constexpr int kRing = kWarps * kStages * kTileBytes;
  static constexpr int kSlots = 2 * kRows * kHeadDim * 4;  // two warp states (o) for the mid-stream merge
  static constexpr int kSlotMl = 2 * 2 * 16 * 4;           // their (m, l) per row
  static constexpr int kFlags = kThreads * 4;              // items whose partials this CTA merges
  static constexpr int kFixed = kRing + kSlots + kSlotMl + kFlags + 128;  // + alignment of the ring
  static_assert(kWarps * kRows * kHeadDim * 4 + 3 * kWarps * 16 * 4 <= kRing, "end-of-stream staging fits the ring");
};

__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <bool kHiRows>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) gqa_decode_kernel(const DecodeArgs a) {
  using Cfg = DecodeSmem<kHiRows>;
  constexpr int kStages = Cfg::kStages;
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  float* slots = reinterpret_cast<float*>(ring + Cfg::kRing);    // [2][kRows][128]
  float* slot_ml = slots + 2 * Cfg::kRows * kHeadDim;           // [2][(m, l)][16]
  int* flags = reinterpret_cast<int*>(slot_ml + 2 * 2 * 16);     // [kThreads]
  int* prefix = flags + kThreads;                                // [items + 1]
  const int H = a.num_kv_heads, G = a.group, Hq = H * G;
  const int items = a.batch * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // A guess made before the counts arrive: every item has sel_stride selected
  // pages (a top-k that fills its budget). Under it, the page ids and lengths
  // of this warp's first 32 pages are loaded beside the counts, and their
  // block-table entries while the prefix is summed; the guess is checked
  // below and the values are used only if it holds.
  const int total_g = items * a.sel_stride;
  const int per_cta_g = max(kMinPagesPerCta, (total_g + (int)gridDim.x - 1) / (int)gridDim.x);
  const int start_g = blockIdx.x * per_cta_g, end_g = min(total_g, start_g + per_cta_g);
  const bool lane_g = start_g + warp + kWarps * lane < end_g;
  int g_it = 0, g_logical = -1, g_L = 0;
  if (lane_g) {
    const int p = start_g + warp + kWarps * lane;
    g_it = p / a.sel_stride;
    g_logical = a.sel[(size_t)g_it * a.sel_stride + (p - g_it * a.sel_stride)];
    g_L = a.seq_lens[g_it / a.num_kv_heads];
  }

  // Selected pages per item, then an exclusive prefix.
  bool full = true;
  for (int i = threadIdx.x; i < items; i += kThreads) {
    int c = a.sel_counts[i];
    full = full && c == a.sel_stride;
    if (c < 0 || c > a.sel_stride) {
      raise_error(a.err, SE_DEVERR_LENGTH);
      c = c < 0 ? 0 : a.sel_stride;
    }
    prefix[i + 1] = c;
  }
  int g_ph = -1;
  if (lane_g) {
    const int L = max(g_L, 0);
    const int n_b = min((L + kPageSize - 1) / kPageSize, a.bt_stride);
    if (g_logical >= 0 && g_logical < n_b) g_ph = a.block_table[(size_t)(g_it / a.num_kv_heads) * a.bt_stride + g_logical];
  }
  const bool guess_ok = __syncthreads_and(full);
  if (warp == 0) {
    const int per = (items + 31) / 32;
    const int lo = min(items, lane * per), hi = min(items, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += prefix[i + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
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
  // Items with no selected page get a zero output and lse = -inf (the empty sum).
  if (blockIdx.x == 0) {
    for (int idx = threadIdx.x; idx < items * G; idx += kThreads) {
      const int i = idx / G;
      if (prefix[i + 1] != prefix[i]) continue;
      const size_t row = (size_t)(i / H) * Hq + (i % H) * G + idx % G;
      for (int d = 0; d < kHeadDim; d += 8) *reinterpret_cast<uint4*>(a.out + row * kHeadDim + d) = make_uint4(0, 0, 0, 0);
      if (a.out_lse) a.out_lse[row] = -INFINITY;
    }
  }
  const int start = blockIdx.x * per_cta;
  const int end = min(total, start + per_cta);
  if (start >= end) return;

  const uint32_t wring = smem_addr(ring) + warp * kStages * kTileBytes;
  const int g = lane >> 2, t = lane & 3;
  const int i_first = find_item(prefix, items, start);
  const int i_last = find_item(prefix, items, end - 1);
  auto nonempty_from = [&](int it) {
    for (; it <= i_last; ++it)
      if (max(start, prefix[it]) < min(end, prefix[it + 1])) return it;
    return -1;
  };
  // This warp's pages of the slice, across item boundaries: start + warp + kWarps kk, kk < np.
  const int np = (end - start > warp) ? (end - start - warp + kWarps - 1) / kWarps : 0;

  // Metadata of page kk: physical page, and valid tokens | KV head << 8
  // (zeros past the slice or on a bad index, which is reported).
  auto meta = [&](int kk, int& phys, int& vh) {
    phys = 0;
    vh = 0;
    if (kk < np) {
      const int p = start + warp + kWarps * kk;
      const int it = find_item(prefix, items, p);
      const int b = it / H;
      const int logical = a.sel[(size_t)it * a.sel_stride + (p - prefix[it])];
      int L = a.seq_lens[b];
      if (L < 0) {
        raise_error(a.err, SE_DEVERR_LENGTH);
        L = 0;
      }
      int n_b = (L + kPageSize - 1) / kPageSize;
      if (n_b > a.bt_stride) {
        raise_error(a.err, SE_DEVERR_LENGTH);
        n_b = a.bt_stride;
        L = n_b * kPageSize;
      }
      if (logical >= 0 && logical < n_b) {
        const int ph = a.block_table[(size_t)b * a.bt_stride + logical];
        if (ph >= 0 && ph < a.num_pages) {
          phys = ph;
          vh = min(kPageSize, L - logical * kPageSize) | ((it % H) << 8);
        } else {
          raise_error(a.err, SE_DEVERR_PAGE_RANGE);
        }
      } else {
        raise_error(a.err, SE_DEVERR_LENGTH);
      }
    }
  };
  // Two windows of 32 pages, one page per lane: [base, base + 32) in *_cur,
  // the next 32 in *_nxt (read only once the copies reach them, so that their
  // loads stay in flight meanwhile).
  int base = 0, ph_cur = 0, vh_cur = 0, ph_nxt = 0, vh_nxt = 0;
  if (guess_ok) {
    // The first window from the values loaded under the guess (which held),
    // with the checks of meta().
    if (lane < np) {
      int L = g_L;
      if (L < 0) {
        raise_error(a.err, SE_DEVERR_LENGTH);
        L = 0;
      }
      int n_b = (L + kPageSize - 1) / kPageSize;
      if (n_b > a.bt_stride) {
        raise_error(a.err, SE_DEVERR_LENGTH);
        n_b = a.bt_stride;
        L = n_b * kPageSize;
      }
      if (g_logical >= 0 && g_logical < n_b) {
        if (g_ph >= 0 && g_ph < a.num_pages) {
          ph_cur = g_ph;
          vh_cur = min(kPageSize, L - g_logical * kPageSize) | ((g_it % H) << 8);
        } else {
          raise_error(a.err, SE_DEVERR_PAGE_RANGE);
        }
      } else {
        raise_error(a.err, SE_DEVERR_LENGTH);
      }
    }
  } else {
    meta(lane, ph_cur, vh_cur);
  }
  auto lookup = [&](int kk, int& phys, int& vh) {
    if (kk < base + 32) {
      phys = __shfl_sync(0xffffffffu, ph_cur, kk & 31);
      vh = __shfl_sync(0xffffffffu, vh_cur, kk & 31);
    } else {
      phys = __shfl_sync(0xffffffffu, ph_nxt, kk & 31);
      vh = __shfl_sync(0xffffffffu, vh_nxt, kk & 31);
    }
  };
  // Block j of the warp's stream (K of page j / 2 for even j, V for odd j) is
  // commit group j of the warp and sits in stage j mod kStages; the stream runs
  // on across item boundaries, so the ring never drains between segments.
  auto issue = [&](int j) {
    const int kk = j >> 1;
    if (kk == base + 64) {  // the copies reach the next window: rotate
      base += 32;
      ph_cur = ph_nxt;
      vh_cur = vh_nxt;
      meta(base + 32 + lane, ph_nxt, vh_nxt);
    }
    if (kk < np) {
      int ph, vh;
      lookup(kk, ph, vh);
      const uint32_t stage = wring + (j % kStages) * kTileBytes;
      if (j & 1)
        issue_block(a.v, a.row_stride_v, H, stage, ph, vh >> 8, vh & 0xff, lane);
      else
        issue_block(a.k, a.row_stride_k, H, stage, ph, vh >> 8, vh & 0xff, lane);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int j = 0; j < kStages; ++j) issue(j);
  meta(lane + 32, ph_nxt, vh_nxt);  // after the first copies: its loads overlap them

  int item = nonempty_from(i_first);
  int kk = 0;
  bool first_segment = true;
  uint32_t qa[8][4];
  float o[16][4];
  while (true) {
    const int b = item / H, h = item % H;
    const int p0 = prefix[item];
    const int seg_hi = min(end, prefix[item + 1]);
    const int kk_hi = seg_hi - start - warp > 0 ? (seg_hi - start - warp + kWarps - 1) / kWarps : 0;
    {
      const uint16_t* qrow0 = a.q + ((size_t)b * Hq + h * G + g) * kHeadDim;
      const uint16_t* qrow1 = a.q + ((size_t)b * Hq + h * G + g + 8) * kHeadDim;
      const bool r0 = g < G, r1 = kHiRows && (g + 8 < G);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c = ks * 16 + 2 * t;
        qa[ks][0] = r0 ? *reinterpret_cast<const uint32_t*>(qrow0 + c) : 0u;
        qa[ks][2] = r0 ? *reinterpret_cast<const uint32_t*>(qrow0 + c + 8) : 0u;
        qa[ks][1] = r1 ? *reinterpret_cast<const uint32_t*>(qrow1 + c) : 0u;
        qa[ks][3] = r1 ? *reinterpret_cast<const uint32_t*>(qrow1 + c + 8) : 0u;
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    for (; kk < kk_hi; ++kk) {
      int ph_k, vh_k;
      lookup(kk, ph_k, vh_k);
      (void)ph_k;
      const int valid = vh_k & 0xff;
      uint32_t pa0 = 0u, pa1 = 0u, pa2 = 0u, pa3 = 0u;
      cp_async_wait<kStages - 1>();  // K of page kk has landed (this thread's copies)
      __syncwarp();                  // ... and every lane's
      if (valid > 0) {
        const uint32_t kt = wring + ((2 * kk) % kStages) * kTileBytes;
        // S = Q K^T : two n-tiles of 8 tokens, 8 k-steps of 16 dims.
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
        // Online softmax in the log2 domain; tokens >= valid are masked.
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + 2 * t + (e & 1);
            sc[nt][e] = tok < valid ? sc[nt][e] * a.scale_log2 : -INFINITY;
          }
        float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float c0 = fast_exp2(m0 - n0), c1 = fast_exp2(m1 - n1);
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
        l0 = l0 * c0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
        l1 = l1 * c1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          o[j][0] *= c0;
          o[j][1] *= c0;
          o[j][2] *= c1;
          o[j][3] *= c1;
        }
        pa0 = pack_bf16x2(p[0][0], p[0][1]);
        pa1 = pack_bf16x2(p[0][2], p[0][3]);
        pa2 = pack_bf16x2(p[1][0], p[1][1]);
        pa3 = pack_bf16x2(p[1][2], p[1][3]);
      }
      __syncwarp();  // every lane is done with the K stage before it is refilled
      issue(2 * kk + kStages);
      cp_async_wait<kStages - 1>();  // V of page kk has landed (this thread's copies)
      __syncwarp();                  // ... and every lane's
      if (valid > 0) {
        const uint32_t vt = wring + ((2 * kk + 1) % kStages) * kTileBytes;
        // O += P V : 16 n-tiles of 8 dims, one k-step of 16 tokens (zero rows past valid).
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
      __syncwarp();  // every lane is done with the V stage before it is refilled
      issue(2 * kk + 1 + kStages);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    const int next = nonempty_from(item + 1);
    const int first_cta = p0 / per_cta;
    const int ns = (prefix[item + 1] - 1) / per_cta - first_cta + 1;  // CTAs the item spans
    const int slot = blockIdx.x - first_cta;
    const size_t row0 = (size_t)b * Hq + h * G;
    if (next >= 0) {
      // ---- A segment that ends mid-stream: the four warps' states merge in
      // two rounds through two shared slots while the copies of the next
      // item's pages stay in flight. Warps 2 and 3 hand their states over and
      // stream on; warp 1 folds in warp 3's and hands the sum to warp 0, which
      // folds in warp 2's and warp 1's and writes the item's output (or its
      // partial, published at the end of the stream). Named barriers: 1 (the
      // slots hold warps 2 and 3), 2 (slot 1 holds warp 1's sum), 3 (warp 0 is
      // done with the slots).
      auto stage_state = [&](int s) {
        float* dst = slots + s * Cfg::kRows * kHeadDim;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          *reinterpret_cast<float2*>(dst + g * kHeadDim + j * 8 + 2 * t) = make_float2(o[j][0], o[j][1]);
          if (kHiRows)
            *reinterpret_cast<float2*>(dst + (g + 8) * kHeadDim + j * 8 + 2 * t) = make_float2(o[j][2], o[j][3]);
        }
        if (t == 0) {
          slot_ml[s * 32 + g] = m0;
          slot_ml[s * 32 + 16 + g] = l0;
          if (kHiRows) {
            slot_ml[s * 32 + g + 8] = m1;
            slot_ml[s * 32 + 16 + g + 8] = l1;
          }
        }
      };
      auto fold_state = [&](int s) {
        const float* src = slots + s * Cfg::kRows * kHeadDim;
#pragma unroll
        for (int half = 0; half < (kHiRows ? 2 : 1); ++half) {
          const int r = g + 8 * half;
          const float ms = slot_ml[s * 32 + r], ls = slot_ml[s * 32 + 16 + r];
          const float mo = half ? m1 : m0, lo = half ? l1 : l0;
          const float M = fmaxf(mo, ms);
          const float fo = (mo == -INFINITY) ? 0.f : fast_exp2(mo - M);
          const float fs = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 v = *reinterpret_cast<const float2*>(src + r * kHeadDim + j * 8 + 2 * t);
            o[j][2 * half] = fo * o[j][2 * half] + fs * v.x;
            o[j][2 * half + 1] = fo * o[j][2 * half + 1] + fs * v.y;
          }
          if (half) {
            m1 = M;
            l1 = fo * lo + fs * ls;
          } else {
            m0 = M;
            l0 = fo * lo + fs * ls;
          }
        }
      };
      if (warp >= 2) {
        if (!first_segment) named_bar_sync(3, 96);
        stage_state(warp - 2);
        named_bar_arrive(1, kThreads);
      } else {
        named_bar_sync(1, kThreads);
        fold_state(warp);  // warp 0 <- warp 2, warp 1 <- warp 3
        if (warp == 1) {
          __syncwarp();  // every lane has read slot 1
          stage_state(1);
          named_bar_arrive(2, 64);
        } else {
          named_bar_sync(2, 64);
          fold_state(1);
#pragma unroll
          for (int half = 0; half < (kHiRows ? 2 : 1); ++half) {
            const int r = g + 8 * half;
            if (r < G) {
              const float l = half ? l1 : l0, m = half ? m1 : m0;
              const bool empty_row = !(l > 0.f);
              const float inv = empty_row ? 0.f : 1.f / l;
              const float lse2 = empty_row ? -INFINITY : m + log2f(l);
              const size_t row = row0 + r;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float x = o[j][2 * half] * inv, y = o[j][2 * half + 1] * inv;
                if (ns == 1)
                  *reinterpret_cast<uint32_t*>(a.out + row * kHeadDim + j * 8 + 2 * t) = pack_bf16x2(x, y);
                else
                  *reinterpret_cast<float2*>(a.o_part + (row * a.max_splits + slot) * kHeadDim + j * 8 + 2 * t) =
                      make_float2(x, y);
              }
              if (t == 0) {
                if (ns == 1) {
                  if (a.out_lse) a.out_lse[row] = lse2 * kLn2;
                } else {
                  a.lse_part[row * a.max_splits + slot] = lse2;
                }
              }
            }
          }
          if (nonempty_from(next + 1) >= 0) named_bar_arrive(3, 96);  // the next mid-stream staging may begin
        }
      }
    } else {
      // ---- The end of the stream: every warp stages its state in the idle
      // ring and all 128 threads merge them.
      cp_async_wait<0>();
      __syncthreads();  // every warp is done with its ring
      float* stg = reinterpret_cast<float*>(ring);       // [kWarps][kRows][128]
      float* mle = stg + kWarps * Cfg::kRows * kHeadDim;  // [2][kWarps][16]: (m, l)
      {
        float* my = stg + warp * Cfg::kRows * kHeadDim;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          *reinterpret_cast<float2*>(my + g * kHeadDim + j * 8 + 2 * t) = make_float2(o[j][0], o[j][1]);
          if (kHiRows)
            *reinterpret_cast<float2*>(my + (g + 8) * kHeadDim + j * 8 + 2 * t) = make_float2(o[j][2], o[j][3]);
        }
        if (t == 0) {
          mle[warp * 16 + g] = m0;
          mle[kWarps * 16 + warp * 16 + g] = l0;
          mle[warp * 16 + g + 8] = m1;
          mle[kWarps * 16 + warp * 16 + g + 8] = l1;
        }
      }
      __syncthreads();
      // Per row: the warps' weights exp2(m_w - M) / sum_w exp2(m_w - M) l_w.
      float* wts = mle + 2 * kWarps * 16;  // [16][kWarps]
      if (threadIdx.x < G) {
        const int r = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mle[w * 16 + r]);
        float f[kWarps], lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = mle[w * 16 + r];
          f[w] = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
          lsum += f[w] * mle[kWarps * 16 + w * 16 + r];
        }
        const bool empty_row = !(lsum > 0.f);
        const float inv = empty_row ? 0.f : 1.f / lsum;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) wts[r * kWarps + w] = f[w] * inv;
        const float lse2 = empty_row ? -INFINITY : M + log2f(lsum);
        const size_t row = row0 + r;
        if (ns == 1) {
          if (a.out_lse) a.out_lse[row] = lse2 * kLn2;
        } else {
          a.lse_part[row * a.max_splits + slot] = lse2;
        }
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < G * (kHeadDim / 4); idx += kThreads) {
        const int r = idx / (kHeadDim / 4), d = (idx % (kHeadDim / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = wts[r * kWarps + w];
          const float4 v = *reinterpret_cast<const float4*>(stg + (w * Cfg::kRows + r) * kHeadDim + d);
          acc.x += f * v.x;
          acc.y += f * v.y;
          acc.z += f * v.z;
          acc.w += f * v.w;
        }
        const size_t row = row0 + r;
        if (ns == 1) {
          uint2 pk;
          pk.x = pack_bf16x2(acc.x, acc.y);
          pk.y = pack_bf16x2(acc.z, acc.w);
          *reinterpret_cast<uint2*>(a.out + row * kHeadDim + d) = pk;
        } else {
          *reinterpret_cast<float4*>(a.o_part + (row * a.max_splits + slot) * kHeadDim + d) = acc;
        }
      }
      break;
    }
    item = next;
    first_segment = false;
  }

  // ---- Publish this CTA's partials: count the CTA in on each split item it
  // holds; the CTA that completes an item's count merges its partials
  // (written by other CTAs: read past L1) and resets the counter. The count is
  // an acquire-release atomic, so the merging CTA needs no further fence, and
  // every item it completes is merged in one pass (their loads in flight together).
  __shared__ int s_nfl[2];  // items listed for merging, per round (two rounds alternate)
  if (threadIdx.x == 0) {
    s_nfl[0] = 0;
    s_nfl[1] = 0;
  }
  __threadfence();  // this thread's partials are visible before any counter moves
  __syncthreads();
  int par = 0;
  for (int it0 = i_first; it0 <= i_last; it0 += kThreads, par ^= 1) {
    const int it = it0 + threadIdx.x;
    if (it <= i_last) {
      const int q0 = prefix[it], q1 = prefix[it + 1];
      if (max(start, q0) < min(end, q1)) {
        const int nsi = (q1 - 1) / per_cta - q0 / per_cta + 1;
        if (nsi > 1) {
          const uint32_t before = atomic_add_acq_rel_gpu(a.arrivals + it, 1u);
          if (before == (uint32_t)nsi - 1) {
            a.arrivals[it] = 0;  // every CTA of the item is in: zero for the next call
            flags[atomicAdd(&s_nfl[par], 1)] = it;
          }
        }
      }
    }
    __syncthreads();
    const int nfl = s_nfl[par];
    if (threadIdx.x == 0) s_nfl[par ^ 1] = 0;  // the next round's list; untouched until the barrier below
    // Elements (item of the list, query row, 4 columns); each thread takes up to
    // kMergeU of them at once and issues every load of a batch of four partials
    // of each at once (one L2 round trip per batch), folding the batches in with
    // an online rescale.
    constexpr int kMergeU = 4;
    const int per_item = G * (kHeadDim / 4);
    const int E = nfl * per_item;
    for (int e0 = threadIdx.x; e0 < E; e0 += kMergeU * kThreads) {
      float M[kMergeU], wsum[kMergeU];
      float4 acc[kMergeU];
      size_t row[kMergeU];
      int d[kMergeU], nsu[kMergeU];
      bool on[kMergeU];
      int nmax = 0;
#pragma unroll
      for (int u = 0; u < kMergeU; ++u) {
        const int e = e0 + u * kThreads;
        on[u] = e < E;
        const int ee = on[u] ? e : e0;
        const int it2 = flags[ee / per_item], r = ee % per_item;
        const int q0 = prefix[it2];
        nsu[u] = (prefix[it2 + 1] - 1) / per_cta - q0 / per_cta + 1;
        row[u] = (size_t)(it2 / H) * Hq + (it2 % H) * G + r / (kHeadDim / 4);
        d[u] = (r % (kHeadDim / 4)) * 4;
        M[u] = -INFINITY;
        wsum[u] = 0.f;
        acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (on[u]) nmax = max(nmax, nsu[u]);
      }
      for (int s0 = 0; s0 < nmax; s0 += 4) {
        float ls[kMergeU][4];
        float4 v[kMergeU][4];
#pragma unroll
        for (int u = 0; u < kMergeU; ++u)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int sl = min(s0 + k, nsu[u] - 1);
            ls[u][k] = __ldcg(a.lse_part + row[u] * a.max_splits + sl);
            v[u][k] = __ldcg(reinterpret_cast<const float4*>(a.o_part + (row[u] * a.max_splits + sl) * kHeadDim + d[u]));
            if (s0 + k >= nsu[u]) ls[u][k] = -INFINITY;  // past the item's last partial: no weight
          }
#pragma unroll
        for (int u = 0; u < kMergeU; ++u) {
          float mn = M[u];
#pragma unroll
          for (int k = 0; k < 4; ++k) mn = fmaxf(mn, ls[u][k]);
          const float sc = (M[u] == -INFINITY) ? 0.f : fast_exp2(M[u] - mn);
          wsum[u] *= sc;
          acc[u].x *= sc;
          acc[u].y *= sc;
          acc[u].z *= sc;
          acc[u].w *= sc;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float fs = (ls[u][k] == -INFINITY) ? 0.f : fast_exp2(ls[u][k] - mn);
            wsum[u] += fs;
            acc[u].x += fs * v[u][k].x;
            acc[u].y += fs * v[u][k].y;
            acc[u].z += fs * v[u][k].z;
            acc[u].w += fs * v[u][k].w;
          }
          M[u] = mn;
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeU; ++u) {
        if (!on[u]) continue;
        const bool empty_row = !(wsum[u] > 0.f);
        const float inv = empty_row ? 0.f : 1.f / wsum[u];
        uint2 pk;
        pk.x = pack_bf16x2(acc[u].x * inv, acc[u].y * inv);
        pk.y = pack_bf16x2(acc[u].z * inv, acc[u].w * inv);
        *reinterpret_cast<uint2*>(a.out + row[u] * kHeadDim + d[u]) = pk;
        if (a.out_lse && d[u] == 0) a.out_lse[row[u]] = empty_row ? -INFINITY : (M[u] + log2f(wsum[u])) * kLn2;
      }
    }
    __syncthreads();
  }
}

size_t decode_smem_bytes(bool hi_rows, int items) {
  return (size_t)(hi_rows ? DecodeSmem<true>::kFixed : DecodeSmem<false>::kFixed) + (size_t)(items + 1) * 4;
}

}  // namespace

DecodePlan plan_gqa_decode(int32_t batch, int32_t num_kv_heads, int32_t sel_stride, int sm_count) {
  (void)batch;
  (void)num_kv_heads;
  DecodePlan p;
  p.pages_per_split = kMinPagesPerCta;
  p.nsplit = (sel_stride + kMinPagesPerCta - 1) / kMinPagesPerCta + 1;  // CTAs one item can span
  p.grid = sm_count * kCtasPerSm;
  return p;
}

size_t gqa_decode_arrivals_offset(int32_t batch, int32_t num_q_heads, int32_t head_dim_v, const DecodePlan& plan) {
  const size_t rows = (size_t)batch * num_q_heads;
  const size_t part = rows * plan.nsplit * ((size_t)head_dim_v + 1) * sizeof(float);
  return (part + 15) & ~size_t(15);
}

size_t gqa_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim_v, const DecodePlan& plan) {
  // partials, then the arrival counters (one per item; items <= rows)
  return gqa_decode_arrivals_offset(batch, num_q_heads, head_dim_v, plan) + (size_t)batch * num_q_heads * sizeof(int32_t);
}

size_t gqa_decode_max_items() {
  const size_t fixed = DecodeSmem<false>::kFixed > DecodeSmem<true>::kFixed ? DecodeSmem<false>::kFixed
                                                                              : DecodeSmem<true>::kFixed;
  return (227 * 1024 - fixed) / 4 - 1;
}

cudaError_t launch_gqa_decode(const KvView& kv, const uint16_t* q, int32_t num_q_heads, const int32_t* block_table,
                              int32_t bt_stride, const int32_t* seq_lens, int32_t batch, const int32_t* sel_pages,
                              const int32_t* sel_counts, int32_t sel_stride, float sm_scale, uint16_t* out,
                              float* out_lse, void* workspace, const DecodePlan& plan, unsigned* err,
                              cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const int H = kv.num_kv_heads;
  DecodeArgs a;
  a.k = kv.k;
  a.v = kv.v;
  a.row_stride_k = kv.row_stride_k;
  a.row_stride_v = kv.row_stride_v;
  a.q = q;
  a.group = num_q_heads / H;
  a.num_kv_heads = H;
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
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o_part = reinterpret_cast<float*>(ws);
  a.lse_part = a.o_part + rows * plan.nsplit * kHeadDim;
  a.arrivals = reinterpret_cast<uint32_t*>(ws + gqa_decode_arrivals_offset(batch, num_q_heads, kHeadDim, plan));
  a.err = err;
  const size_t smem = decode_smem_bytes(a.group > 8, batch * H);
  cudaError_t e;
  if (a.group > 8) {
    e = cudaFuncSetAttribute(gqa_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    {
      const cudaError_t le = launch_pdl(gqa_decode_kernel<true>, dim3(plan.grid), dim3(kThreads), smem, stream, a);
      if (le != cudaSuccess) return le;
    }
  } else {
    e = cudaFuncSetAttribute(gqa_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    {
      const cudaError_t le = launch_pdl(gqa_decode_kernel<false>, dim3(plan.grid), dim3(kThreads), smem, stream, a);
      if (le != cudaSuccess) return le;
    }
  }
  return cudaGetLastError();
}

}  // namespace se
