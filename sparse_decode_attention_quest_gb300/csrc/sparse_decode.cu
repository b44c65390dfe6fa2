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
//    is read from HBM once. The four warps of a CTA take every fourth page of a
//    segment; each warp streams its pages through its own 3-stage ring with
//    16-byte cp.async copies (two pages in flight while it computes a third).
//    The copies write the 128-byte-swizzled layout that makes the ldmatrix
//    reads conflict-free, and token rows at or past the request's length are
//    zero-filled instead of read, so stale cache slots (even NaN) never reach
//    the output;
//  * per page: S = Q K^T and O += P V on the tensor cores with the m16n8k16
//    bf16 MMA (query heads are the 16 rows), an online softmax in the log2
//    domain, fp32 accumulation;
//  * at the end of a segment the four warps' states merge in shared memory. An
//    item held by one CTA writes its output directly; an item spread over
//    several CTAs writes normalised partials (output, log-sum-exp), and the
//    CTA that publishes the item's last partial merges them:
//    o = sum_s exp(lse_s - LSE) o_s. Each CTA counts itself in on a per-item
//    arrival counter in the workspace; the last one resets it to zero, so a
//    workspace that starts zeroed is left zeroed by every call.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kHeadDim = 128;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kHalfBytes = 16 * 64 * 2;     // one 64-column half of a (page, head) block
constexpr int kTileBytes = 2 * kHalfBytes;  // one (page, head) block of K or V
constexpr int kPageBytes = 2 * kTileBytes;  // K block then V block
constexpr int kWarpRing = kStages * kPageBytes;
constexpr int kRingBytes = kWarps * kWarpRing;
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

// Copy one (page, head) K block and V block into a stage; rows >= valid are
// zero-filled without reading the cache.
__device__ __forceinline__ void issue_page(const DecodeArgs& a, uint32_t stage, int phys, int h, int valid,
                                           int lane) {
  const size_t blk = ((size_t)phys * a.num_kv_heads + h) * kPageSize;
  const uint16_t* kp = a.k + blk * a.row_stride_k;
  const uint16_t* vp = a.v + blk * a.row_stride_v;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int c = lane + 32 * it;  // 16-byte chunk 0..255 of the 16 x 256-byte block
    const int r = c >> 4, q16 = c & 15;
    const uint32_t off = (uint32_t)(q16 >> 3) * kHalfBytes + swz128(r, q16 & 7);
    const bool in = r < valid;
    const uint32_t bytes = in ? 16u : 0u;
    cp_async16(stage + off, kp + (size_t)(in ? r : 0) * a.row_stride_k + q16 * 8, bytes);
    cp_async16(stage + kTileBytes + off, vp + (size_t)(in ? r : 0) * a.row_stride_v + q16 * 8, bytes);
  }
}

template <bool kHiRows>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) gqa_decode_kernel(const DecodeArgs a) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* red_ml = reinterpret_cast<float*>(ring + kRingBytes);       // [2][kWarps][16]: (m, l) per warp and row
  int* prefix = reinterpret_cast<int*>(red_ml + 2 * kWarps * 16);    // [items + 1]
  __shared__ int s_last;  // this CTA published the last partial of the segment's item
  const int H = a.num_kv_heads, G = a.group, Hq = H * G;
  const int items = a.batch * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Selected pages per item, then an exclusive prefix.
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

  const uint32_t wring = smem_addr(ring) + warp * kWarpRing;
  // This warp's state at the end of a segment waits for the merge in the last
  // stage of its ring (16 rows x 128 fp32 = one stage); the next segment's
  // prologue only fills the other stages, so its copies are in flight while
  // the CTA merges the previous segment.
  float* my_red = reinterpret_cast<float*>(ring + warp * kWarpRing + (kStages - 1) * kPageBytes);
  const int g = lane >> 2, t = lane & 3;
  const int i_first = find_item(prefix, items, start);
  const int i_last = find_item(prefix, items, end - 1);
  auto nonempty_from = [&](int it) {
    for (; it <= i_last; ++it)
      if (max(start, prefix[it]) < min(end, prefix[it + 1])) return it;
    return -1;
  };

  // Per-segment values (the segment = this CTA's pages of one item).
  int item = nonempty_from(i_first);
  int b = 0, h = 0, n_b = 0, L = 0, np = 0;
  const int32_t* sel_row = nullptr;
  const int32_t* bt_row = nullptr;
  int base = 0, ph_cur = 0, va_cur = 0, ph_nxt = 0, va_nxt = 0;
  uint32_t qa[8][4];
  // Metadata of page k of this warp (physical page, valid tokens), one page per lane.
  auto meta = [&](int k, int& phys, int& valid) {
    phys = 0;
    valid = 0;
    if (k < np) {
      const int logical = sel_row[kWarps * k];
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
  // Two batches of 32 pages: [base, base + 32) in *_cur, the next 32 in *_nxt.
  auto lookup = [&](int k, int& phys, int& valid) {
    const int pc = __shfl_sync(0xffffffffu, ph_cur, k & 31), vc = __shfl_sync(0xffffffffu, va_cur, k & 31);
    const int pn = __shfl_sync(0xffffffffu, ph_nxt, k & 31), vn = __shfl_sync(0xffffffffu, va_nxt, k & 31);
    const bool in_cur = k < base + 32;
    phys = in_cur ? pc : pn;
    valid = in_cur ? vc : vn;
  };
  // Opens segment `it`: its values, metadata windows, the first kStages - 1
  // pages in flight (stages 0 .. kStages - 2) and the query fragments.
  auto open_segment = [&](int it) {
    const int p0 = prefix[it];
    const int lo = max(start, p0) - p0, hi = min(end, prefix[it + 1]) - p0;  // item-local pages
    b = it / H;
    h = it % H;
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
    // This warp's pages of the segment: lo + warp + kWarps k, k < np.
    np = (hi - lo > warp) ? (hi - lo - warp + kWarps - 1) / kWarps : 0;
    sel_row = a.sel + (size_t)it * a.sel_stride + lo + warp;
    bt_row = a.block_table + (size_t)b * a.bt_stride;
    base = 0;
    meta(lane, ph_cur, va_cur);
    meta(lane + 32, ph_nxt, va_nxt);
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
      if (k < np) {
        int ph, va;
        lookup(k, ph, va);
        issue_page(a, wring + (k % kStages) * kPageBytes, ph, h, va, lane);
      }
      cp_async_commit();
    }
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
  };

  open_segment(item);
  while (true) {
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    for (int k = 0; k < np; ++k) {
      const int kn = k + kStages - 1;
      if (kn == base + 32 + 32) {  // the next batch is needed by the copy ahead: rotate
        base += 32;
        ph_cur = ph_nxt;
        va_cur = va_nxt;
        meta(base + 32 + lane, ph_nxt, va_nxt);
      }
      if (kn < np) {
        int ph, va;
        lookup(kn, ph, va);
        issue_page(a, wring + (kn % kStages) * kPageBytes, ph, h, va, lane);
      }
      cp_async_commit();
      cp_async_wait<kStages - 1>();  // page k has landed (this thread's copies)
      __syncwarp();                  // ... and every lane's
      int ph_k, valid;
      lookup(k, ph_k, valid);
      (void)ph_k;
      if (valid > 0) {
        const uint32_t kt = wring + (k % kStages) * kPageBytes;
        const uint32_t vt = kt + kTileBytes;
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
        const uint32_t pa0 = pack_bf16x2(p[0][0], p[0][1]);
        const uint32_t pa1 = pack_bf16x2(p[0][2], p[0][3]);
        const uint32_t pa2 = pack_bf16x2(p[1][0], p[1][1]);
        const uint32_t pa3 = pack_bf16x2(p[1][2], p[1][3]);
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
      __syncwarp();  // every lane is done with this stage before it is refilled
    }
    cp_async_wait<0>();  // every copy of this warp has landed: the ring is idle
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (t == 0) {
      red_ml[warp * 16 + g] = m0;
      red_ml[kWarps * 16 + warp * 16 + g] = l0;
      red_ml[warp * 16 + g + 8] = m1;
      red_ml[kWarps * 16 + warp * 16 + g + 8] = l1;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      *reinterpret_cast<float2*>(my_red + g * kHeadDim + j * 8 + 2 * t) = make_float2(o[j][0], o[j][1]);
      *reinterpret_cast<float2*>(my_red + (g + 8) * kHeadDim + j * 8 + 2 * t) = make_float2(o[j][2], o[j][3]);
    }
    // The segment's values are needed by the merge after the next one opens.
    const int cur = item, cur_b = b, cur_h = h;
    const int next = nonempty_from(item + 1);
    if (next >= 0) open_segment(next);
    __syncthreads();  // every warp's state is staged

    // ---- merge the warps' states of segment `cur`
    const int p0 = prefix[cur];
    const int cnt = prefix[cur + 1] - p0;
    const int first_cta = p0 / per_cta;
    const int ns = (p0 + cnt - 1) / per_cta - first_cta + 1;
    const int slot = blockIdx.x - first_cta;
    for (int idx = threadIdx.x; idx < G * kHeadDim; idx += kThreads) {
      const int r = idx / kHeadDim, d = idx % kHeadDim;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_ml[w * 16 + r]);
      float lsum = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = red_ml[w * 16 + r];
        const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
        lsum += f * red_ml[kWarps * 16 + w * 16 + r];
        const float* wred = reinterpret_cast<const float*>(ring + w * kWarpRing + (kStages - 1) * kPageBytes);
        acc += f * wred[r * kHeadDim + d];
      }
      const bool empty_row = !(lsum > 0.f);
      const float val = empty_row ? 0.f : acc / lsum;
      const float lse2 = empty_row ? -INFINITY : M + log2f(lsum);
      const size_t row = (size_t)cur_b * Hq + cur_h * G + r;
      if (ns == 1) {
        a.out[row * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
        if (a.out_lse && d == 0) a.out_lse[row] = lse2 * kLn2;
      } else {
        a.o_part[(row * a.max_splits + slot) * kHeadDim + d] = val;
        if (d == 0) a.lse_part[row * a.max_splits + slot] = lse2;
      }
    }
    if (ns > 1) __threadfence();  // this CTA's partial is visible before it counts itself in
    __syncthreads();  // the staged states are read: the last stages may be refilled
    if (ns > 1) {
      if (threadIdx.x == 0) {
        const uint32_t before = atomicAdd(a.arrivals + cur, 1u);
        const bool last = before == (uint32_t)ns - 1;
        if (last) a.arrivals[cur] = 0;  // every CTA of the item is in: zero for the next call
        s_last = last ? 1 : 0;
      }
      __syncthreads();
      if (s_last) {
        // The item's last partial: merge all ns of them (written by other CTAs:
        // read past L1).
        __threadfence();
        for (int idx = threadIdx.x; idx < G * (kHeadDim / 4); idx += kThreads) {
          const int r = idx / (kHeadDim / 4), d = (idx % (kHeadDim / 4)) * 4;
          const size_t row = (size_t)cur_b * Hq + cur_h * G + r;
          const float* lp = a.lse_part + row * a.max_splits;
          float M = -INFINITY;
          for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(lp + s));
          float wsum = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int s = 0; s < ns; ++s) {
            const float ls = __ldcg(lp + s);
            if (ls == -INFINITY) continue;
            const float f = fast_exp2(ls - M);
            wsum += f;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(a.o_part + (row * a.max_splits + s) * kHeadDim + d));
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
          }
          const bool empty_row = !(wsum > 0.f);
          const float inv = empty_row ? 0.f : 1.f / wsum;
          uint2 pk;
          pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
          *reinterpret_cast<uint2*>(a.out + row * kHeadDim + d) = pk;
          if (a.out_lse && d == 0) a.out_lse[row] = empty_row ? -INFINITY : (M + log2f(wsum)) * kLn2;
        }
      }
    }
    if (next < 0) break;
    item = next;
  }
}

size_t decode_smem_bytes(int items) {
  return (size_t)kRingBytes + 1024 + 2 * kWarps * 16 * 4 + (size_t)(items + 1) * 4;
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

size_t gqa_decode_max_items() { return (227 * 1024 - (size_t)kRingBytes - 1024 - 2 * kWarps * 16 * 4) / 4 - 1; }

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
  const size_t smem = decode_smem_bytes(batch * H);
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
