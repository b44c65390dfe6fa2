// Sparse paged flash-decode over the Quest-selected pages (SparseEngine:
// Sparse-First Inference Engine, Figure 2 caption: attention execution reads
// the method's view of the cache; Table 7: the logit z and weight alpha, the
// history includes the current token).
//
// GQA path (head_dim = head_dim_v = 128, 1..16 query heads per KV head):
//  * one CTA per (request, KV head, split of the selected pages) serves the whole
//    query group, so every selected (page, head) block is read from HBM once;
//  * a producer warp streams each page's K and V blocks (4 KB each) into a
//    12-stage shared-memory ring with tiled TMA copies (two 64-column boxes per
//    block, 128-byte swizzle so the ldmatrix reads below are conflict-free),
//    completion tracked by mbarriers;
//  * four consumer warps each take every fourth page of the split and run an
//    online softmax: S = Q K^T and O += P V on the tensor cores with the
//    m16n8k16 bf16 MMA (query heads are the 16 rows, G <= 16), fp32 accumulate;
//  * the warps' states merge in shared memory; a split writes its normalised
//    partial output and log-sum-exp, and combine_kernel merges the splits
//    (o = sum_s exp(lse_s - LSE) o_s). With one split the CTA writes the output.
// Tokens at positions >= seq_len on a request's last page are masked, and their
// value rows are zeroed in shared memory, so stale cache contents (even NaN)
// never reach the output.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kHeadDim = 128;
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 12;
constexpr int kHalfBytes = 16 * 64 * 2;     // one 64-column box of a (page, head) block
constexpr int kTileBytes = 2 * kHalfBytes;  // one (page, head) block of K or V
constexpr int kStageBytes = 2 * kTileBytes; // K block then V block
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kDecodeSmem = kRingBytes + kStages * 8 * 2 + kStages * 4 + 1024;  // + barriers, meta, alignment
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeArgs {
  const uint16_t* q;
  int32_t group;
  int32_t num_kv_heads;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* sel;
  const int32_t* sel_counts;
  int32_t sel_stride;
  int32_t pages_per_split;
  int32_t nsplit;
  int32_t num_pages;
  float scale_log2;  // sm_scale * log2(e)
  uint16_t* out;
  float* out_lse;
  float* o_part;     // [B][Hq][nsplit][128]
  float* lse_part;   // [B][Hq][nsplit], log2 domain
  unsigned* err;
};

template <bool kHiRows>
__global__ void __launch_bounds__(kDecodeThreads, 2) gqa_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                      const __grid_constant__ CUtensorMap vmap,
                                                                      const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kRingBytes);
  uint64_t* empty = full + kStages;
  int* meta = reinterpret_cast<int*>(empty + kStages);

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int H = a.num_kv_heads, G = a.group, Hq = H * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int L = a.seq_lens[b];
  if (L < 0) {
    if (threadIdx.x == 0) raise_error(a.err, SE_DEVERR_LENGTH);
    L = 0;
  }
  int n_b = (L + kPageSize - 1) / kPageSize;
  if (n_b > a.bt_stride) {  // a length beyond the block table: clip to it
    if (threadIdx.x == 0) raise_error(a.err, SE_DEVERR_LENGTH);
    n_b = a.bt_stride;
    L = n_b * kPageSize;
  }
  int cnt_total = a.sel_counts[b * H + h];
  if (cnt_total < 0 || cnt_total > a.sel_stride) {
    if (threadIdx.x == 0 && split == 0) raise_error(a.err, SE_DEVERR_LENGTH);
    cnt_total = cnt_total < 0 ? 0 : a.sel_stride;
  }
  const int start = split * a.pages_per_split;
  const int cnt = min(a.pages_per_split, cnt_total - start);
  if (cnt <= 0) {
    if (split == 0 && a.nsplit == 1) {  // nothing selected: zero output, lse = -inf
      for (int i = threadIdx.x; i < G * kHeadDim; i += kDecodeThreads) {
        a.out[((size_t)b * Hq + h * G + i / kHeadDim) * kHeadDim + i % kHeadDim] = 0;
        if (a.out_lse && i % kHeadDim == 0) a.out_lse[(size_t)b * Hq + h * G + i / kHeadDim] = -INFINITY;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // Consumer state (rows g and g + 8 of the MMA tile; unused by the producer warp).
  const int g = lane >> 2, t = lane & 3;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
    }
    const uint64_t policy = l2_evict_first_policy();
    const int32_t* sel_row = a.sel + ((size_t)b * H + h) * a.sel_stride + start;
    const int32_t* bt = a.block_table + (size_t)b * a.bt_stride;
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < cnt && ok; base += 32) {
      int phys = -1, valid = 0;
      if (base + lane < cnt) {
        const int logical = sel_row[base + lane];
        if (logical >= 0 && logical < n_b) {
          phys = bt[logical];
          valid = min(kPageSize, L - logical * kPageSize);
        }
      }
      const int m = min(32, cnt - base);
      for (int j = 0; j < m; ++j) {
        const int ph = __shfl_sync(0xffffffffu, phys, j);
        const int v = __shfl_sync(0xffffffffu, valid, j);
        const int i = base + j, s = i % kStages;
        if (lane == 0) {
          if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1)) {
            raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
            ok = false;
          } else if (v <= 0 || ph < 0 || ph >= a.num_pages) {
            raise_error(a.err, v <= 0 ? SE_DEVERR_LENGTH : SE_DEVERR_PAGE_RANGE);
            meta[s] = 0;
            mbar_arrive(&full[s]);
            ++issued;
          } else {
            meta[s] = v;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            const int y = (ph * H + h) * kPageSize;
            uint8_t* st = ring + s * kStageBytes;
            tma_load_2d(st, &kmap, 0, y, &full[s], policy);
            tma_load_2d(st + kHalfBytes, &kmap, 64, y, &full[s], policy);
            tma_load_2d(st + kTileBytes, &vmap, 0, y, &full[s], policy);
            tma_load_2d(st + kTileBytes + kHalfBytes, &vmap, 64, y, &full[s], policy);
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        if (!ok) break;
      }
    }
    // Drain: every copy this CTA issued has landed before any thread leaves.
    if (lane == 0) {
      for (int i = max(0, issued - kStages); i < issued; ++i) {
        if (!mbar_wait(&full[i % kStages], (i / kStages) & 1)) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Query fragments (A operand, rows = query heads of the group, zero past G).
    uint32_t qa[8][4];
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
    const uint32_t ring_addr = smem_addr(ring);
    for (int i = warp; i < cnt; i += kConsumerWarps) {
      const int s = i % kStages;
      if (!mbar_wait(&full[s], (i / kStages) & 1)) {
        if (lane == 0) raise_error(a.err, SE_DEVERR_WAIT_TIMEOUT);
        break;
      }
      const int valid = meta[s];
      if (valid > 0) {
        const uint32_t kt = ring_addr + s * kStageBytes;
        const uint32_t vt = kt + kTileBytes;
        if (valid < kPageSize) {
          // Zero value rows past the length in both 64-column boxes.
          uint4* vrow = reinterpret_cast<uint4*>(ring + s * kStageBytes + kTileBytes);
          const int nchunk = (kPageSize - valid) * 8;  // 16-byte chunks per box
          for (int c = lane; c < 2 * nchunk; c += 32) {
            const int box = c / nchunk, r = c % nchunk;
            vrow[box * (kHalfBytes / 16) + valid * 8 + r] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        // S = Q K^T : two n-tiles of 8 tokens, 8 k-steps of 16 dims.
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = (lane & 7) + ((lane >> 4) << 3);
        const int ksub = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t addr = kt + (ks >> 2) * kHalfBytes + swz128(krow, ((ks & 3) << 1) + ksub);
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4(r0, r1, r2, r3, addr);
          mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r0, r1);
          mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r2, r3);
        }
        // Online softmax in the log2 domain.
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + 2 * t + (e & 1);
            sc[nt][e] = tok < valid ? sc[nt][e] * a.scale_log2 : -INFINITY;
          }
        }
        float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float c0 = exp2f(m0 - n0), c1 = exp2f(m1 - n1);
        m0 = n0;
        m1 = n1;
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          p[nt][0] = exp2f(sc[nt][0] - n0);
          p[nt][1] = exp2f(sc[nt][1] - n0);
          p[nt][2] = exp2f(sc[nt][2] - n1);
          p[nt][3] = exp2f(sc[nt][3] - n1);
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
        // O += P V : 16 n-tiles of 8 dims, one k-step of 16 tokens.
        const int vtok = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int vsub = lane >> 4;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int chunk = 2 * j + vsub;  // 16-byte chunk of 8 dims, 0..15
          const uint32_t addr = vt + (chunk >> 3) * kHalfBytes + swz128(vtok, chunk & 7);
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(r0, r1, r2, r3, addr);
          mma_bf16_16816(o[2 * j], pa0, pa1, pa2, pa3, r0, r1);
          mma_bf16_16816(o[2 * j + 1], pa0, pa1, pa2, pa3, r2, r3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }

  __syncthreads();  // every warp is done with the ring (all copies drained): reuse it for the merge
  if (warp < kConsumerWarps) {
    float* red_m = reinterpret_cast<float*>(ring);         // [4][16]
    float* red_l = red_m + kConsumerWarps * 16;            // [4][16]
    float* red_o = red_l + kConsumerWarps * 16;            // [4][16][128]
    if (t == 0) {
      red_m[warp * 16 + g] = m0;
      red_l[warp * 16 + g] = l0;
      red_m[warp * 16 + g + 8] = m1;
      red_l[warp * 16 + g + 8] = l1;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float* r0p = red_o + ((size_t)warp * 16 + g) * kHeadDim + j * 8 + 2 * t;
      float* r1p = red_o + ((size_t)warp * 16 + g + 8) * kHeadDim + j * 8 + 2 * t;
      *reinterpret_cast<float2*>(r0p) = make_float2(o[j][0], o[j][1]);
      *reinterpret_cast<float2*>(r1p) = make_float2(o[j][2], o[j][3]);
    }
  }
  __syncthreads();  // merge inputs written

  const float* red_m = reinterpret_cast<const float*>(ring);
  const float* red_l = red_m + kConsumerWarps * 16;
  const float* red_o = red_l + kConsumerWarps * 16;
  for (int idx = threadIdx.x; idx < G * kHeadDim; idx += kDecodeThreads) {
    const int r = idx / kHeadDim, d = idx % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * 16 + r]);
    float lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = red_m[w * 16 + r];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      lsum += f * red_l[w * 16 + r];
      acc += f * red_o[((size_t)w * 16 + r) * kHeadDim + d];
    }
    const bool empty_row = !(lsum > 0.f);
    const float val = empty_row ? 0.f : acc / lsum;
    const float lse2 = empty_row ? -INFINITY : M + log2f(lsum);
    const size_t row = (size_t)b * Hq + h * G + r;
    if (a.nsplit == 1) {
      a.out[row * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
      if (a.out_lse && d == 0) a.out_lse[row] = lse2 * kLn2;
    } else {
      a.o_part[(row * a.nsplit + split) * kHeadDim + d] = val;
      if (d == 0) a.lse_part[row * a.nsplit + split] = lse2;
    }
  }
}

// Merge the split partials of one (request, query head) per warp.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ o_part,
                                                      const float* __restrict__ lse_part,
                                                      const int32_t* __restrict__ sel_counts, int32_t batch,
                                                      int32_t Hq, int32_t group, int32_t sel_stride,
                                                      int32_t pages_per_split, int32_t nsplit, int32_t Dv,
                                                      uint16_t* __restrict__ out, float* __restrict__ out_lse) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= batch * Hq) return;
  const int lane = threadIdx.x & 31;
  const int b = row / Hq, h = (row % Hq) / group, H = Hq / group;
  int cnt = sel_counts[b * H + h];
  cnt = cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);
  const int ns = min(nsplit, (cnt + pages_per_split - 1) / pages_per_split);
  const float* lp = lse_part + (size_t)row * nsplit;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, lp[s]);
  float wsum = 0.f;
  for (int s = 0; s < ns; ++s) wsum += (lp[s] == -INFINITY) ? 0.f : exp2f(lp[s] - M);
  const bool empty_row = !(wsum > 0.f);
  for (int d = lane * 4; d < Dv; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ns; ++s) {
      if (lp[s] == -INFINITY) continue;
      const float f = exp2f(lp[s] - M);
      const float4 v = *reinterpret_cast<const float4*>(o_part + ((size_t)row * nsplit + s) * Dv + d);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    const float inv = empty_row ? 0.f : 1.f / wsum;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out + (size_t)row * Dv + d) = pk;
  }
  if (out_lse && lane == 0) out_lse[row] = empty_row ? -INFINITY : (M + log2f(wsum)) * kLn2;
}

}  // namespace

DecodePlan plan_gqa_decode(int32_t batch, int32_t num_kv_heads, int32_t sel_stride, int sm_count) {
  const long long items = (long long)batch * num_kv_heads;
  const long long target = (long long)sm_count * 2 * 4;  // about 4 waves of 2 CTAs per SM
  long long ns = items > 0 ? (target + items - 1) / items : 1;
  if (ns < 1) ns = 1;
  if (ns > sel_stride) ns = sel_stride;
  int pps = (int)((sel_stride + ns - 1) / ns);
  pps = ((pps + 3) / 4) * 4;
  if (pps < 8) pps = 8;
  DecodePlan p;
  p.pages_per_split = pps;
  p.nsplit = (sel_stride + pps - 1) / pps;
  if (p.nsplit < 1) p.nsplit = 1;
  return p;
}

size_t gqa_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim_v, const DecodePlan& plan) {
  if (plan.nsplit <= 1) return 0;
  return (size_t)batch * num_q_heads * plan.nsplit * ((size_t)head_dim_v + 1) * sizeof(float);
}

cudaError_t launch_gqa_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const KvView& kv,
                              const uint16_t* q, int32_t num_q_heads, const int32_t* block_table,
                              int32_t bt_stride, const int32_t* seq_lens, int32_t batch,
                              const int32_t* sel_pages, const int32_t* sel_counts, int32_t sel_stride,
                              float sm_scale, uint16_t* out, float* out_lse, void* workspace,
                              const DecodePlan& plan, unsigned* err, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const int H = kv.num_kv_heads;
  DecodeArgs a;
  a.q = q;
  a.group = num_q_heads / H;
  a.num_kv_heads = H;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.sel = sel_pages;
  a.sel_counts = sel_counts;
  a.sel_stride = sel_stride;
  a.pages_per_split = plan.pages_per_split;
  a.nsplit = plan.nsplit;
  a.num_pages = kv.num_pages;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = out;
  a.out_lse = out_lse;
  a.o_part = reinterpret_cast<float*>(workspace);
  a.lse_part = a.o_part ? a.o_part + (size_t)batch * num_q_heads * plan.nsplit * kHeadDim : nullptr;
  a.err = err;
  dim3 grid(plan.nsplit, H, batch);
  cudaError_t e;
  if (a.group > 8) {
    e = cudaFuncSetAttribute(gqa_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecodeSmem);
    if (e != cudaSuccess) return e;
    gqa_decode_kernel<true><<<grid, kDecodeThreads, kDecodeSmem, stream>>>(kmap, vmap, a);
  } else {
    e = cudaFuncSetAttribute(gqa_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecodeSmem);
    if (e != cudaSuccess) return e;
    gqa_decode_kernel<false><<<grid, kDecodeThreads, kDecodeSmem, stream>>>(kmap, vmap, a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || plan.nsplit == 1) return e;
  const int rows = batch * num_q_heads;
  combine_kernel<<<(rows + 3) / 4, 128, 0, stream>>>(a.o_part, a.lse_part, sel_counts, batch, num_q_heads, a.group,
                                                    sel_stride, plan.pages_per_split, plan.nsplit, kHeadDim, out,
                                                    out_lse);
  return cudaGetLastError();
}

}  // namespace se
