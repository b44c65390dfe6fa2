// Sparse paged decode over a latent (MLA-style) cache (SparseEngine:
// Sparse-First Inference Engine, Figure 5 caption: GLM-4.7-Flash, an MLA model,
// decoding at 32K/128K; Table 7: logit z and weight alpha over the history).
//
// One cache row per token holds 576 dims (512 latent + 64 RoPE) and serves as
// the key; its first 512 dims are the value. All 16 x HG query heads share the
// one KV head, so every selected page (16 rows x 1152 bytes) is read once and
// used by all heads.
//
//  * Work split as in the GQA decode: the selected pages of all requests form
//    one flattened range and every CTA takes an equal slice (>= 16 pages).
//  * 2 x HG warps: warp (hg, dh) owns query heads 16 hg .. 16 hg + 15 and output
//    dims 256 dh .. 256 dh + 255, so its output accumulator is 128 registers. Its
//    query fragments cover dims 288 dh .. 288 dh + 287 (72 registers); the two
//    warps of a head group add their partial logits through shared memory, so
//    both see the full 576-dim logits and run the same online softmax.
//  * A CTA-wide 8-stage ring of pages, filled with 16-byte cp.async copies into
//    a layout of nine 64-dim chunks per page, 128-byte swizzled; rows at or past
//    the request's length are zero-filled, never read. Page metadata (physical
//    page, valid rows) sits in lanes, two windows of 32 pages per warp, loaded
//    25 pages before the copies need it.
//  * S = Q K^T and O += P V use the m16n8k16 bf16 MMA with fp32 accumulation.
#include "se_ptx.cuh"

namespace se {
namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kChunks = kD / 64;                      // 9 chunks of 64 dims
constexpr int kChunkBytes = kPageSize * 128;          // 16 rows x 128 bytes
constexpr int kPageBytes = kChunks * kChunkBytes;     // 18 KB
constexpr int kStages = 8;
constexpr int kRingBytes = kStages * kPageBytes;
constexpr int kMinPagesPerCta = 16;
constexpr int kKStepsPerHalf = kD / 2 / 16;           // 18
constexpr float kLn2 = 0.6931471805599453f;

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
  float* o_part;     // [B * Hq][max_splits][512]
  float* lse_part;   // [B * Hq][max_splits], log2 domain
  int32_t* item_ns;  // [B]
  unsigned* err;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ int find_item(const int* prefix, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Barrier of the two warps of head group hg (named barriers 1 .. HG).
__device__ __forceinline__ void pair_barrier(int hg) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + hg) : "memory");
}

template <int HG>
__global__ void __launch_bounds__(64 * HG, 1) mla_decode_kernel(const MlaArgs a) {
  pdl_enter();
  constexpr int kThreads = 64 * HG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xbuf = reinterpret_cast<float*>(ring + kRingBytes);  // [2 parity][HG][2 dh][32 lanes][8]
  int* prefix = reinterpret_cast<int*>(xbuf + 2 * HG * 2 * 32 * 8);
  const int items = a.batch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hg = warp >> 1, dh = warp & 1;
  const int g = lane >> 2, t = lane & 3;

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

  const uint32_t ring_addr = smem_addr(ring);
  const int i_first = find_item(prefix, items, start);
  const int i_last = find_item(prefix, items, end - 1);
  int page_ctr = 0;  // pages processed by this CTA (exchange buffer parity)
  for (int item = i_first; item <= i_last; ++item) {
    const int p0 = prefix[item];
    const int lo = max(start, p0) - p0, hi = min(end, prefix[item + 1]) - p0;
    if (lo >= hi) continue;
    const int b = item;
    int L = a.seq_lens[b];
    if (L < 0) {
      if (threadIdx.x == 0) raise_error(a.err, SE_DEVERR_LENGTH);
      L = 0;
    }
    int n_b = (L + kPageSize - 1) / kPageSize;
    if (n_b > a.bt_stride) {
      if (threadIdx.x == 0) raise_error(a.err, SE_DEVERR_LENGTH);
      n_b = a.bt_stride;
      L = n_b * kPageSize;
    }
    const int np = hi - lo;
    const int32_t* sel_row = a.sel + (size_t)item * a.sel_stride + lo;
    const int32_t* bt_row = a.block_table + (size_t)b * a.bt_stride;
    // Metadata of page k (physical page, valid rows; 0 rows: skip), one page per
    // lane: every warp holds pages [base, base + 32) and [base + 32, base + 64).
    auto meta = [&](int k, int& phys, int& valid) {
      phys = 0;
      valid = 0;
      if (k < np) {
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
    int base = 0, ph_cur, va_cur, ph_nxt, va_nxt;
    meta(lane, ph_cur, va_cur);
    meta(lane + 32, ph_nxt, va_nxt);
    auto lookup = [&](int k, int& phys, int& valid) {
      const int pc = __shfl_sync(0xffffffffu, ph_cur, k & 31), vc = __shfl_sync(0xffffffffu, va_cur, k & 31);
      const int pn = __shfl_sync(0xffffffffu, ph_nxt, k & 31), vn = __shfl_sync(0xffffffffu, va_nxt, k & 31);
      const bool in_cur = k < base + 32;
      phys = in_cur ? pc : pn;
      valid = in_cur ? vc : vn;
    };
    auto issue = [&](int k) {
      int phys, valid;
      lookup(k, phys, valid);
      const uint32_t st = ring_addr + (k % kStages) * kPageBytes;
      const uint16_t* src = a.kv + (size_t)phys * kPageSize * a.row_stride;
      for (int c = threadIdx.x; c < kPageSize * kChunks * 8; c += kThreads) {  // 1152 16-byte pieces
        const int r = c / (kChunks * 8), q = c % (kChunks * 8);
        const bool in = r < valid;
        cp_async16(st + (q >> 3) * kChunkBytes + swz128(r, q & 7),
                   src + (size_t)(in ? r : 0) * a.row_stride + q * 8, in ? 16u : 0u);
      }
    };
#pragma unroll 1
    for (int k = 0; k < kStages - 1; ++k) {
      if (k < np) issue(k);
      cp_async_commit();
    }
    // Query fragments: heads 16 hg + {g, g + 8}, k-steps over dims 288 dh ..
    uint32_t qa[kKStepsPerHalf][4];
    {
      const uint16_t* q0 = a.q + ((size_t)b * a.Hq + hg * 16 + g) * kD;
      const uint16_t* q1 = q0 + 8 * kD;
#pragma unroll
      for (int ks = 0; ks < kKStepsPerHalf; ++ks) {
        const int c = (dh * kKStepsPerHalf + ks) * 16 + 2 * t;
        qa[ks][0] = *reinterpret_cast<const uint32_t*>(q0 + c);
        qa[ks][2] = *reinterpret_cast<const uint32_t*>(q0 + c + 8);
        qa[ks][1] = *reinterpret_cast<const uint32_t*>(q1 + c);
        qa[ks][3] = *reinterpret_cast<const uint32_t*>(q1 + c + 8);
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[32][4];
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    const int krow = (lane & 7) + ((lane >> 4) << 3), ksub = (lane >> 3) & 1;
    const int vtok = (lane & 7) + (((lane >> 3) & 1) << 3), vsub = lane >> 4;

    for (int k = 0; k < np; ++k, ++page_ctr) {
      // Page k has left the first window: rotate. The window loaded here is
      // first needed 25 pages later (the copies run kStages - 1 pages ahead).
      if (k == base + 32) {
        base += 32;
        ph_cur = ph_nxt;
        va_cur = va_nxt;
        meta(base + 32 + lane, ph_nxt, va_nxt);
      }
      if (k + kStages - 1 < np) issue(k + kStages - 1);
      cp_async_commit();
      cp_async_wait<kStages - 1>();
      __syncthreads();  // page k is in shared memory (every thread's copies)
      int phys_k, valid;
      lookup(k, phys_k, valid);
      (void)phys_k;
      if (valid > 0) {
        const uint32_t st = ring_addr + (k % kStages) * kPageBytes;
        // Partial S over this warp's 288 dims.
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < kKStepsPerHalf; ++ks) {
          const int d0 = (dh * kKStepsPerHalf + ks) * 16;
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4(r0, r1, r2, r3, st + (d0 >> 6) * kChunkBytes + swz128(krow, ((d0 & 63) >> 3) + ksub));
          mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r0, r1);
          mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r2, r3);
        }
        // Add the partner warp's partial (same head group, other half of the dims).
        float* mine = xbuf + ((((page_ctr & 1) * HG + hg) * 2 + dh) * 32 + lane) * 8;
        const float* other = xbuf + ((((page_ctr & 1) * HG + hg) * 2 + (dh ^ 1)) * 32 + lane) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) mine[e] = sc[e >> 2][e & 3];
        pair_barrier(hg);
#pragma unroll
        for (int e = 0; e < 8; ++e) sc[e >> 2][e & 3] += other[e];
        // Online softmax in the log2 domain (identical in both warps of the pair).
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
        for (int j = 0; j < 32; ++j) {
          o[j][0] *= c0;
          o[j][1] *= c0;
          o[j][2] *= c1;
          o[j][3] *= c1;
        }
        const uint32_t pa0 = pack_bf16x2(p[0][0], p[0][1]);
        const uint32_t pa1 = pack_bf16x2(p[0][2], p[0][3]);
        const uint32_t pa2 = pack_bf16x2(p[1][0], p[1][1]);
        const uint32_t pa3 = pack_bf16x2(p[1][2], p[1][3]);
        // O[:, 256 dh + 16 j ..] += P V (value = first 512 dims of the row).
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n0d = dh * 256 + 16 * j;
          const int q = ((n0d & 63) >> 3) + vsub;
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(r0, r1, r2, r3, st + (n0d >> 6) * kChunkBytes + swz128(vtok, q));
          mma_bf16_16816(o[2 * j], pa0, pa1, pa2, pa3, r0, r1);
          mma_bf16_16816(o[2 * j + 1], pa0, pa1, pa2, pa3, r2, r3);
        }
      }
      __syncthreads();  // stage k % kStages is refilled next
    }
    cp_async_wait<0>();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    // Output rows of this warp: heads 16 hg + g (m0, l0) and + g + 8 (m1, l1).
    const int cnt = prefix[item + 1] - p0;
    const int first_cta = p0 / per_cta;
    const int ns = (p0 + cnt - 1) / per_cta - first_cta + 1;
    const int slot = blockIdx.x - first_cta;
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const size_t row0 = (size_t)b * a.Hq + hg * 16 + g, row1 = row0 + 8;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int d = dh * 256 + 8 * j + 2 * t;
      if (ns == 1) {
        *reinterpret_cast<uint32_t*>(a.out + row0 * kDv + d) = pack_bf16x2(o[j][0] * inv0, o[j][1] * inv0);
        *reinterpret_cast<uint32_t*>(a.out + row1 * kDv + d) = pack_bf16x2(o[j][2] * inv1, o[j][3] * inv1);
      } else {
        *reinterpret_cast<float2*>(a.o_part + (row0 * a.max_splits + slot) * kDv + d) =
            make_float2(o[j][0] * inv0, o[j][1] * inv0);
        *reinterpret_cast<float2*>(a.o_part + (row1 * a.max_splits + slot) * kDv + d) =
            make_float2(o[j][2] * inv1, o[j][3] * inv1);
      }
    }
    if (dh == 0 && t == 0) {
      const float lse0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY, lse1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
      if (ns == 1) {
        if (a.out_lse) {
          a.out_lse[row0] = lse0 * kLn2;
          a.out_lse[row1] = lse1 * kLn2;
        }
      } else {
        a.lse_part[row0 * a.max_splits + slot] = lse0;
        a.lse_part[row1 * a.max_splits + slot] = lse1;
      }
    }
    __syncthreads();  // the ring is refilled by the next segment
  }
}

// Merge of the partials of requests spread over several CTAs (one warp per
// row); rows of requests with no selected page get 0 and lse = -inf.
__global__ void __launch_bounds__(128) mla_combine_kernel(const float* __restrict__ o_part,
                                                          const float* __restrict__ lse_part,
                                                          const int32_t* __restrict__ item_ns, int32_t batch,
                                                          int32_t Hq, int32_t max_splits, uint16_t* __restrict__ out,
                                                          float* __restrict__ out_lse) {
  pdl_enter();
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= batch * Hq) return;
  const int lane = threadIdx.x & 31;
  const int ns = min(item_ns[row / Hq], max_splits);
  if (ns == 1) return;
  const float* lp = lse_part + (size_t)row * max_splits;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, lp[s]);
  float wsum = 0.f;
  for (int s = 0; s < ns; ++s) wsum += (lp[s] == -INFINITY) ? 0.f : fast_exp2(lp[s] - M);
  const bool empty_row = !(wsum > 0.f);
  const float inv = empty_row ? 0.f : 1.f / wsum;
  for (int d = lane * 4; d < kDv; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ns; ++s) {
      if (lp[s] == -INFINITY) continue;
      const float f = fast_exp2(lp[s] - M);
      const float4 v = *reinterpret_cast<const float4*>(o_part + ((size_t)row * max_splits + s) * kDv + d);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out + (size_t)row * kDv + d) = pk;
  }
  if (out_lse && lane == 0) out_lse[row] = empty_row ? -INFINITY : (M + log2f(wsum)) * kLn2;
}

size_t smem_bytes(int HG, int32_t batch) {
  return (size_t)kRingBytes + 1024 + (size_t)2 * HG * 2 * 32 * 8 * 4 + (size_t)(batch + 1) * 4;
}

template <int HG>
cudaError_t launch_hg(const MlaArgs& a, int grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<HG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  {
    const cudaError_t le = launch_pdl(mla_decode_kernel<HG>, dim3(grid), dim3(64 * HG), smem, stream, a);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

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

// Requests one launch takes: the per-request prefix must fit beside the ring
// in shared memory (at 64 query heads).
size_t mla_decode_max_items() { return (227 * 1024 - smem_bytes(4, 0)) / 4; }

cudaError_t launch_mla_decode(const KvView& kv, const uint16_t* q, int32_t num_q_heads, const int32_t* block_table,
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
  const int HG = num_q_heads / 16;
  const size_t smem = smem_bytes(HG, batch);
  cudaError_t e;
  switch (HG) {
    case 1: e = launch_hg<1>(a, plan.grid, smem, stream); break;
    case 2: e = launch_hg<2>(a, plan.grid, smem, stream); break;
    case 3: e = launch_hg<3>(a, plan.grid, smem, stream); break;
    default: e = launch_hg<4>(a, plan.grid, smem, stream); break;
  }
  if (e != cudaSuccess) return e;
  {
    const cudaError_t le = launch_pdl(mla_combine_kernel, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, stream,
                                      a.o_part, a.lse_part, a.item_ns, batch, num_q_heads, plan.nsplit, out, out_lse);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace se
