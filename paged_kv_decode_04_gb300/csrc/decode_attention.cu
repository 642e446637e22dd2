// decode_attention.cu -- paged decode attention with an FP32 online softmax.
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗", paged decode attention
// item: every query head streams its own sequence's cached pages and
// accumulates softmax-weighted values with an online (running-max) softmax in
// FP32, never gathering a contiguous prefix and never storing the scores.
//
// Decomposition for sm_103a
// -------------------------
//  * One CTA per (sequence b, kv head g, split).  The 4 query heads that share
//    kv head g (j = 4g..4g+3) are handled together, so each K/V row fetched
//    from HBM serves all four.
//  * Each of the 4 warps owns every 4th page of the CTA's page range and a
//    private ring of kStages page tiles in shared memory.  Lane 0 fills the
//    ring with 3-D TMA copies (one 4 KiB box per page: the 16 K rows and the
//    16 V rows of head g, 128 B each, 128-byte swizzled) completing on one
//    mbarrier per stage, kStages pages ahead of the math.
//  * Math per page on the tensor cores (mma.sync m16n8k16, bf16 in, FP32
//    accumulate): S^T = K Q^T with the 16 page tokens as M and the 4 query
//    rows (padded to 8) as N, then O^T += V^T P^T with the 64 head dims as M.
//    K comes from shared memory through ldmatrix, V through ldmatrix.trans;
//    the probabilities P enter the second product as two bf16 terms
//    (hi + lo), which keeps about 16 significant bits of every weight.
//  * Softmax: scores, running max, exponentials and sums stay in FP32.  The
//    running max is a lazily updated reference: a page only forces a rescale
//    of the accumulators when one of its scores exceeds the reference by more
//    than kRescaleLog2 (so the weights stay <= 2^kRescaleLog2); the final
//    normalisation by the running sum makes the result independent of the
//    reference, exactly as in the textbook online softmax.
//  * With more than one split per sequence the CTA writes an unnormalised
//    (max, sum, acc) partial and a small merge kernel combines the splits of
//    each (b, j) in fixed order, so results are run-to-run deterministic.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr int kRowBytes = kHeadDim * 2;                   // 128 B: one head's row
constexpr int kTileBytes = 2 * kPageSize * kRowBytes;     // 4 KiB: K then V
constexpr int kStageBytes = kWarps * kStages * kTileBytes;
constexpr int kBarBytes = kWarps * kStages * 8;
// A page rescales the accumulators only when a score exceeds the running
// reference maximum by more than this many powers of two.
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxPagesPerSplit = 1024;
constexpr unsigned kFull = 0xFFFFFFFFu;

static_assert(kWarps * (2 * kGroup + kGroup * kHeadDim) * 4 <= kStageBytes,
              "end-of-CTA merge scratch must fit in the stage buffers");

__host__ __device__ constexpr size_t smem_bytes(int pages_per_split) {
  return 1024 /* alignment slack */ + kStageBytes + kBarBytes +
         static_cast<size_t>(pages_per_split) * 4;
}

template <bool kAppend>
__global__ void __launch_bounds__(kThreads, 3)
    paged_decode_kernel(const __grid_constant__ CUtensorMap pool_map,
                        const AttnArgs a, const AppendArgs ap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStageBytes);
  int32_t* s_pages = reinterpret_cast<int32_t*>(smem + kStageBytes + kBarBytes);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g = blockIdx.x % kNumKvHeads;
  const int split = blockIdx.x / kNumKvHeads;
  const int b = blockIdx.y;
  const int pps = a.plan.pages_per_split;

  // ---- sequence extent and this CTA's page range
  int L = a.seq_lens[b];
  const int Lmax = a.max_blocks * kPageSize;
  if (L < 0 || L > Lmax) {
    if (tid == 0 && blockIdx.x == 0) record_error(a.dev_err, kErrSeqLen);
    L = L < 0 ? 0 : Lmax;
  }
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int nsplit = npages > 0 ? (npages + pps - 1) / pps : 1;
  if (split >= nsplit) return;
  const int p_begin = split * pps;
  const int n = min(pps, npages - p_begin);  // 0 only when L == 0

  for (int i = tid; i < n; i += kThreads) {
    int32_t pid = a.block_table[static_cast<int64_t>(b) * a.max_blocks + p_begin + i];
    if (pid < 0 || pid >= a.num_pages) {
      record_error(a.dev_err, kErrPage);
      pid = -1;
    }
    s_pages[i] = pid;
  }
  const uint32_t bar0 = smem_addr(bars) + warp * kStages * 8;
  const uint32_t tile0 = smem_addr(smem) + warp * kStages * kTileBytes;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ---- lane geometry: mma fragment coordinates and ldmatrix row addresses
  const int fg = lane >> 2;  // fragment group: token (S^T) / head dim (O^T) row
  const int ft = lane & 3;   // thread in group: query rows 2ft, 2ft + 1
  const int lr = lane & 7;   // ldmatrix: row within an 8x8 matrix
  const int li = lane >> 3;  // ldmatrix: which of the four matrices
  // Q^T as the B operand of S^T = K Q^T: columns 0..3 are the group's query
  // rows, columns 4..7 are zero padding.
  uint32_t qb[4][2];
  {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(
        a.q + (static_cast<int64_t>(b) * kNumQHeads + g * kGroup + (fg & 3)) * kHeadDim);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      qb[kk][0] = fg < kGroup ? qw[kk * 8 + ft] : 0u;
      qb[kk][1] = fg < kGroup ? qw[kk * 8 + 4 + ft] : 0u;
    }
  }
  // Swizzled row addresses (TMA 128-byte swizzle: 16-byte chunk c of row r
  // sits at chunk c ^ (r & 7); every row used below has r & 7 == lr).
  // K, non-transposed: matrix li covers tokens 8*(li & 1).., dims chunk 2kk + (li >> 1).
  const uint32_t k_row = static_cast<uint32_t>((lr + 8 * (li & 1)) * kRowBytes);
  const int k_chunk = li >> 1;
  // V, transposed: matrix li covers tokens 8*(li >> 1).., dims chunk 2mt + (li & 1).
  const uint32_t v_row = static_cast<uint32_t>((lr + 8 * (li >> 1)) * kRowBytes);
  const int v_chunk = li & 1;
  // P^T as the B operand of O^T += V^T P^T: lane (fg, ft) needs row fg's
  // weights for tokens 2ft, 2ft+1, 2ft+8, 2ft+9, held by lanes 8ft + (fg >> 1)
  // and 8ft + 4 + (fg >> 1) in the S^T fragment layout.
  const int src_a = 8 * ft + (fg >> 1);
  const int src_b = src_a + 4;
  const bool odd_row = (fg & 1) != 0;
  const float c = a.scale_log2;

  const int nw = n > warp ? (n - warp + kWarps - 1) / kWarps : 0;
  const uint64_t policy = l2_policy_evict_first();

  // ---- fused append: the warp that owns the sequence's last page rotates
  // the new token's key for head g (lane i: pair i, i + 32), copies its value
  // (lane i: dims 2i, 2i + 1), writes both into the pool slot for later steps
  // and keeps them to patch its copy of that page in shared memory.
  const int last_local = npages - 1 - p_begin;  // index of the last page in this range
  const bool owns_last = kAppend && npages > 0 && last_local >= 0 && last_local < n &&
                         last_local % kWarps == warp;
  uint16_t ky1 = 0, ky2 = 0;
  uint32_t vv = 0;
  const int a_slot = (L - 1) % kPageSize;
  if (owns_last) {
    const int pos = L - 1;
    const int64_t src = (static_cast<int64_t>(b) * kNumKvHeads + g) * kHeadDim;
    const uint16_t x1 = ap.k_new[src + lane];
    const uint16_t x2 = ap.k_new[src + lane + 32];
    vv = reinterpret_cast<const uint32_t*>(ap.v_new + src)[lane];
    double sn, cs;
    sincos(__dmul_rn(static_cast<double>(pos), ap.freqs.inv_freq[lane]), &sn, &cs);
    rotate_pair(x1, x2, cs, sn, &ky1, &ky2);
    const int pid = s_pages[last_local];
    if (pid >= 0) {
      const int64_t row = kNumKvHeads * kHeadDim;
      uint16_t* kd = ap.pool + ((static_cast<int64_t>(pid) * 2 + 0) * kPageSize + a_slot) * row +
                     g * kHeadDim;
      uint16_t* vd = ap.pool + ((static_cast<int64_t>(pid) * 2 + 1) * kPageSize + a_slot) * row +
                     g * kHeadDim;
      kd[lane] = ky1;
      kd[lane + 32] = ky2;
      reinterpret_cast<uint32_t*>(vd)[lane] = vv;
    }
  }
  auto issue = [&](int k) {
    const int st = k % kStages;
    const int pid = s_pages[warp + k * kWarps];
    const uint32_t bar = bar0 + 8 * st;
    if (pid >= 0) {
      mbar_arrive_expect_tx(bar, kTileBytes);
      tma_load_3d(tile0 + st * kTileBytes, &pool_map, bar, g * kHeadDim, 0, pid, policy);
    } else {
      mbar_arrive(bar);  // keep the stage's phase sequence in step
    }
  };
  if (lane == 0) {
    tma_prefetch_desc(&pool_map);
    for (int k = 0; k < kStages && k < nw; ++k) issue(k);
  }

  float m_ref[2] = {-INFINITY, -INFINITY};  // per query row 2ft + rr, log2 units
  float l_run[2] = {0.f, 0.f};              // this lane's share of the row sums
  float oacc[4][4];                         // O^T fragments: dims 16mt + fg (+8), rows 2ft (+1)
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;

  for (int k = 0; k < nw; ++k) {
    const int st = k % kStages;
    const bool ready = mbar_wait_bounded(bar0 + 8 * st, (k / kStages) & 1);
    if (!__all_sync(kFull, ready)) {
      if (lane == 0) record_error(a.dev_err, kErrTimeout);
      break;
    }
    const int local = warp + k * kWarps;
    const int pid = s_pages[local];
    if (pid >= 0) {
      const int valid = min(kPageSize, L - (p_begin + local) * kPageSize);
      const uint32_t kt = tile0 + st * kTileBytes;
      const uint32_t vt = kt + kPageSize * kRowBytes;
      if (owns_last && local == last_local) {
        // put the appended token's K and V rows into the (swizzled) tile
        const uint32_t sw = static_cast<uint32_t>(a_slot & 7);
        const uint32_t kr = kt + a_slot * kRowBytes;
        const uint32_t vr = vt + a_slot * kRowBytes;
        sts16(kr + (((static_cast<uint32_t>(lane) >> 3) ^ sw) << 4) + ((lane & 7) << 1), ky1);
        sts16(kr + (((4u + (static_cast<uint32_t>(lane) >> 3)) ^ sw) << 4) + ((lane & 7) << 1),
              ky2);
        sts32(vr + (((static_cast<uint32_t>(lane) >> 2) ^ sw) << 4) + ((lane & 3) << 2), vv);
        __syncwarp();
      }

      // S^T = K Q^T: s[0], s[1] = token fg, rows 2ft, 2ft+1; s[2], s[3] = token fg + 8
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ka[4];
        ldsm_x4(kt + k_row + (static_cast<uint32_t>((2 * kk + k_chunk) ^ lr) << 4), ka);
        mma_16816_bf16(s, ka, qb[kk][0], qb[kk][1]);
      }
      if (valid < kPageSize) {
        // tokens at or past the sequence end: no weight, and their V rows
        // (whatever bytes they hold) are zeroed before the second product
        if (fg >= valid) s[0] = s[1] = -INFINITY;
        if (fg + 8 >= valid) s[2] = s[3] = -INFINITY;
        for (int idx = lane; idx < (kPageSize - valid) * 8; idx += 32)
          sts128_zero(vt + (valid + (idx >> 3)) * kRowBytes + ((idx & 7) << 4));
        __syncwarp();
      }
      float mx0 = fmaxf(s[0], s[2]) * c;
      float mx1 = fmaxf(s[1], s[3]) * c;
      const bool grow = mx0 > m_ref[0] + kRescaleLog2 || mx1 > m_ref[1] + kRescaleLog2;
      if (__any_sync(kFull, grow)) {
#pragma unroll
        for (int x = 4; x <= 16; x <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, x));
          mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, x));
        }
        const float mx[2] = {mx0, mx1};
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const float m_new = fmaxf(m_ref[rr], mx[rr]);
          const float alpha = fast_exp2(m_ref[rr] - m_new);  // 0 on the first page
          l_run[rr] *= alpha;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            oacc[mt][rr] *= alpha;
            oacc[mt][2 + rr] *= alpha;
          }
          m_ref[rr] = m_new;
        }
      }
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = fast_exp2(fmaf(s[e], c, -m_ref[e & 1]));
      l_run[0] += p[0] + p[2];
      l_run[1] += p[1] + p[3];

      // P^T fragments.  P is carried as two bf16 terms, hi = bf16(P) and
      // lo = bf16(P - hi), so the weights keep ~16 significant bits through
      // the bf16 tensor-core product.  Words: (row 2ft | row 2ft+1) x
      // (token fg in the low half, token fg+8 in the high half).
      const uint32_t eh = pack_bf16x2(p[0], p[2]);
      const uint32_t oh = pack_bf16x2(p[1], p[3]);
      const uint32_t el = pack_bf16x2(p[0] - __uint_as_float(eh << 16),
                                      p[2] - __uint_as_float(eh & 0xFFFF0000u));
      const uint32_t ol = pack_bf16x2(p[1] - __uint_as_float(oh << 16),
                                      p[3] - __uint_as_float(oh & 0xFFFF0000u));
      uint32_t pb[2][2];
      {
        const uint32_t w_even[2] = {eh, el};
        const uint32_t w_odd[2] = {oh, ol};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ea = __shfl_sync(kFull, w_even[h], src_a);
          const uint32_t oa = __shfl_sync(kFull, w_odd[h], src_a);
          const uint32_t eb = __shfl_sync(kFull, w_even[h], src_b);
          const uint32_t ob = __shfl_sync(kFull, w_odd[h], src_b);
          const uint32_t wa = odd_row ? oa : ea;  // tokens 2ft (lo), 2ft+8 (hi)
          const uint32_t wb = odd_row ? ob : eb;  // tokens 2ft+1 (lo), 2ft+9 (hi)
          pb[h][0] = prmt(wa, wb, 0x5410u);
          pb[h][1] = prmt(wa, wb, 0x7632u);
        }
      }

      // O^T += V^T (P_hi + P_lo)^T over the four 16-dim slices
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t va[4];
        ldsm_x4_trans(vt + v_row + (static_cast<uint32_t>((2 * mt + v_chunk) ^ lr) << 4), va);
        mma_16816_bf16(oacc[mt], va, pb[0][0], pb[0][1]);
        mma_16816_bf16(oacc[mt], va, pb[1][0], pb[1][1]);
      }
    }
    __syncwarp();
    if (lane == 0 && k + kStages < nw) {
      fence_proxy_async_smem();
      issue(k + kStages);
    }
  }

  // ---- merge the warps' streams
#pragma unroll
  for (int x = 4; x <= 16; x <<= 1) {
    l_run[0] += __shfl_xor_sync(kFull, l_run[0], x);
    l_run[1] += __shfl_xor_sync(kFull, l_run[1], x);
  }
  __syncthreads();  // every warp is done with its stage ring
  float* sm_m = reinterpret_cast<float*>(smem);
  float* sm_l = sm_m + kWarps * kGroup;
  float* sm_o = sm_l + kWarps * kGroup;
  if (ft < 2) {
    if (fg == 0) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        sm_m[warp * kGroup + 2 * ft + rr] = m_ref[rr];
        sm_l[warp * kGroup + 2 * ft + rr] = l_run[rr];
      }
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      float* o0 = sm_o + (warp * kGroup + 2 * ft) * kHeadDim + 16 * mt + fg;
      o0[0] = oacc[mt][0];
      o0[kHeadDim] = oacc[mt][1];
      o0[8] = oacc[mt][2];
      o0[kHeadDim + 8] = oacc[mt][3];
    }
  }
  __syncthreads();

  {
    const int r = warp;  // 4 warps <-> 4 query rows
    const int d = 2 * lane;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * kGroup + r]);
    float Ls = 0.f;
    float2 O = make_float2(0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float ms = sm_m[w * kGroup + r];
        if (ms == -INFINITY) continue;
        const float wt = fast_exp2(ms - M);
        Ls += sm_l[w * kGroup + r] * wt;
        const float2 os =
            *reinterpret_cast<const float2*>(sm_o + (w * kGroup + r) * kHeadDim + d);
        O.x = fmaf(wt, os.x, O.x);
        O.y = fmaf(wt, os.y, O.y);
      }
    }
    const int j = g * kGroup + r;
    const int64_t row = static_cast<int64_t>(b) * kNumQHeads + j;
    if (nsplit == 1) {
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      const uint32_t packed = static_cast<uint32_t>(float_to_bf16_rne(O.x * inv)) |
                              (static_cast<uint32_t>(float_to_bf16_rne(O.y * inv)) << 16);
      *reinterpret_cast<uint32_t*>(a.out + row * kHeadDim + d) = packed;
    } else {
      const int64_t idx = row * a.plan.num_splits + split;
      *reinterpret_cast<float2*>(a.part_acc + idx * kHeadDim + d) = O;
      if (lane == 0) *reinterpret_cast<float2*>(a.part_ml + idx * 2) = make_float2(M, Ls);
    }
  }
}

// Combine the split partials of one (b, j): grid (Hq, B), one warp, 2 dims per lane.
__global__ void __launch_bounds__(32) merge_splits_kernel(const AttnArgs a) {
  const int j = blockIdx.x;
  const int b = blockIdx.y;
  const int lane = threadIdx.x;
  const int pps = a.plan.pages_per_split;
  int L = a.seq_lens[b];
  const int Lmax = a.max_blocks * kPageSize;
  L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int nsplit = npages > 0 ? (npages + pps - 1) / pps : 1;
  if (nsplit == 1) return;  // written directly by the attention kernel
  const int64_t row = static_cast<int64_t>(b) * kNumQHeads + j;
  const int64_t base = row * a.plan.num_splits;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) {
    const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (base + s) * 2);
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  float Ls = 0.f;
  float2 O = make_float2(0.f, 0.f);
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (base + s) * 2);
      if (!(ml.y > 0.f)) continue;
      const float w = fast_exp2(ml.x - M);
      Ls += ml.y * w;
      const float2 acc =
          *reinterpret_cast<const float2*>(a.part_acc + (base + s) * kHeadDim + 2 * lane);
      O.x = fmaf(w, acc.x, O.x);
      O.y = fmaf(w, acc.y, O.y);
    }
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  const uint32_t packed = static_cast<uint32_t>(float_to_bf16_rne(O.x * inv)) |
                          (static_cast<uint32_t>(float_to_bf16_rne(O.y * inv)) << 16);
  *reinterpret_cast<uint32_t*>(a.out + row * kHeadDim + 2 * lane) = packed;
}

}  // namespace

size_t workspace_bytes_for(int batch, int num_q_heads, int head_dim,
                           const SplitPlan& plan) {
  if (plan.num_splits <= 1) return 0;
  return static_cast<size_t>(batch) * num_q_heads * plan.num_splits *
         (static_cast<size_t>(head_dim) + 2) * sizeof(float);
}

int max_pages_per_split() { return kMaxPagesPerSplit; }

namespace {

// The dynamic shared-memory opt-in is per device and per kernel.
template <bool kAppend>
cudaError_t configure_once(int device) {
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (device & 63);
  if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(paged_decode_kernel<kAppend>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem_bytes(kMaxPagesPerSplit)));
  if (err == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
  return err;
}

}  // namespace

cudaError_t launch_paged_decode_attention(const CUtensorMap& pool_map,
                                          const AttnArgs& args,
                                          cudaStream_t stream,
                                          const AppendArgs* append) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  const dim3 grid(kNumKvHeads * args.plan.num_splits, args.batch);
  const size_t smem = smem_bytes(args.plan.pages_per_split);
  if (append != nullptr) {
    err = configure_once<true>(device);
    if (err != cudaSuccess) return err;
    paged_decode_kernel<true><<<grid, kThreads, smem, stream>>>(pool_map, args, *append);
  } else {
    err = configure_once<false>(device);
    if (err != cudaSuccess) return err;
    AppendArgs none{};
    paged_decode_kernel<false><<<grid, kThreads, smem, stream>>>(pool_map, args, none);
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (args.plan.num_splits > 1) {
    merge_splits_kernel<<<dim3(kNumQHeads, args.batch), 32, 0, stream>>>(args);
    err = cudaGetLastError();
  }
  return err;
}

}  // namespace pkv
