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
//  * Math per page, lane = (tg = lane & 7, dg = lane >> 3): tokens tg and
//    tg + 8, head dims [16 dg, 16 dg + 16).  QK^T partial sums use packed FP32
//    FMAs; the 8 partial scores are reduced across the 4 d-groups with a
//    transposing butterfly that leaves each lane two finished scores.  Each
//    token group tg keeps its own running max / sum / accumulator (an
//    independent online-softmax stream); the streams of all groups and warps
//    are merged once at the end through shared memory.
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
constexpr int kStreams = kWarps * 8;  // online-softmax streams per CTA
constexpr int kMaxPagesPerSplit = 1024;
constexpr unsigned kFull = 0xFFFFFFFFu;

static_assert(kStreams * (2 * kGroup + kGroup * kHeadDim) * 4 <= kStageBytes,
              "end-of-CTA merge scratch must fit in the stage buffers");

__host__ __device__ constexpr size_t smem_bytes(int pages_per_split) {
  return 1024 /* alignment slack */ + kStageBytes + kBarBytes +
         static_cast<size_t>(pages_per_split) * 4;
}

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

__global__ void __launch_bounds__(kThreads, 3)
    paged_decode_kernel(const __grid_constant__ CUtensorMap pool_map,
                        const AttnArgs a) {
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

  // ---- lane geometry and the 4 query rows (pre-scaled into log2 units)
  const int tg = lane & 7;
  const int dg = lane >> 3;
  const bool hi4 = (lane & 16) != 0;  // which of the two tokens after reduction
  const bool hi3 = (lane & 8) != 0;   // which row pair after reduction
  float2 qf[kGroup][8];
  {
    const uint16_t* qrow =
        a.q + (static_cast<int64_t>(b) * kNumQHeads + g * kGroup) * kHeadDim + 16 * dg;
#pragma unroll
    for (int r = 0; r < kGroup; ++r) {
      const uint4 w0 = *reinterpret_cast<const uint4*>(qrow + r * kHeadDim);
      const uint4 w1 = *reinterpret_cast<const uint4*>(qrow + r * kHeadDim + 8);
      const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 x = bf16x2_to_float2(w[e]);
        qf[r][e] = make_float2(x.x * a.scale_log2, x.y * a.scale_log2);
      }
    }
  }
  // Swizzled byte offsets of this lane's two 16-byte chunks within a row
  // (TMA 128-byte swizzle: chunk c of row r sits at chunk c ^ (r & 7); both
  // tokens of this lane have r & 7 == tg).
  const uint32_t off_a = static_cast<uint32_t>(((2 * dg) ^ tg) << 4);
  const uint32_t off_b = static_cast<uint32_t>(((2 * dg + 1) ^ tg) << 4);

  const int nw = n > warp ? (n - warp + kWarps - 1) / kWarps : 0;
  const uint64_t policy = l2_policy_evict_first();
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

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float2 o[kGroup][8];
#pragma unroll
  for (int r = 0; r < kGroup; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[r][e] = make_float2(0.f, 0.f);

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

      // scores: s[i][r] = partial dot over this lane's 16 dims, token tg + 8i
      float s[2][kGroup];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t row = kt + (tg + 8 * i) * kRowBytes;
        const uint4 ka = lds128(row + off_a);
        const uint4 kb = lds128(row + off_b);
        const uint32_t w[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
        float2 kf[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) kf[e] = bf16x2_to_float2(w[e]);
#pragma unroll
        for (int r = 0; r < kGroup; ++r) {
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = ffma2(qf[r][e], kf[e], acc);
          s[i][r] = acc.x + acc.y;
        }
      }
      // transposing reduction over the 4 d-groups (lanes ^16, ^8)
      float u[kGroup];
#pragma unroll
      for (int r = 0; r < kGroup; ++r) {
        const float send = hi4 ? s[0][r] : s[1][r];
        const float keep = hi4 ? s[1][r] : s[0][r];
        u[r] = keep + __shfl_xor_sync(kFull, send, 16);
      }
      float sc[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float send = hi3 ? u[rr] : u[2 + rr];
        const float keep = hi3 ? u[2 + rr] : u[rr];
        sc[rr] = keep + __shfl_xor_sync(kFull, send, 8);
      }
      // this lane now owns token tg + 8*hi4, rows 2*hi3 + {0, 1}
      if (valid < kPageSize && tg + (hi4 ? 8 : 0) >= valid) sc[0] = sc[1] = -INFINITY;

      float p[2], alpha[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float pm = fmaxf(sc[rr], __shfl_xor_sync(kFull, sc[rr], 16));
        const float m_new = fmaxf(m_run[rr], pm);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        p[rr] = fast_exp2(sc[rr] - m_use);
        alpha[rr] = fast_exp2(m_run[rr] - m_use);
        l_run[rr] = l_run[rr] * alpha[rr] + p[rr];
        m_run[rr] = m_new;
      }
      // gather the group's rescale factors (4 rows) and weights (2 tokens x 4 rows)
      const float ao0 = __shfl_xor_sync(kFull, alpha[0], 8);
      const float ao1 = __shfl_xor_sync(kFull, alpha[1], 8);
      const float a4[kGroup] = {hi3 ? ao0 : alpha[0], hi3 ? ao1 : alpha[1],
                                hi3 ? alpha[0] : ao0, hi3 ? alpha[1] : ao1};
      float pp[2][kGroup];
#pragma unroll
      for (int src = 0; src < 4; ++src) {
        const int sl = tg + 8 * src;
        pp[src >> 1][2 * (src & 1) + 0] = __shfl_sync(kFull, p[0], sl);
        pp[src >> 1][2 * (src & 1) + 1] = __shfl_sync(kFull, p[1], sl);
      }
#pragma unroll
      for (int r = 0; r < kGroup; ++r)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][e] = fmul2(o[r][e], f2(a4[r]));
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (valid == kPageSize || tg + 8 * i < valid) {
          const uint32_t row = vt + (tg + 8 * i) * kRowBytes;
          const uint4 va = lds128(row + off_a);
          const uint4 vb = lds128(row + off_b);
          const uint32_t w[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 vf = bf16x2_to_float2(w[e]);
#pragma unroll
            for (int r = 0; r < kGroup; ++r) o[r][e] = ffma2(f2(pp[i][r]), vf, o[r][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && k + kStages < nw) {
      fence_proxy_async_smem();
      issue(k + kStages);
    }
  }

  // ---- merge the 32 streams of this CTA
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) l_run[rr] += __shfl_xor_sync(kFull, l_run[rr], 16);
  __syncthreads();  // every warp is done with its stage ring
  float* sm_m = reinterpret_cast<float*>(smem);
  float* sm_l = sm_m + kStreams * kGroup;
  float* sm_o = sm_l + kStreams * kGroup;
  const int stream = warp * 8 + tg;
  if (!hi4) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      sm_m[stream * kGroup + 2 * hi3 + rr] = m_run[rr];
      sm_l[stream * kGroup + 2 * hi3 + rr] = l_run[rr];
    }
  }
#pragma unroll
  for (int r = 0; r < kGroup; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e)
      *reinterpret_cast<float2*>(sm_o + (stream * kGroup + r) * kHeadDim + 16 * dg + 2 * e) =
          o[r][e];
  __syncthreads();

  {
    const int r = warp;  // 4 warps <-> 4 query rows
    const int d = 2 * lane;
    float M = -INFINITY;
#pragma unroll 8
    for (int sidx = 0; sidx < kStreams; ++sidx) M = fmaxf(M, sm_m[sidx * kGroup + r]);
    float Ls = 0.f;
    float2 O = make_float2(0.f, 0.f);
    if (M != -INFINITY) {
      for (int sidx = 0; sidx < kStreams; ++sidx) {
        const float ms = sm_m[sidx * kGroup + r];
        if (ms == -INFINITY) continue;
        const float w = fast_exp2(ms - M);
        Ls += sm_l[sidx * kGroup + r] * w;
        const float2 os =
            *reinterpret_cast<const float2*>(sm_o + (sidx * kGroup + r) * kHeadDim + d);
        O = ffma2(f2(w), os, O);
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
      O = ffma2(f2(w), acc, O);
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

cudaError_t launch_paged_decode_attention(const CUtensorMap& pool_map,
                                          const AttnArgs& args,
                                          cudaStream_t stream) {
  // The dynamic shared-memory opt-in is per device; set it once per device.
  static std::atomic<unsigned long long> configured{0};
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  const unsigned long long bit = 1ull << (device & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(paged_decode_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes(kMaxPagesPerSplit)));
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const dim3 grid(kNumKvHeads * args.plan.num_splits, args.batch);
  paged_decode_kernel<<<grid, kThreads, smem_bytes(args.plan.pages_per_split), stream>>>(
      pool_map, args);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (args.plan.num_splits > 1) {
    merge_splits_kernel<<<dim3(kNumQHeads, args.batch), 32, 0, stream>>>(args);
    err = cudaGetLastError();
  }
  return err;
}

}  // namespace pkv
