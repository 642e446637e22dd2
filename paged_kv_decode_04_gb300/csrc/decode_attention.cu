// decode_attention.cu -- paged decode attention with an FP32 online softmax,
// one CTA per (sequence, kv head, split).
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗", paged decode attention
// item: every query head streams its own sequence's cached pages and
// accumulates softmax-weighted values with an online (running-max) softmax in
// FP32, never gathering a contiguous prefix and never storing the scores.
//
// Decomposition
// -------------
//  * One CTA per (sequence b, kv head g, split).  The 4 query heads that share
//    kv head g (j = 4g..4g+3) are handled together, so each K/V row fetched
//    from HBM serves all four.
//  * Each of the 4 warps owns every 4th page of the CTA's page range and a
//    private ring of kStages page tiles in shared memory.  Lane 0 fills the
//    ring with 3-D TMA copies (one 4 KiB box per page: the 16 K rows and the
//    16 V rows of head g, 128 B each, 128-byte swizzled) completing on one
//    mbarrier per stage, kStages pages ahead of the math.
//  * The per-page math (tensor-core QK^T and PV with the FP32 online softmax)
//    is in decode_page.cuh; the warps' states are merged through shared
//    memory at the end.
//  * With more than one split per sequence the CTA writes an unnormalised
//    (max, sum, acc) partial and a small merge kernel combines the splits of
//    each (b, j) in fixed order, so results are run-to-run deterministic.
//  * kAppend: the fused decode step.  The warp that owns the sequence's last
//    page computes the new token's K/V row for head g, writes it to the pool
//    and patches its copy of the page before the math.
//  * kPlanned: the work comes from a host-built plan (planner.cpp): CTA
//    (g, i) takes item i, either a range of one sequence (as above) or up to
//    4 short sequences, one per warp, each warp writing its own rows.  These
//    grids launch in clusters of two kv heads of an item, which start
//    together (launch_variant).
//  * kStages: the per-warp ring depth -- 4 tiles (3 CTAs per SM) when it can
//    hold every page a warp gets, else 3 tiles at 4 CTAs per SM.
//  * Before griddepcontrol.wait a CTA only prefetches its first ring fill
//    into L2 (prefetch_first_tiles), so that a CTA made resident while the
//    previous grid drains already pulls its pages.
//  * kBeside (planned, a shared-prefix plan's beside layout): the grid runs
//    next to the shared-prefix grid launched just before it and waits for
//    it only at its end; its CTAs share each SM with a shared-prefix CTA.
//  * Batches that fill the SMs go to decode_pagebox.cu instead (one CTA per
//    sequence range for all heads, whole-page boxes).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "decode_page.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kHeadPair = 2;  // CTAs per cluster of a planned launch (grid x = kv head)
static_assert(kNumKvHeads % kHeadPair == 0, "clusters of kv heads");
constexpr int kMaxPagesPerSplit = 1024;
static_assert(kWarps == kPlanWarps, "work plans pack one sequence per warp");

// Stage ring depth per warp.  With at most kDeepStages pages per warp the
// ring holds all of them at once (3 CTAs per SM fit); longer ranges use
// kShallowStages, which keeps the bytes in flight per SM the same with 4
// CTAs per SM (measured on a mixed 16..2048-token batch: 7.5 % faster; on
// sequences of 3-4 pages per warp the deep ring is 17 % faster).
constexpr int kDeepStages = 4;
constexpr int kShallowStages = 3;

__host__ __device__ constexpr int stage_bytes(int stages) { return kWarps * stages * kTileBytes; }
__host__ __device__ constexpr int bar_bytes(int stages) { return kWarps * stages * 8; }
__host__ __device__ constexpr int ctas_per_sm(int stages) { return stages == kShallowStages ? 4 : 3; }

static_assert(kWarps * (2 * kGroup + kGroup * kHeadDim) * 4 <= stage_bytes(kShallowStages),
              "end-of-CTA merge scratch must fit in the stage buffers");

__host__ __device__ constexpr size_t smem_bytes(int stages, int pages_per_split) {
  return 1024 /* alignment slack */ + stage_bytes(stages) + bar_bytes(stages) +
         static_cast<size_t>(pages_per_split) * 4;
}

// Merge of one query row over the partial slots base + s * stride, s < nr,
// into a bf16 output row: one warp, lane l holding dims 2l and 2l + 1.  The
// splits are taken 16 at a time: lane s loads split s's (max, sum) pair and
// every lane loads its two dims of all 16 accumulators at once (they do not
// depend on the max), so one round of loads serves up to 16 splits; the
// pairs are combined with shuffles and the accumulators added in split
// order (deterministic).  Splits that saw no valid key (sum 0) get weight 0.
// The partials are read through L2 (ld.global.cg).
constexpr int kMergeBatch = 16;
constexpr int kMergeRowsMax = 4;  // query rows (warps) per CTA of merge_plan_kernel
static_assert(kNumQHeads % kMergeRowsMax == 0, "merge CTAs cover whole sequences");

__device__ __forceinline__ void merge_row(const AttnArgs& a, int64_t base, int64_t stride,
                                          int nr, uint16_t* out_row, int lane) {
  float M = -INFINITY, Ls = 0.f;
  float2 O = make_float2(0.f, 0.f);
  for (int s0 = 0; s0 < nr; s0 += kMergeBatch) {
    const int cnt = min(kMergeBatch, nr - s0);
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < cnt)
      ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + (base + (s0 + lane) * stride) * 2));
    float2 acc[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u)
      acc[u] = u < cnt ? __ldcg(reinterpret_cast<const float2*>(
                             a.part_acc + (base + (s0 + u) * stride) * kHeadDim + 2 * lane))
                       : make_float2(0.f, 0.f);
    float m = ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
    if (m == -INFINITY) continue;  // no valid key in these splits
    // rescale what earlier batches gathered to the new maximum
    const float Mn = fmaxf(M, m);
    const float r = M == -INFINITY ? 0.f : fast_exp2(M - Mn);
    Ls *= r;
    O.x *= r;
    O.y *= r;
    M = Mn;
    const float wgt = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
    float lw = ml.y * wgt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(kFullMask, lw, o);
    Ls += lw;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float wu = __shfl_sync(kFullMask, wgt, u);
      O.x = fmaf(wu, acc[u].x, O.x);
      O.y = fmaf(wu, acc[u].y, O.y);
    }
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  *reinterpret_cast<uint32_t*>(out_row + 2 * lane) =
      static_cast<uint32_t>(float_to_bf16_rne(O.x * inv)) |
      (static_cast<uint32_t>(float_to_bf16_rne(O.y * inv)) << 16);
}

// pick(v, i): component i of an int4.
__device__ __forceinline__ int pick(int4 v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Before griddepcontrol.wait: prefetch into L2 the head-g tiles that the
// CTA's first ring fill will load, so that a CTA made resident while the
// previous grid drains finds them there.  The plan item (head, bs, ls) is
// read before the wait: a plan is filled by a copy, never by a kernel, so it
// is complete before this grid starts.  The lengths and block-table entries
// read here may still be written by the previous grid, so they are only
// addresses for the prefetch: reads bypass L1, every index is range-checked,
// nothing is recorded, and the kernel reads them again after the wait.  (A mixed 16..2048-token
// batch, 16 layers: 267.5 -> 252.4 us per step; prefetching twice the ring
// fill: 257.0 us.)
template <int kStages, bool kPlanned>
__device__ __forceinline__ void prefetch_first_tiles(const CUtensorMap* map, const AttnArgs& a,
                                                     int g, int tid, int4 head, int4 bs, int4 ls) {
  int b = -1, p = -1;  // this thread's tile: sequence b, logical page p
  if constexpr (kPlanned) {
    if (head.x == kPlanKindPacked) {
      const int w = tid >> 5, l = tid & 31;
      if (l < kStages) {
        b = pick(bs, w);
        if (l * kPageSize < pick(ls, w)) p = l;
      }
    } else if (tid < kWarps * kStages && tid < head.w) {
      b = bs.x;
      p = head.z + tid;
    }
  } else {
    const int split = blockIdx.x / kNumKvHeads;
    const int pps = a.plan.pages_per_split;
    const int L = ld_cg(a.seq_lens + blockIdx.y);
    const int np = (min(max(L, 0), a.max_blocks * kPageSize) + kPageSize - 1) / kPageSize;
    if (tid < kWarps * kStages && tid < pps && split * pps + tid < np) {
      b = blockIdx.y;
      p = split * pps + tid;
    }
  }
  if (b >= 0 && b < a.batch && p >= 0 && p < a.max_blocks) {
    const int pid = ld_cg(a.block_table + static_cast<int64_t>(b) * a.max_blocks + p);
    if (pid >= 0 && pid < a.num_pages) tma_prefetch_l2_3d(map, g * kHeadDim, 0, pid);
  }
}

template <bool kAppend, int kStages, bool kPlanned, bool kBeside = false>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(kStages))
    paged_decode_kernel(const __grid_constant__ CUtensorMap pool_map,
                        const AttnArgs a, const AppendArgs ap) {
  static_assert(kPlanned || !kBeside, "only planned grids run beside the shared-prefix grid");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + stage_bytes(kStages));
  int32_t* s_pages = reinterpret_cast<int32_t*>(smem + stage_bytes(kStages) + bar_bytes(kStages));

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g = blockIdx.x % kNumKvHeads;
  if (tid == 0) tma_prefetch_desc(&pool_map);
  // planned: the item {kind, slot, p_begin, n}, the warps' sequences and
  // lengths (plan data: complete before this grid starts)
  int4 p_head = make_int4(0, 0, 0, 0), p_bs = p_head, p_ls = p_head;
  if constexpr (kPlanned) {
    const int4* it = a.plan_items + static_cast<int64_t>(blockIdx.y) * (kPlanItemWords / 4);
    p_head = it[0];
    p_bs = it[1];
    p_ls = it[2];
  }
  prefetch_first_tiles<kStages, kPlanned>(&pool_map, a, g, tid, p_head, p_bs, p_ls);
  // Beside (a shared-prefix plan's layout 1): the grid before this one is the
  // shared-prefix grid, whose CTAs let this grid launch only after their own
  // wait, so this CTA's inputs are final; that grid reads only shared pages
  // (never a sequence's last page) and writes only its partial slots.  So
  // this CTA starts at once and waits for that grid only before it exits.
  if constexpr (!kBeside) wait_for_prior_grids();
  allow_dependent_grids();

  // ---- this CTA's work.  Range: the 4 warps share the logical pages
  // [p_begin, p_begin + n) of sequence b (warp w takes every 4th page from
  // p_begin + w).  Packed (work plans only): warp w attends the whole of its
  // own sequence wb (-1: none), pages [0, pages(wL)).
  bool packed = false;
  int wb, wL;         // this warp's sequence and its length
  int p_begin = 0, n = 0;
  int64_t part_row0 = -1;  // partial slot of query row 4g, -1: write the output itself
  int dev_len = -2;        // planned: device length of wb, read for the plan check
  int plan_len = 0;        // planned: the length the plan was built for
  int part_step = 0;       // slot distance between consecutive query rows
  const int Lmax = a.max_blocks * kPageSize;
  if constexpr (kPlanned) {
    const int4 head = p_head;  // (kind, slot, p_begin, n)
    const int4 bs = p_bs;      // sequence of each warp
    const int4 ls = p_ls;      // its length, as the plan was built for
    packed = head.x == kPlanKindPacked;
    p_begin = head.z;
    n = head.w;
    wb = pick(bs, packed ? warp : 0);
    wL = pick(ls, packed ? warp : 0);
    plan_len = wL;
    if (head.y >= 0) {
      part_row0 = static_cast<int64_t>(head.y) * kNumQHeads + g * kGroup;
      part_step = 1;
    }
    // the lengths come from the plan; seq_lens is only checked against it
    // (the load is consumed at the end of the kernel, off the critical path)
    if (wb >= 0 && lane == 0 && (packed || warp == 0) && g == 0) dev_len = a.seq_lens[wb];
    wL = wL < 0 ? 0 : (wL > Lmax ? Lmax : wL);
  } else {
    const int split = blockIdx.x / kNumKvHeads;
    const int pps = a.plan.pages_per_split;
    wb = blockIdx.y;
    wL = a.seq_lens[wb];
    if (wL < 0 || wL > Lmax) {
      if (tid == 0 && blockIdx.x == 0) record_error(a.dev_err, kErrSeqLen);
      wL = wL < 0 ? 0 : Lmax;
    }
    const int np = (wL + kPageSize - 1) / kPageSize;
    const int nsplit = np > 0 ? (np + pps - 1) / pps : 1;
    if (split >= nsplit) return;
    p_begin = split * pps;
    n = min(pps, np - p_begin);  // 0 only when L == 0
    if (nsplit > 1) {
      part_row0 = (static_cast<int64_t>(wb) * kNumQHeads + g * kGroup) * a.plan.num_splits + split;
      part_step = a.plan.num_splits;
    }
  }
  const int npages = (wL + kPageSize - 1) / kPageSize;  // pages of this warp's sequence

  // ---- page ids of the CTA's pages (range) or of each warp's (packed)
  int s_base, s_step, nw, l_base, l_step;
  if (packed) {
    nw = wb >= 0 ? min(npages, kPackPages) : 0;
    s_base = warp * kPackPages;
    s_step = 1;
    l_base = 0;
    l_step = 1;
    for (int i = lane; i < nw; i += 32) {
      int32_t pid = a.block_table[static_cast<int64_t>(wb) * a.max_blocks + i];
      if (pid < 0 || pid >= a.num_pages) {
        record_error(a.dev_err, kErrPage);
        pid = -1;
      }
      s_pages[s_base + i] = pid;
    }
  } else {
    nw = n > warp ? (n - warp + kWarps - 1) / kWarps : 0;
    s_base = warp;
    s_step = kWarps;
    l_base = p_begin + warp;
    l_step = kWarps;
    for (int i = tid; i < n; i += kThreads) {
      int32_t pid = a.block_table[static_cast<int64_t>(wb) * a.max_blocks + p_begin + i];
      if (pid < 0 || pid >= a.num_pages) {
        record_error(a.dev_err, kErrPage);
        pid = -1;
      }
      s_pages[i] = pid;
    }
  }
  const uint32_t bar0 = smem_addr(bars) + warp * kStages * 8;
  const uint32_t tile0 = smem_addr(smem) + warp * kStages * kTileBytes;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
  }
  __syncthreads();

  const LaneGeom G(lane);
  uint32_t qb[4][2] = {};
  if (wb >= 0)
    load_q_frags(a.q + (static_cast<int64_t>(wb) * kNumQHeads + g * kGroup) * kHeadDim, G, qb);
  const float c = a.scale_log2;

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int k) {
    const int st = k % kStages;
    const int pid = s_pages[s_base + k * s_step];
    const uint32_t bar = bar0 + 8 * st;
    if (pid >= 0) {
      mbar_arrive_expect_tx(bar, kTileBytes);
      tma_load_3d(tile0 + st * kTileBytes, &pool_map, bar, g * kHeadDim, 0, pid, policy);
    } else {
      mbar_arrive(bar);  // keep the stage's phase sequence in step
    }
  };
  if (lane == 0)
    for (int k = 0; k < kStages && k < nw; ++k) issue(k);

  // ---- fused append: computed while the first copies are in flight.  The
  // owner is the warp whose page list holds the sequence's last page; k_last
  // is that page's position in the list.
  int k_last = -1;
  if (kAppend && npages > 0) {
    const int d = npages - 1 - l_base;
    if (d >= 0 && d % l_step == 0 && d / l_step < nw) k_last = d / l_step;
  }
  const int a_slot = (wL - 1) % kPageSize;
  AppendRow arow{};
  if (k_last >= 0) {
    const int64_t src = (static_cast<int64_t>(wb) * kNumKvHeads + g) * kHeadDim;
    arow = make_append_row(ap.k_new + src, ap.v_new + src, wL - 1, ap.freqs, lane);
    const int pid = s_pages[s_base + k_last * s_step];
    if (pid >= 0) store_append_row(ap.pool, pid, a_slot, g, arow, lane);
  }

  AttnState S;
  S.reset();
  for (int k = 0; k < nw; ++k) {
    const int st = k % kStages;
    const bool ready = mbar_wait_bounded(bar0 + 8 * st, (k / kStages) & 1, a.wait_ns);
    if (!__all_sync(kFullMask, ready)) {
      // give up on this warp's pages, but not before the copies it issued
      // (pages k .. k + kStages - 1, one in flight per stage) have landed --
      // each wait bounded again, by the full limit -- since the epilogue
      // reuses the stage buffers
      if (lane == 0) {
        record_error(a.dev_err, kErrTimeout);
        for (int j = k; j < k + kStages && j < nw; ++j)
          mbar_wait_bounded(bar0 + 8 * (j % kStages), (j / kStages) & 1);
      }
      __syncwarp();
      break;
    }
    if (s_pages[s_base + k * s_step] >= 0) {
      const uint32_t kt = tile0 + st * kTileBytes;
      if (k == k_last) patch_append_row(kt, a_slot, arow, lane);
      const int valid = min(kPageSize, wL - (l_base + k * l_step) * kPageSize);
      attend_page(kt, valid, qb, c, G, lane, S);
    }
    __syncwarp();
    if (lane == 0 && k + kStages < nw) {
      fence_proxy_async_smem();
      issue(k + kStages);
    }
  }

  // ---- the warps' states through shared memory
  reduce_row_sums(S);
  __syncthreads();  // every warp is done with its stage ring
  float* sm_m = reinterpret_cast<float*>(smem);
  float* sm_l = sm_m + kWarps * kGroup;
  float* sm_o = sm_l + kWarps * kGroup;
  if (G.ft < 2) {
    if (G.fg == 0) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        sm_m[warp * kGroup + 2 * G.ft + rr] = S.m_ref[rr];
        sm_l[warp * kGroup + 2 * G.ft + rr] = S.l_run[rr];
      }
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      float* o0 = sm_o + (warp * kGroup + 2 * G.ft) * kHeadDim + 16 * mt + G.fg;
      o0[0] = S.oacc[mt][0];
      o0[kHeadDim] = S.oacc[mt][1];
      o0[8] = S.oacc[mt][2];
      o0[kHeadDim + 8] = S.oacc[mt][3];
    }
  }
  __syncthreads();

  const int d = 2 * lane;
  auto write_row = [&](int seq, int r, float M, float Ls, float2 O, int64_t part) {
    if (part < 0) {
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      const uint32_t v = static_cast<uint32_t>(float_to_bf16_rne(O.x * inv)) |
                         (static_cast<uint32_t>(float_to_bf16_rne(O.y * inv)) << 16);
      const int64_t row = static_cast<int64_t>(seq) * kNumQHeads + g * kGroup + r;
      *reinterpret_cast<uint32_t*>(a.out + row * kHeadDim + d) = v;
    } else {
      *reinterpret_cast<float2*>(a.part_acc + part * kHeadDim + d) = O;
      if (lane == 0) *reinterpret_cast<float2*>(a.part_ml + part * 2) = make_float2(M, Ls);
    }
  };
  if (kPlanned && dev_len != -2 && dev_len != plan_len) record_error(a.dev_err, kErrPlan);
  if (packed) {
    // each warp normalises its own 4 rows
    if (wb >= 0) {
#pragma unroll
      for (int r = 0; r < kGroup; ++r) {
        const float M = sm_m[warp * kGroup + r];
        const float Ls = M == -INFINITY ? 0.f : sm_l[warp * kGroup + r];
        const float2 O = M == -INFINITY ? make_float2(0.f, 0.f)
                                        : *reinterpret_cast<const float2*>(
                                              sm_o + (warp * kGroup + r) * kHeadDim + d);
        write_row(wb, r, M, Ls, O, -1);
      }
    }
  } else {
    const int r = warp;  // 4 warps <-> 4 query rows
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
    write_row(wb, r, M, Ls, O, part_row0 < 0 ? -1 : part_row0 + static_cast<int64_t>(r) * part_step);
  }
  // Beside: no CTA ends before the shared-prefix grid has, so that this
  // grid's completion (what the merge waits for) covers that grid's partials
  if constexpr (kBeside) wait_for_prior_grids();
}

// Combine the split partials of one (b, j): grid (Hq, B), one warp.
__global__ void __launch_bounds__(32) merge_splits_kernel(const AttnArgs a) {
  const int j = blockIdx.x;
  const int b = blockIdx.y;
  const int pps = a.plan.pages_per_split;
  allow_dependent_grids();  // the next grid may launch; it waits for this one itself
  wait_for_prior_grids();
  int L = a.seq_lens[b];
  const int Lmax = a.max_blocks * kPageSize;
  L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  const int npages = (L + kPageSize - 1) / kPageSize;
  const int nsplit = npages > 0 ? (npages + pps - 1) / pps : 1;
  if (nsplit == 1) return;  // written directly by the attention kernel
  const int64_t row = static_cast<int64_t>(b) * kNumQHeads + j;
  merge_row(a, row * a.plan.num_splits, 1, nsplit, a.out + row * kHeadDim, threadIdx.x);
}

// Work plan: combine the ranges of the split sequences the plan lists;
// grid (Hq / rows, merges), one warp per (sequence, query row), `rows` =
// blockDim.x / 32 query rows per CTA.
__global__ void __launch_bounds__(kMergeRowsMax * 32) merge_plan_kernel(const AttnArgs a) {
  allow_dependent_grids();  // the next grid may launch; it waits for this one itself
  // (b, first slot, ranges, 0): plan data, complete before this grid starts
  const int4 e = a.plan_merges[blockIdx.y];
  wait_for_prior_grids();
  const int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t row = static_cast<int64_t>(e.x) * kNumQHeads + j;
  merge_row(a, static_cast<int64_t>(e.y) * kNumQHeads + j, kNumQHeads, e.z,
            a.out + row * kHeadDim, threadIdx.x & 31);
}

// Query rows per merge CTA: one (more CTAs, for few merged sequences) or
// kMergeRowsMax once there are at least as many merged sequences as SMs.
// Measured: 256 merged sequences 82.4 -> 78.7 us per step with 4 rows, one
// 16-range sequence 88.1 -> 90.1 us, so the switch.
int merge_rows_per_cta(int num_merges) {
  static std::atomic<int> sms_of[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  std::atomic<int>& c = sms_of[dev & 63];
  int sms = c.load(std::memory_order_relaxed);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    c.store(sms, std::memory_order_relaxed);
  }
  return num_merges >= sms ? kMergeRowsMax : 1;
}

cudaError_t launch_merge_plan(const AttnArgs& args, int num_merges, cudaStream_t stream) {
  const int rows = merge_rows_per_cta(num_merges);
  return launch_pdl(merge_plan_kernel, dim3(kNumQHeads / rows, num_merges), dim3(32 * rows), 0,
                    stream, args);
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

// The dynamic shared-memory opt-in is per device and per kernel; beside
// instances also ask for the largest shared-memory carveout, the one the
// shared-prefix CTAs they run next to ask for (CTAs of two kernels share an
// SM only under one L1 / shared-memory split).
template <bool kAppend, int kStages, bool kPlanned, bool kBeside>
cudaError_t configure_once(int device) {
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (device & 63);
  if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(
      paged_decode_kernel<kAppend, kStages, kPlanned, kBeside>,
      cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(smem_bytes(kStages, kMaxPagesPerSplit)));
  if (err == cudaSuccess && kBeside)
    err = cudaFuncSetAttribute(paged_decode_kernel<kAppend, kStages, kPlanned, kBeside>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
  if (err == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
  return err;
}

template <bool kAppend, int kStages, bool kPlanned, bool kBeside>
cudaError_t launch_variant(const CUtensorMap& pool_map, const AttnArgs& args,
                           const AppendArgs& append, dim3 grid, int page_list, int device,
                           cudaStream_t stream) {
  const cudaError_t err = configure_once<kAppend, kStages, kPlanned, kBeside>(device);
  if (err != cudaSuccess) return err;
  if constexpr (kPlanned) {
    // Planned grids (kv head, item) run in clusters of kHeadPair CTAs: kv
    // heads 2i and 2i + 1 of an item, whose rows of every page are one
    // contiguous 256-byte span, start together and so stream the same pages
    // side by side.  Measured, same box: a mixed 16..2048-token batch of 16
    // layers 250.2 -> 243.5 us, a 2048-token sequence of 16 layers 92.8 ->
    // 90.6 us; clusters of 4 and 8 (harder to place in one wave) 267 and
    // 277 us on the mixed batch.
    return launch_pdl_cluster(paged_decode_kernel<kAppend, kStages, kPlanned, kBeside>, grid,
                              dim3(kThreads), smem_bytes(kStages, page_list), stream, kHeadPair,
                              pool_map, args, append);
  }
  return launch_pdl(paged_decode_kernel<kAppend, kStages, kPlanned, kBeside>, grid,
                    dim3(kThreads), smem_bytes(kStages, page_list), stream, pool_map, args,
                    append);
}

// Ring depth by the pages a warp gets: deep when the ring holds them all.
template <bool kPlanned, bool kBeside = false>
cudaError_t launch_attention_kernel(const CUtensorMap& pool_map, const AttnArgs& args,
                                    const AppendArgs* append, dim3 grid, int range_pages,
                                    int page_list, int device, cudaStream_t stream) {
  const bool deep = range_pages <= kWarps * kDeepStages;
  const AppendArgs none{};
  if (append != nullptr)
    return deep ? launch_variant<true, kDeepStages, kPlanned, kBeside>(
                      pool_map, args, *append, grid, page_list, device, stream)
                : launch_variant<true, kShallowStages, kPlanned, kBeside>(
                      pool_map, args, *append, grid, page_list, device, stream);
  return deep ? launch_variant<false, kDeepStages, kPlanned, kBeside>(
                    pool_map, args, none, grid, page_list, device, stream)
              : launch_variant<false, kShallowStages, kPlanned, kBeside>(
                    pool_map, args, none, grid, page_list, device, stream);
}

}  // namespace

cudaError_t launch_paged_decode_attention(const CUtensorMap& pool_map,
                                          const AttnArgs& args,
                                          cudaStream_t stream,
                                          const AppendArgs* append) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  const int pps = args.plan.pages_per_split;
  err = launch_attention_kernel<false>(pool_map, args, append,
                                       dim3(kNumKvHeads * args.plan.num_splits, args.batch), pps,
                                       pps, device, stream);
  if (err != cudaSuccess) return err;
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (args.plan.num_splits > 1) {
    err = launch_pdl(merge_splits_kernel, dim3(kNumQHeads, args.batch), dim3(32), 0, stream,
                     args);
  }
  return err;
}

cudaError_t launch_split_merge(const AttnArgs& args, int num_merges, cudaStream_t stream) {
  if (args.plan_items != nullptr)
    return num_merges > 0 ? launch_merge_plan(args, num_merges, stream) : cudaSuccess;
  return args.plan.num_splits > 1 ? launch_pdl(merge_splits_kernel,
                                               dim3(kNumQHeads, args.batch), dim3(32), 0, stream,
                                               args)
                                  : cudaSuccess;
}

cudaError_t launch_planned_decode_attention(const CUtensorMap& pool_map,
                                            const AttnArgs& args, int num_items,
                                            int num_merges, int range_pages,
                                            cudaStream_t stream, const AppendArgs* append,
                                            bool beside) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  const int page_list = range_pages > kWarps * kPackPages ? range_pages : kWarps * kPackPages;
  const dim3 grid(kNumKvHeads, num_items);
  err = beside ? launch_attention_kernel<true, true>(pool_map, args, append, grid, range_pages,
                                                     page_list, device, stream)
               : launch_attention_kernel<true>(pool_map, args, append, grid, range_pages,
                                               page_list, device, stream);
  if (err != cudaSuccess) return err;
  if (num_merges > 0) err = launch_merge_plan(args, num_merges, stream);
  return err;
}

}  // namespace pkv
