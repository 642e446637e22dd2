// decode_segments.cu -- paged decode attention in which one CTA streams an
// equal share of a layer's pages, across sequence boundaries, through one
// ring of whole-page TMA boxes: all 8 kv heads at once, one warp per head.
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗", paged decode attention
// item: every query head streams its own sequence's cached pages with an FP32
// online softmax, never gathering a contiguous prefix or storing scores;
// batched decode packs one token per active sequence and each sequence's
// attention reads only its own cache.
//
// Why: with one CTA per sequence range, a ragged batch (a few long
// sequences among many short ones) has CTAs of very different lengths, short
// sequences each pay a CTA's prologue for a few pages, and the layer ends
// with the longest ranges.  A segment plan (planner.cpp) packs the layer's
// pages into one wave of two CTAs per SM with near-equal page counts: a CTA
// holds up to kSegMax segments {sequence, length, first page, pages, slot}
// -- whole short sequences, or pieces of long ones -- and streams their
// pages back to back through the same ring, so every CTA is busy for the
// whole layer and all of them end together.  A segment that is a whole
// sequence writes its output rows; a piece writes an unnormalised partial
// that the merge kernel combines.  Under a shared-prefix plan the
// shared-prefix kernel is launched first, and a member whose own pages are
// one segment folds that kernel's partials for it into its rows and writes
// the output itself, so such a sequence needs no merge.  In the plan's
// beside layout the CTAs (one per SM, a deeper ring) run next to the
// shared-prefix CTAs, whose kernel is bound by its own MMA and softmax
// chain rather than by DRAM: they stream from the start and wait for that
// kernel only to fold its partials.
//
// Per CTA, at the start: the segments' q rows (4 KiB each) arrive by bulk
// copies; each warp computes the appended token's row of its head for every
// segment that holds its sequence's last page (fused step), writes it to the
// pool and keeps it in shared memory to patch that page's tile.  Then the
// ring streams the pages (the per-page math of decode_page.cuh, as in
// decode_pagebox.cu); at each segment's last page every warp normalises its
// own 4 query rows through a small per-warp exchange area and writes them.
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

constexpr int kSgWarps = kNumKvHeads;  // one warp per kv head
constexpr int kSgThreads = kSgWarps * 32;
constexpr int kSgStages = 2;           // page boxes in the ring (2 CTAs per SM)
constexpr int kSgBesideStages = 4;     // the same beside a shared-prefix CTA (1 CTA per SM)
constexpr int kSgBoxBytes = kNumKvHeads * kTileBytes;  // 32 KiB: one page
constexpr int kQBytes = kNumQHeads * kHeadDim * 2;     // 4 KiB: q of one sequence
constexpr int kXchFloats = 2 * kGroup + kGroup * kHeadDim;  // a warp's rows: m, l, o

// Shared memory from a 1024-byte aligned base, for a ring of kStages boxes.
template <int kStages>
struct SgLayout {
  static constexpr int kPrefetchPages = 2 * kStages;  // into L2 before the grid wait
  static constexpr int kOffRing = 0;
  static constexpr int kOffQ = kOffRing + kStages * kSgBoxBytes;
  static constexpr int kOffArow = kOffQ + kSegMax * kQBytes;
  static constexpr int kOffXch = kOffArow + kSegMax * kSgWarps * 32 * 8;
  static constexpr int kOffBars = kOffXch + kSgWarps * kXchFloats * 4;
  static constexpr int kNumBars = kStages + 1;  // full[stages], q copies
  static constexpr int kOffCounters = kOffBars + 8 * kNumBars;  // done[], last_issued[]
  static constexpr int kOffSegs = (kOffCounters + 8 * kStages + 15) & ~15;
  static constexpr int kOffPages = kOffSegs + kSegMax * kPlanSegWords * 4;
  static_assert(kOffBars % 8 == 0 && kOffSegs % 16 == 0, "shared-memory alignment");
  static constexpr size_t smem_bytes(int pages) {
    return 1024 /* alignment slack */ + kOffPages + static_cast<size_t>(pages) * 4;
  }
};
static_assert(2 * (1024 + SgLayout<kSgStages>::kOffPages + 4 * 256 + 1024) <= 228 * 1024,
              "two CTAs per SM for CTAs of up to 256 pages");
// Beside one shared-prefix CTA, for CTAs of any size up to kSegMaxPages pages.
static_assert(SgLayout<kSgBesideStages>::smem_bytes(kSegMaxPages) + 1024 + kSharedBesideSmemMax <=
                  228 * 1024,
              "a beside CTA fits next to a shared-prefix CTA");
static_assert(2 * (SgLayout<kSgBesideStages>::smem_bytes(0) + 1024) > 228 * 1024,
              "beside CTAs run one per SM");

// 4-D tiled copy of one whole page (coordinates {0, 0, 0, page}).
__device__ __forceinline__ void tma_load_page(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                              int page, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%3, %3, %3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(bar), "r"(0), "r"(page), "l"(policy)
      : "memory");
}

// Before griddepcontrol.wait: prefetch into L2 the first pages of the CTA's
// first segment `seg` (plan data, read before the wait: a plan is filled by a
// copy, never by a kernel, so it is complete before this grid starts).  The
// block-table entries read here may still be being written by the previous
// grid, so they only serve as prefetch addresses (L1-bypassing loads, every
// index range-checked, nothing recorded); the kernel reads them again after
// the wait.
__device__ __forceinline__ void prefetch_first_pages(const CUtensorMap* map, const AttnArgs& a,
                                                     int tid, int4 seg, int pages) {
  if (tid >= pages) return;
  const int b = seg.x, p = seg.z + tid;
  if (tid < seg.w && b >= 0 && b < a.batch && p >= 0 && p < a.max_blocks) {
    const int pid = ld_cg(a.block_table + static_cast<int64_t>(b) * a.max_blocks + p);
    if (pid >= 0 && pid < a.num_pages) tma_prefetch_l2_4d(map, 0, 0, 0, pid);
  }
}

template <bool kAppend, int kStages, bool kBeside>
__global__ void __launch_bounds__(kSgThreads, 2)
    paged_decode_segments_kernel(const __grid_constant__ CUtensorMap page_map, const AttnArgs a,
                                 const AppendArgs ap) {
  using Ly = SgLayout<kStages>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t ring0 = sb + Ly::kOffRing;
  const uint32_t full0 = sb + Ly::kOffBars;                      // full[stage]
  const uint32_t qbar = sb + Ly::kOffBars + 8 * kStages;       // the q copies
  int32_t* done = reinterpret_cast<int32_t*>(smem + Ly::kOffCounters);  // warps done per stage
  int32_t* last_issued = done + kStages;  // the last page each stage was given (-1: none)
  int4* s_segs = reinterpret_cast<int4*>(smem + Ly::kOffSegs);
  int32_t* s_pages = reinterpret_cast<int32_t*>(smem + Ly::kOffPages);
  AppendRow* s_arow = reinterpret_cast<AppendRow*>(smem + Ly::kOffArow);  // [seg][warp][lane]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int g = tid >> 5;  // this warp's kv head
  if (tid == 0) tma_prefetch_desc(&page_map);

  // ---- this CTA's segments {b, L, p_begin, n, slot, fold, fold_slot, 0},
  // and the barriers, before the grid wait (plan data: complete before this
  // grid starts)
  const int4 head = a.plan_items[static_cast<int64_t>(blockIdx.x) * (kPlanItemWords / 4)];
  const int first = head.y, nseg = head.z, total = head.w;
  if (tid < 2 * nseg)
    s_segs[tid] = a.plan_segs[static_cast<int64_t>(first) * (kPlanSegWords / 4) + tid];
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      done[s] = 0;
      last_issued[s] = -1;
    }
    mbar_init(qbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  prefetch_first_pages(&page_map, a, tid, s_segs[0], Ly::kPrefetchPages);
  if constexpr (!kBeside) {
    wait_for_prior_grids();
  } else {
    // Beside the shared-prefix grid launched just before: everything that
    // grid waited for has completed (its CTAs let this grid launch only after
    // their own wait), so the inputs read below -- q, k_new, v_new, the
    // tables, the lengths and the members' own pages -- are final.  That grid
    // writes only its partial slots and reads only shared pages, which are
    // never a member's last page; so this CTA streams its pages, appends its
    // token and writes outputs and its own partials without waiting, and
    // waits for it only before folding its partials.
  }
  allow_dependent_grids();
  const int Lmax = a.max_blocks * kPageSize;
  auto seg_b = [&](int s) { return s_segs[2 * s].x; };
  auto seg_L = [&](int s) { return min(max(s_segs[2 * s].y, 0), Lmax); };
  auto seg_p0 = [&](int s) { return s_segs[2 * s].z; };
  auto seg_n = [&](int s) { return s_segs[2 * s].w; };
  auto seg_slot = [&](int s) { return s_segs[2 * s + 1].x; };
  auto seg_fold = [&](int s) { return s_segs[2 * s + 1].y; };
  auto seg_fold_slot = [&](int s) { return s_segs[2 * s + 1].z; };

  // page ids of the concatenated segments
  for (int i = tid; i < total; i += kSgThreads) {
    int s = 0, off = 0;
    while (s + 1 < nseg && i >= off + seg_n(s)) off += seg_n(s++);
    int32_t pid = a.block_table[static_cast<int64_t>(seg_b(s)) * a.max_blocks + seg_p0(s) +
                                (i - off)];
    if (pid < 0 || pid >= a.num_pages) {
      record_error(a.dev_err, kErrPage);
      pid = -1;
    }
    s_pages[i] = pid;
  }
  // the lengths come from the plan; seq_lens is only compared with them
  if (tid < nseg && a.seq_lens[seg_b(tid)] != s_segs[2 * tid].y) record_error(a.dev_err, kErrPlan);
  __syncthreads();

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int k) {  // one thread
    const int st = k % kStages;
    const int pid = s_pages[k];
    const uint32_t bar = full0 + 8 * st;
    last_issued[st] = k;
    if (pid >= 0) {
      mbar_arrive_expect_tx(bar, kSgBoxBytes);
      tma_load_page(ring0 + st * kSgBoxBytes, &page_map, bar, pid, policy);
    } else {
      mbar_arrive(bar);  // keep the stage's phase sequence in step
    }
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(qbar, nseg * kQBytes);
    for (int s = 0; s < nseg; ++s)
      bulk_load(sb + Ly::kOffQ + s * kQBytes, a.q + static_cast<int64_t>(seg_b(s)) * (kQBytes / 2),
                kQBytes, qbar, policy);
    for (int k = 0; k < kStages && k < total; ++k) issue(k);
  }

  // ---- fused append: every warp computes its head's row of each segment
  // that holds its sequence's last page, writes it to the pool and keeps it
  // for the patch of that page's tile
  if (kAppend) {
    int off = 0;
    for (int s = 0; s < nseg; ++s) {
      const int L = seg_L(s), p0 = seg_p0(s), n = seg_n(s);
      const int last = (L + kPageSize - 1) / kPageSize - 1;  // the sequence's last page
      if (L > 0 && last >= p0 && last < p0 + n) {
        const int64_t src = (static_cast<int64_t>(seg_b(s)) * kNumKvHeads + g) * kHeadDim;
        const AppendRow r = make_append_row(ap.k_new + src, ap.v_new + src, L - 1, ap.freqs, lane);
        const int pid = s_pages[off + last - p0];
        if (pid >= 0) store_append_row(ap.pool, pid, (L - 1) % kPageSize, g, r, lane);
        s_arow[(s * kSgWarps + g) * 32 + lane] = r;
      }
      off += n;
    }
  }

  const LaneGeom G(lane);
  const float c = a.scale_log2;
  float* xch = reinterpret_cast<float*>(smem + Ly::kOffXch) + g * kXchFloats;
  bool ok = __all_sync(kFullMask, mbar_wait_bounded(qbar, 0, a.wait_ns));
  if (!ok && lane == 0) record_error(a.dev_err, kErrTimeout);

  int k = 0;  // position in the CTA's page list
  for (int s = 0; s < nseg; ++s) {
    const int L = seg_L(s), p0 = seg_p0(s), n = seg_n(s);
    const int last = (L + kPageSize - 1) / kPageSize - 1;
    AttnState S;
    S.reset();
    if (ok) {
      uint32_t qb[4][2];
      load_q_frags(reinterpret_cast<const uint16_t*>(smem + Ly::kOffQ + s * kQBytes) +
                       g * kGroup * kHeadDim, G, qb);
      for (int i = 0; i < n; ++i, ++k) {
        const int st = k % kStages;
        const bool ready = mbar_wait_bounded(full0 + 8 * st, (k / kStages) & 1, a.wait_ns);
        if (!__all_sync(kFullMask, ready)) {
          // stop; this warp never releases stage st again, so the other
          // warps time out on it in turn, and the copies still in flight are
          // drained below
          if (lane == 0) record_error(a.dev_err, kErrTimeout);
          ok = false;
          break;
        }
        if (s_pages[k] >= 0) {
          const uint32_t kt = ring0 + st * kSgBoxBytes + g * kTileBytes;
          if (kAppend && p0 + i == last)
            patch_append_row(kt, (L - 1) % kPageSize, s_arow[(s * kSgWarps + g) * 32 + lane],
                             lane);
          const int valid = min(kPageSize, L - (p0 + i) * kPageSize);
          attend_page(kt, valid, qb, c, G, lane, S);
        }
        __syncwarp();
        if (lane == 0) {
          // release the stage; the last of the 8 warps refills it
          __threadfence_block();
          if (atomicAdd(done + st, 1) == kSgWarps - 1) {
            done[st] = 0;
            __threadfence_block();
            if (k + kStages < total) {
              fence_proxy_async_smem();
              issue(k + kStages);
            }
          }
        }
      }
    }
    // ---- the segment's rows (after a timeout: whatever this warp has, or
    // zero rows, so that every output is written and finite)
    reduce_row_sums(S);
    if (G.ft < 2) {
      if (G.fg == 0) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          xch[2 * G.ft + rr] = S.m_ref[rr];
          xch[kGroup + 2 * G.ft + rr] = S.l_run[rr];
        }
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        float* o0 = xch + 2 * kGroup + (2 * G.ft) * kHeadDim + 16 * mt + G.fg;
        o0[0] = S.oacc[mt][0];
        o0[kHeadDim] = S.oacc[mt][1];
        o0[8] = S.oacc[mt][2];
        o0[kHeadDim + 8] = S.oacc[mt][3];
      }
    }
    __syncwarp();
    const int b = seg_b(s), slot = seg_slot(s), nf = seg_fold(s);
    const int d = 2 * lane;
    float Mr[kGroup], Lr[kGroup];
    float2 Or[kGroup];
#pragma unroll
    for (int r = 0; r < kGroup; ++r) {
      Mr[r] = xch[r];
      Lr[r] = Mr[r] == -INFINITY ? 0.f : xch[kGroup + r];
      Or[r] = Mr[r] == -INFINITY ? make_float2(0.f, 0.f)
                                 : *reinterpret_cast<const float2*>(
                                       xch + 2 * kGroup + r * kHeadDim + d);
    }
    if (nf > 0) {
      // fold in the partials of the sequence's shared ranges (slots
      // fold_slot.., written by the shared-prefix kernel, which ended before
      // this grid's wait returned), in slot order, then this segment's own
      // rows, by an online combine; two slots' loads for all 4 rows are in
      // flight at once
      if constexpr (kBeside) wait_for_prior_grids();
      float Mx[kGroup], Lf[kGroup];
      float2 Of[kGroup];
#pragma unroll
      for (int r = 0; r < kGroup; ++r) {
        Mx[r] = -INFINITY;
        Lf[r] = 0.f;
        Of[r] = make_float2(0.f, 0.f);
      }
      auto combine = [&](int r, float m, float l, float2 o) {
        if (!(l > 0.f)) return;
        const float mn = fmaxf(Mx[r], m);
        const float sc = Mx[r] == -INFINITY ? 0.f : fast_exp2(Mx[r] - mn);
        const float w = fast_exp2(m - mn);
        Lf[r] = fmaf(l, w, Lf[r] * sc);
        Of[r].x = fmaf(w, o.x, Of[r].x * sc);
        Of[r].y = fmaf(w, o.y, Of[r].y * sc);
        Mx[r] = mn;
      };
      const int64_t p0 = static_cast<int64_t>(seg_fold_slot(s)) * kNumQHeads + g * kGroup;
      for (int f = 0; f < nf; f += 2) {
        float2 ml[2][kGroup], acc[2][kGroup];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int r = 0; r < kGroup; ++r) {
            const int64_t part = p0 + static_cast<int64_t>(f + u) * kNumQHeads + r;
            const bool has = f + u < nf;
            ml[u][r] = has ? __ldcg(reinterpret_cast<const float2*>(a.part_ml + part * 2))
                           : make_float2(-INFINITY, 0.f);
            acc[u][r] = has ? __ldcg(reinterpret_cast<const float2*>(
                                  a.part_acc + part * kHeadDim + d))
                            : make_float2(0.f, 0.f);
          }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int r = 0; r < kGroup; ++r) combine(r, ml[u][r].x, ml[u][r].y, acc[u][r]);
      }
#pragma unroll
      for (int r = 0; r < kGroup; ++r) {
        combine(r, Mr[r], Lr[r], Or[r]);
        Mr[r] = Mx[r];
        Lr[r] = Lf[r];
        Or[r] = Of[r];
      }
    }
#pragma unroll
    for (int r = 0; r < kGroup; ++r) {
      const float M = Mr[r], Ls = Lr[r];
      const float2 O = Or[r];
      if (slot < 0) {
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const uint32_t v = static_cast<uint32_t>(float_to_bf16_rne(O.x * inv)) |
                           (static_cast<uint32_t>(float_to_bf16_rne(O.y * inv)) << 16);
        const int64_t row = static_cast<int64_t>(b) * kNumQHeads + g * kGroup + r;
        *reinterpret_cast<uint32_t*>(a.out + row * kHeadDim + d) = v;
      } else {
        const int64_t part = static_cast<int64_t>(slot) * kNumQHeads + g * kGroup + r;
        *reinterpret_cast<float2*>(a.part_acc + part * kHeadDim + d) = O;
        if (lane == 0) *reinterpret_cast<float2*>(a.part_ml + part * 2) = make_float2(M, Ls);
      }
    }
    __syncwarp();  // the exchange area is reused by the next segment
  }

  // ---- before the CTA exits, every copy it issued has landed: after a
  // timeout the last page each stage was given may still be in flight (a
  // stage is refilled only once every warp released its previous page, so it
  // is the only one that can be), waited for by the full limit; the q copies
  // likewise
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s)
      if (last_issued[s] >= 0) mbar_wait_bounded(full0 + 8 * s, (last_issued[s] / kStages) & 1);
    mbar_wait_bounded(qbar, 0);
  }
  // Beside: no CTA ends before the shared-prefix grid has, even one that
  // folds nothing, so that this grid's completion -- what the next launch
  // (the merge, or the next layer) waits for -- covers that grid's partials
  // and its use of the workspace too.
  if constexpr (kBeside) wait_for_prior_grids();
}

template <bool kAppend, int kStages, bool kBeside>
cudaError_t configure_sg_once(int device) {
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (device & 63);
  if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(
      paged_decode_segments_kernel<kAppend, kStages, kBeside>,
      cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(SgLayout<kStages>::smem_bytes(kSegMaxPages)));
  if (err != cudaSuccess) return err;
  if (kBeside) {
    // one L1 / shared-memory split for both kernels of the beside layout
    // (CTAs of two kernels share an SM only under the same split)
    err = cudaFuncSetAttribute(paged_decode_segments_kernel<kAppend, kStages, kBeside>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
  }
  configured.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <bool kAppend, int kStages, bool kBeside>
cudaError_t launch_sg(const CUtensorMap& page_map, const AttnArgs& args, const AppendArgs& ap,
                      int num_items, int max_pages, cudaStream_t stream) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  err = configure_sg_once<kAppend, kStages, kBeside>(device);
  if (err != cudaSuccess) return err;
  return launch_pdl(paged_decode_segments_kernel<kAppend, kStages, kBeside>, dim3(num_items),
                    dim3(kSgThreads), SgLayout<kStages>::smem_bytes(max_pages), stream,
                    page_map, args, ap);
}

}  // namespace

cudaError_t launch_segments_attention(const CUtensorMap& page_map, const AttnArgs& args,
                                      int num_items, int max_pages, cudaStream_t stream,
                                      const AppendArgs* append, bool beside) {
  if (num_items < 1 || max_pages < 1 || max_pages > kSegMaxPages) return cudaErrorInvalidValue;
  const AppendArgs none{};
  if (beside)
    return append != nullptr
               ? launch_sg<true, kSgBesideStages, true>(page_map, args, *append, num_items,
                                                        max_pages, stream)
               : launch_sg<false, kSgBesideStages, true>(page_map, args, none, num_items,
                                                         max_pages, stream);
  return append != nullptr
             ? launch_sg<true, kSgStages, false>(page_map, args, *append, num_items, max_pages,
                                                 stream)
             : launch_sg<false, kSgStages, false>(page_map, args, none, num_items, max_pages,
                                                  stream);
}

}  // namespace pkv
