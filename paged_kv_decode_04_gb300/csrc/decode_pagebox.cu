// decode_pagebox.cu -- paged decode attention with one CTA per (sequence,
// range) covering all kv heads: each page arrives as one 32 KiB TMA box.
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗", paged decode attention
// item: every query head streams its own sequence's cached pages with an FP32
// online softmax, never gathering a contiguous prefix or storing scores.
//
// Why a second decomposition: the per-(sequence, kv head) kernel fetches a
// page as 8 boxes of 4 KiB (one per head, from 8 CTAs).  Streaming the same
// pool with one 32 KiB box per page measured 4-6 % faster on this part (the
// copy engine's cost is per box, and DRAM sees each page requested at once);
// with the math, 2.8 % on 256 x 2048 tokens and 6 % on the prefix-shared
// batch.  Batches with at least one CTA per SM use this kernel.
//
// Layout: the pool is viewed as a 4-D tensor (dim, row, head, page) with
// strides (2 B, 1 KiB, 128 B, 32 KiB), so the box {64, 32, 8, 1} lands in
// shared memory as [head][32 rows][64] -- each head's 4 KiB sub-tile is
// exactly the 128-byte-swizzled tile the per-page math of decode_page.cuh
// expects.
//
// Roles: warp g (8 warps) attends kv head g over every page of the CTA's
// range, holding its 4 query rows' state to the end (no cross-warp merge).
// The CTA shares a ring of kPbStages page boxes; the last warp done with a
// stage refills it with the page kPbStages ahead (a shared counter per
// stage), so no warp waits on a CTA-wide barrier inside the loop.
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

constexpr int kPbWarps = kNumKvHeads;  // one warp per kv head
constexpr int kPbThreads = kPbWarps * 32;
// Two page boxes per CTA (2 CTAs per SM): measured faster than three on 256
// x 2048-token sequences (158.2 vs 161.3 us per step, the per-(sequence, kv
// head) kernel 162.7 us on the same box), as was a plain streaming probe of
// the same boxes.
constexpr int kPbStages = 2;
constexpr int kPageBoxBytes = kNumKvHeads * kTileBytes;  // 32 KiB
constexpr int kPbRingBytes = kPbStages * kPageBoxBytes;
// Pages prefetched into L2 before griddepcontrol.wait: twice the ring (on
// 256 x 2048-token steps: 157.7 us with 2, 156.8 with 4, 156.7 with 8).
constexpr int kPbPrefetchPages = 2 * kPbStages;
constexpr int kPbMaxPages = 1024;

static_assert(kPbWarps * (2 * kGroup + kGroup * kHeadDim) * 4 <= kPbRingBytes,
              "end-of-CTA state exchange must fit in the ring");

__host__ __device__ constexpr size_t pb_smem_bytes(int range_pages) {
  return 1024 /* alignment slack */ + kPbRingBytes + 8 * kPbStages /* bars */ +
         8 * kPbStages /* counters, last pages issued */ + static_cast<size_t>(range_pages) * 4;
}

// 4-D tiled copy of one whole page (coordinates {0, 0, 0, page}).
__device__ __forceinline__ void tma_load_page(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                              int page, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%3, %3, %3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(bar), "r"(0), "r"(page), "l"(policy)
      : "memory");
}

// Before griddepcontrol.wait: prefetch into L2 the CTA's first
// kPbPrefetchPages pages (as prefetch_first_tiles does for the per-head
// kernel: the plan item, read before the wait, is plan data and complete;
// the lengths and block-table entries read here are only addresses for the
// prefetch: reads bypass L1, indices are range-checked, and they are read
// again after the wait).
template <bool kPlanned>
__device__ __forceinline__ void prefetch_first_pages(const CUtensorMap* map, const AttnArgs& a,
                                                     int tid, int4 head, int item_b) {
  int b = -1, p = -1;
  if constexpr (kPlanned) {
    if (tid < kPbPrefetchPages && tid < head.w) {
      b = item_b;
      p = head.z + tid;
    }
  } else if (tid < kPbPrefetchPages) {
    const int pps = a.plan.pages_per_split;
    const int L = ld_cg(a.seq_lens + blockIdx.y);
    const int np = (min(max(L, 0), a.max_blocks * kPageSize) + kPageSize - 1) / kPageSize;
    if (tid < pps && static_cast<int>(blockIdx.x) * pps + tid < np) {
      b = blockIdx.y;
      p = blockIdx.x * pps + tid;
    }
  }
  if (b >= 0 && b < a.batch && p >= 0 && p < a.max_blocks) {
    const int pid = ld_cg(a.block_table + static_cast<int64_t>(b) * a.max_blocks + p);
    if (pid >= 0 && pid < a.num_pages) tma_prefetch_l2_4d(map, 0, 0, 0, pid);
  }
}

template <bool kAppend, bool kPlanned>
__global__ void __launch_bounds__(kPbThreads, 2)
    paged_decode_pagebox_kernel(const __grid_constant__ CUtensorMap page_map,
                                const AttnArgs a, const AppendArgs ap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPbRingBytes);
  int32_t* done = reinterpret_cast<int32_t*>(full + kPbStages);  // warps finished per stage
  int32_t* last_issued = done + kPbStages;  // the last page each stage was given (-1: none)
  int32_t* s_pages = last_issued + kPbStages;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int g = tid >> 5;  // this warp's kv head
  if (tid == 0) tma_prefetch_desc(&page_map);
  // planned: the item {kind = range, slot, p_begin, n}, its sequence and
  // length (plan data: complete before this grid starts)
  int4 p_head = make_int4(0, 0, 0, 0);
  int p_b = -1, p_L = 0;
  if constexpr (kPlanned) {
    const int4* it = a.plan_items + static_cast<int64_t>(blockIdx.x) * (kPlanItemWords / 4);
    p_head = it[0];
    p_b = it[1].x;
    p_L = it[2].x;
  }
  prefetch_first_pages<kPlanned>(&page_map, a, tid, p_head, p_b);
  wait_for_prior_grids();
  allow_dependent_grids();

  // ---- this CTA's sequence b and logical pages [p_begin, p_begin + n)
  int b, L, p_begin, n;
  int64_t part_row0 = -1;  // partial slot of query row 4g, -1: write the output itself
  int part_step = 0;
  int dev_len = -2, plan_len = 0;  // work plan: device length read for the plan check
  const int Lmax = a.max_blocks * kPageSize;
  if constexpr (kPlanned) {
    const int4 head = p_head;  // (kind = range, slot, p_begin, n)
    b = p_b;
    L = p_L;
    plan_len = L;
    // the lengths come from the plan; seq_lens is only checked against it
    // (the load is consumed at the end of the kernel, off the critical path)
    if (g == 0 && lane == 0) dev_len = a.seq_lens[b];
    L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
    p_begin = head.z;
    n = head.w;
    if (head.y >= 0) {
      part_row0 = static_cast<int64_t>(head.y) * kNumQHeads + g * kGroup;
      part_step = 1;
    }
  } else {
    const int split = blockIdx.x;
    const int pps = a.plan.pages_per_split;
    b = blockIdx.y;
    L = a.seq_lens[b];
    if (L < 0 || L > Lmax) {
      if (tid == 0 && split == 0) record_error(a.dev_err, kErrSeqLen);
      L = L < 0 ? 0 : Lmax;
    }
    const int np = (L + kPageSize - 1) / kPageSize;
    const int nsplit = np > 0 ? (np + pps - 1) / pps : 1;
    if (split >= nsplit) return;
    p_begin = split * pps;
    n = min(pps, np - p_begin);
    if (nsplit > 1) {
      part_row0 = (static_cast<int64_t>(b) * kNumQHeads + g * kGroup) * a.plan.num_splits + split;
      part_step = a.plan.num_splits;
    }
  }
  const int npages = (L + kPageSize - 1) / kPageSize;

  for (int i = tid; i < n; i += kPbThreads) {
    int32_t pid = a.block_table[static_cast<int64_t>(b) * a.max_blocks + p_begin + i];
    if (pid < 0 || pid >= a.num_pages) {
      record_error(a.dev_err, kErrPage);
      pid = -1;
    }
    s_pages[i] = pid;
  }
  const uint32_t bar0 = smem_addr(full);
  const uint32_t ring0 = smem_addr(smem);
  if (tid == 0) {
    for (int s = 0; s < kPbStages; ++s) {
      mbar_init(bar0 + 8 * s, 1);
      done[s] = 0;
      last_issued[s] = -1;
    }
    fence_barrier_init();
  }
  __syncthreads();

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int k) {  // one thread
    const int st = k % kPbStages;
    const int pid = s_pages[k];
    const uint32_t bar = bar0 + 8 * st;
    last_issued[st] = k;
    if (pid >= 0) {
      mbar_arrive_expect_tx(bar, kPageBoxBytes);
      tma_load_page(ring0 + st * kPageBoxBytes, &page_map, bar, pid, policy);
    } else {
      mbar_arrive(bar);  // keep the stage's phase sequence in step
    }
  };
  if (tid == 0)
    for (int k = 0; k < kPbStages && k < n; ++k) issue(k);

  const LaneGeom G(lane);
  uint32_t qb[4][2];
  load_q_frags(a.q + (static_cast<int64_t>(b) * kNumQHeads + g * kGroup) * kHeadDim, G, qb);
  const float c = a.scale_log2;

  // ---- fused append: every warp writes its own head's row of the new token
  const int k_last = npages - 1 - p_begin;  // the last page's position in this range
  const bool has_last = kAppend && npages > 0 && k_last >= 0 && k_last < n;
  const int a_slot = (L - 1) % kPageSize;
  AppendRow arow{};
  if (has_last) {
    const int64_t src = (static_cast<int64_t>(b) * kNumKvHeads + g) * kHeadDim;
    arow = make_append_row(ap.k_new + src, ap.v_new + src, L - 1, ap.freqs, lane);
    const int pid = s_pages[k_last];
    if (pid >= 0) store_append_row(ap.pool, pid, a_slot, g, arow, lane);
  }

  AttnState S;
  S.reset();
  for (int k = 0; k < n; ++k) {
    const int st = k % kPbStages;
    const bool ready = mbar_wait_bounded(bar0 + 8 * st, (k / kPbStages) & 1, a.wait_ns);
    if (!__all_sync(kFullMask, ready)) {
      // stop; the copies this CTA issued are still to be drained (below).
      // This warp never releases stage st again, so the other warps time out
      // on it in turn.
      if (lane == 0) record_error(a.dev_err, kErrTimeout);
      break;
    }
    if (s_pages[k] >= 0) {
      const uint32_t kt = ring0 + st * kPageBoxBytes + g * kTileBytes;
      if (has_last && k == k_last) patch_append_row(kt, a_slot, arow, lane);
      const int valid = min(kPageSize, L - (p_begin + k) * kPageSize);
      attend_page(kt, valid, qb, c, G, lane, S);
    }
    __syncwarp();
    if (lane == 0) {
      // release the stage; the last of the 8 warps refills it
      __threadfence_block();
      if (atomicAdd(done + st, 1) == kPbWarps - 1) {
        done[st] = 0;
        __threadfence_block();
        if (k + kPbStages < n) {
          fence_proxy_async_smem();
          issue(k + kPbStages);
        }
      }
    }
  }

  // ---- each warp normalises its own 4 rows (state through shared memory,
  // once every copy of the ring has landed)
  reduce_row_sums(S);
  __syncthreads();
  if (tid == 0) {
    // after a timeout a box may still be in flight: wait (bounded by the full
    // limit) for the phase of the last page each stage was given -- a stage
    // is refilled only once every warp has released its previous page, so
    // that is its only phase that can be outstanding -- before the ring is
    // reused and the CTA exits
    for (int s = 0; s < kPbStages; ++s)
      if (last_issued[s] >= 0)
        mbar_wait_bounded(bar0 + 8 * s, (last_issued[s] / kPbStages) & 1);
  }
  __syncthreads();
  float* sm_m = reinterpret_cast<float*>(smem);
  float* sm_l = sm_m + kPbWarps * kGroup;
  float* sm_o = sm_l + kPbWarps * kGroup;
  if (G.ft < 2) {
    if (G.fg == 0) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        sm_m[g * kGroup + 2 * G.ft + rr] = S.m_ref[rr];
        sm_l[g * kGroup + 2 * G.ft + rr] = S.l_run[rr];
      }
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      float* o0 = sm_o + (g * kGroup + 2 * G.ft) * kHeadDim + 16 * mt + G.fg;
      o0[0] = S.oacc[mt][0];
      o0[kHeadDim] = S.oacc[mt][1];
      o0[8] = S.oacc[mt][2];
      o0[kHeadDim + 8] = S.oacc[mt][3];
    }
  }
  __syncwarp();
  if (kPlanned && dev_len != -2 && dev_len != plan_len) record_error(a.dev_err, kErrPlan);
  const int d = 2 * lane;
#pragma unroll
  for (int r = 0; r < kGroup; ++r) {
    const float M = sm_m[g * kGroup + r];
    const float Ls = M == -INFINITY ? 0.f : sm_l[g * kGroup + r];
    const float2 O = M == -INFINITY
                         ? make_float2(0.f, 0.f)
                         : *reinterpret_cast<const float2*>(sm_o + (g * kGroup + r) * kHeadDim + d);
    if (part_row0 < 0) {
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      const uint32_t v = static_cast<uint32_t>(float_to_bf16_rne(O.x * inv)) |
                         (static_cast<uint32_t>(float_to_bf16_rne(O.y * inv)) << 16);
      const int64_t row = static_cast<int64_t>(b) * kNumQHeads + g * kGroup + r;
      *reinterpret_cast<uint32_t*>(a.out + row * kHeadDim + d) = v;
    } else {
      const int64_t part = part_row0 + static_cast<int64_t>(r) * part_step;
      *reinterpret_cast<float2*>(a.part_acc + part * kHeadDim + d) = O;
      if (lane == 0) *reinterpret_cast<float2*>(a.part_ml + part * 2) = make_float2(M, Ls);
    }
  }
}

template <bool kAppend, bool kPlanned>
cudaError_t configure_pb_once(int device) {
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (device & 63);
  if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(
      paged_decode_pagebox_kernel<kAppend, kPlanned>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(pb_smem_bytes(kPbMaxPages)));
  if (err == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
  return err;
}

template <bool kAppend, bool kPlanned>
cudaError_t launch_pb(const CUtensorMap& page_map, const AttnArgs& args, const AppendArgs& ap,
                      dim3 grid, int range_pages, cudaStream_t stream) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  err = configure_pb_once<kAppend, kPlanned>(device);
  if (err != cudaSuccess) return err;
  return launch_pdl(paged_decode_pagebox_kernel<kAppend, kPlanned>, grid, dim3(kPbThreads),
                    pb_smem_bytes(range_pages), stream, page_map, args, ap);
}

}  // namespace

int pagebox_max_range_pages() { return kPbMaxPages; }

cudaError_t launch_pagebox_attention(const CUtensorMap& page_map, const AttnArgs& args,
                                     int num_items, int range_pages, cudaStream_t stream,
                                     const AppendArgs* append) {
  const AppendArgs none{};
  const bool planned = args.plan_items != nullptr;
  const dim3 grid = planned ? dim3(num_items)
                            : dim3(args.plan.num_splits, args.batch);
  if (append != nullptr)
    return planned ? launch_pb<true, true>(page_map, args, *append, grid, range_pages, stream)
                   : launch_pb<true, false>(page_map, args, *append, grid, range_pages, stream);
  return planned ? launch_pb<false, true>(page_map, args, none, grid, range_pages, stream)
                 : launch_pb<false, false>(page_map, args, none, grid, range_pages, stream);
}

}  // namespace pkv
