// decode_shared.cu -- paged decode attention over pages that a group of
// sequences shares (a common prompt prefix), each page read once per group.
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗": attention streams each
// sequence's cached pages with an FP32 online softmax; "Tiny-vLLMでゼロから
// 構築する高性能LLM推論エンジン", section "KV Cache": requests whose block
// tables name the same physical pages share those pages' K/V.
//
// A host work plan (planner.cpp, pkv_plan_build_shared) finds runs of
// consecutive sequences whose block tables start with the same pages and
// emits shared-prefix items: pages [p_begin, p_begin + n) common to up to 16
// members.  One CTA per (item, kv head g): warp w holds the 4 query rows of
// head g of members 2w and 2w + 1 as the 8 columns of its tensor-core tiles
// (the per-page math computes 8 query rows anyway; a group of 4 rows uses
// half of them).  The CTA streams head g's 4 KiB tile of each page once into
// a shared ring (the last warp done with a stage refills it, as in the
// whole-page kernel), and every warp folds that tile into its two members'
// online-softmax states.  Each warp then writes its members' unnormalised
// (max, sum, acc) partials to the slots the plan gives them; the members' own
// pages are attended by the ordinary planned kernels into the following
// slots, and the merge kernel combines them.  A shared page is never a
// member's last page, so every shared page is full and none takes the
// step's append.
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

constexpr int kShWarps = kSharedMembers / 2;  // warp w <-> members 2w, 2w + 1
constexpr int kShRows = 2 * kGroup;            // query rows per warp
constexpr int kShThreads = kShWarps * 32;
// Eight 4 KiB tiles in the ring (32 KiB per CTA).  Three CTAs per SM (78
// registers) against two (88): 79.3 -> 75.9 us per step on 256 x 2048
// tokens with 16-way shared 1536-token prefixes; the kernel is bound by its
// per-page math, so more resident warps help.
constexpr int kShStages = 8;
constexpr int kShCtasPerSm = kSharedCtasPerSm;
constexpr int kShRingBytes = kShStages * kTileBytes;
constexpr int kShMaxPages = 1024;

static_assert(kShWarps * (2 * kShRows + kShRows * kHeadDim) * 4 <= kShRingBytes,
              "end-of-CTA scratch must fit in the ring");

__host__ __device__ constexpr size_t sh_smem_bytes(int pages) {
  return 1024 /* alignment slack */ + kShRingBytes + 8 * kShStages /* bars */ +
         4 * kShStages /* counters */ + static_cast<size_t>(pages) * 4;
}

// Q^T of two members as the B operand of S^T = K Q^T: columns 0..3 are
// member a's 4 rows, 4..7 member b's (qa / qb: their [4][64] bf16 rows, or
// nullptr for zeros).
__device__ __forceinline__ void load_q_frags_pair(const uint16_t* qa, const uint16_t* qb,
                                                  const LaneGeom& G, uint32_t (&f)[4][2]) {
  const uint16_t* base = G.fg < kGroup ? qa : qb;
  const uint32_t* qw =
      base != nullptr ? reinterpret_cast<const uint32_t*>(base + (G.fg & 3) * kHeadDim) : nullptr;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    f[kk][0] = qw != nullptr ? qw[kk * 8 + G.ft] : 0u;
    f[kk][1] = qw != nullptr ? qw[kk * 8 + 4 + G.ft] : 0u;
  }
}

__global__ void __launch_bounds__(kShThreads, kShCtasPerSm)
    paged_decode_shared_kernel(const __grid_constant__ CUtensorMap pool_map, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kShRingBytes);
  int32_t* done = reinterpret_cast<int32_t*>(full + kShStages);  // warps finished per stage
  int32_t* s_pages = done + kShStages;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;  // this warp's members: 2 warp, 2 warp + 1
  const int g = blockIdx.x;   // kv head
  if (tid == 0) tma_prefetch_desc(&pool_map);
  wait_for_prior_grids();
  allow_dependent_grids();

  // ---- the item: {members, p_begin, n, 0, seq[16], slot[16]}
  const int32_t* it = reinterpret_cast<const int32_t*>(a.plan_shared) +
                      static_cast<int64_t>(blockIdx.y) * kPlanSharedWords;
  const int members = it[0], p_begin = it[1], n = it[2];
  const int leader = it[4];
  int mseq[2], mslot[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = 2 * warp + h;
    mseq[h] = m < members ? it[4 + m] : -1;
    mslot[h] = m < members ? it[4 + kSharedMembers + m] : -1;
  }

  // page ids: the leader's table (every member's holds the same ones here)
  for (int i = tid; i < n; i += kShThreads) {
    int32_t pid = a.block_table[static_cast<int64_t>(leader) * a.max_blocks + p_begin + i];
    if (pid < 0 || pid >= a.num_pages) {
      record_error(a.dev_err, kErrPage);
      pid = -1;
    }
    s_pages[i] = pid;
  }
  const uint32_t bar0 = smem_addr(full);
  const uint32_t ring0 = smem_addr(smem);
  if (tid == 0) {
    for (int s = 0; s < kShStages; ++s) {
      mbar_init(bar0 + 8 * s, 1);
      done[s] = 0;
    }
    fence_barrier_init();
  }
  __syncthreads();

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int k) {  // one thread
    const int st = k % kShStages;
    const int pid = s_pages[k];
    const uint32_t bar = bar0 + 8 * st;
    if (pid >= 0) {
      mbar_arrive_expect_tx(bar, kTileBytes);
      tma_load_3d(ring0 + st * kTileBytes, &pool_map, bar, g * kHeadDim, 0, pid, policy);
    } else {
      mbar_arrive(bar);  // keep the stage's phase sequence in step
    }
  };
  if (tid == 0)
    for (int k = 0; k < kShStages && k < n; ++k) issue(k);

  const LaneGeom G(lane);
  uint32_t qb[4][2];
  auto qrows = [&](int seq) {
    return seq >= 0 ? a.q + (static_cast<int64_t>(seq) * kNumQHeads + g * kGroup) * kHeadDim
                    : nullptr;
  };
  load_q_frags_pair(qrows(mseq[0]), qrows(mseq[1]), G, qb);
  const float c = a.scale_log2;

  AttnState S;
  S.reset();
  for (int k = 0; k < n; ++k) {
    const int st = k % kShStages;
    const bool ready = mbar_wait_bounded(bar0 + 8 * st, (k / kShStages) & 1);
    if (!__all_sync(kFullMask, ready)) {
      // stop; the copies this CTA issued are still to be drained (below)
      if (lane == 0) record_error(a.dev_err, kErrTimeout);
      break;
    }
    if (mseq[0] >= 0 && s_pages[k] >= 0)
      attend_page(ring0 + st * kTileBytes, kPageSize, qb, c, G, lane, S);
    __syncwarp();
    if (lane == 0) {
      // release the stage; the last of the warps refills it
      __threadfence_block();
      if (atomicAdd(done + st, 1) == kShWarps - 1) {
        done[st] = 0;
        __threadfence_block();
        if (k + kShStages < n) {
          fence_proxy_async_smem();
          issue(k + kShStages);
        }
      }
    }
  }

  // ---- each warp writes its members' partials (state through shared
  // memory, once every copy of the ring has landed)
  reduce_row_sums(S);
  __syncthreads();
  if (tid == 0) {
    // after a timeout some tiles may still be in flight: wait for each
    // stage's outstanding phase (bounded) before the ring is reused
    for (int s = 0; s < kShStages && s < n; ++s) {
      const int last_k = s + ((n - 1 - s) / kShStages) * kShStages;  // last page of stage s
      mbar_wait_bounded(bar0 + 8 * s, (last_k / kShStages) & 1);
    }
  }
  __syncthreads();
  if (mseq[0] < 0) return;
  float* sm_m = reinterpret_cast<float*>(smem);
  float* sm_l = sm_m + kShWarps * kShRows;
  float* sm_o = sm_l + kShWarps * kShRows;
  if (G.fg == 0) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      sm_m[warp * kShRows + 2 * G.ft + rr] = S.m_ref[rr];
      sm_l[warp * kShRows + 2 * G.ft + rr] = S.l_run[rr];
    }
  }
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    float* o0 = sm_o + (warp * kShRows + 2 * G.ft) * kHeadDim + 16 * mt + G.fg;
    o0[0] = S.oacc[mt][0];
    o0[kHeadDim] = S.oacc[mt][1];
    o0[8] = S.oacc[mt][2];
    o0[kHeadDim + 8] = S.oacc[mt][3];
  }
  __syncwarp();
  const int d = 2 * lane;
#pragma unroll
  for (int r = 0; r < kShRows; ++r) {
    const int h = r / kGroup;  // member 2 warp + h
    if (mseq[h] < 0) continue;
    const float M = sm_m[warp * kShRows + r];
    const float Ls = M == -INFINITY ? 0.f : sm_l[warp * kShRows + r];
    const float2 O = M == -INFINITY ? make_float2(0.f, 0.f)
                                    : *reinterpret_cast<const float2*>(
                                          sm_o + (warp * kShRows + r) * kHeadDim + d);
    const int64_t part = static_cast<int64_t>(mslot[h]) * kNumQHeads + g * kGroup + (r & 3);
    *reinterpret_cast<float2*>(a.part_acc + part * kHeadDim + d) = O;
    if (lane == 0) *reinterpret_cast<float2*>(a.part_ml + part * 2) = make_float2(M, Ls);
  }
}

cudaError_t configure_sh_once(int device) {
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (device & 63);
  if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t err =
      cudaFuncSetAttribute(paged_decode_shared_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sh_smem_bytes(kShMaxPages)));
  if (err == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
  return err;
}

}  // namespace

cudaError_t launch_shared_prefix_attention(const CUtensorMap& pool_map, const AttnArgs& args,
                                           int num_shared, int range_pages, cudaStream_t stream) {
  if (num_shared < 1 || range_pages < 1 || range_pages > kShMaxPages) return cudaErrorInvalidValue;
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  err = configure_sh_once(device);
  if (err != cudaSuccess) return err;
  return launch_pdl(paged_decode_shared_kernel, dim3(kNumKvHeads, num_shared), dim3(kShThreads),
                    sh_smem_bytes(range_pages), stream, pool_map, args);
}

}  // namespace pkv
