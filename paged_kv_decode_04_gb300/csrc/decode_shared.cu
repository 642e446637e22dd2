// decode_shared.cu -- paged decode attention over pages that a group of
// sequences shares (a common prompt prefix), each page read once per group,
// on the fifth-generation tensor cores (tcgen05, accumulators in TMEM).
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
// members.  One CTA per (item, kv head g).  The members' 4 query rows of head
// g stack into 64 rows, so a batch of 4 pages (64 tokens) is two small dense
// contractions, run by tcgen05.mma with M = 128 and the A operand in TMEM:
//
//   S = Q K^T   (128 x 64 tokens, K = 64 head dims: 4 MMAs; Q in TMEM, the
//                batch's K rows in shared memory)
//   O += P V    (128 x 64 dims, K = 16 tokens per MMA: 2 per page, P as hi
//                and lo bf16 terms in TMEM, V rows in shared memory)
//
// With N = 64 an MMA whose A operand came from shared memory would spend most
// of its time re-reading A; from TMEM only B is read.
//
// Rows 0..63 and 64..127 hold the same 64 query rows.  The two copies split
// each batch's tokens: a row of the upper half weighs pages 0, 1 of the
// batch, its copy in the lower half pages 2, 3 (its P is zero elsewhere),
// each with its own online-softmax state and O row; the two are combined at
// the end like two split-K partials.  So all four softmax warps work (TMEM
// lane 32w + i belongs to warp w), on 32 scores each.
//
// TMEM (256 columns): X0 = 0..63 and X1 = 64..127 take S_b for batches
// b = 0, 1 mod 2 and then, written over it by the softmax, P_b (hi for page p
// in columns 8p..8p+7, lo in 32 + 8p..); O = 128..191; Q = 192..223.
//
// Roles (8 warps; one thread of each of warps 4..7 works):
//   warp 6: K producer.  Per batch, head g's K rows of its 4 pages into one
//     8 KiB region (64 rows: the N = 64 K-major B operand of S), in a ring of
//     5 regions freed as soon as the batch's S has been computed.
//   warp 7: V producer.  The V rows likewise into a ring of 5 regions (four
//     MN-major B operands of PV), freed once the batch's PV is done.  Both
//     128B-swizzled by TMA, which is the operand layout the MMA reads.
//   warp 5: issues S_b = Q K_b^T into X(b mod 2) once K_b has landed and
//     PV_{b-2} (which read P_{b-2} from there) is done.
//   warp 4: allocates the TMEM and issues PV_j once P_j is written and V_j
//     has landed.
//   warps 0..3: the softmax, thread = TMEM lane = MMA row.  Per batch: wait
//     for S_j, read the row's 32 scores, take the FP32 online-softmax step (a
//     lazily updated reference maximum), and write P_j as hi = bf16(p) and
//     lo = bf16(p - hi) (about 16 significant bits together) over S_j.  Only
//     when the maximum moves does the row wait for PV_{j-1} and rescale its O
//     row in TMEM.  At the end each query row's (max, sum, acc) partial,
//     unnormalised, goes to the slot the plan gives its member; the members'
//     own pages are attended by the ordinary planned kernels into the
//     following slots, and the merge kernel (or the member's own segment)
//     combines them.  In the plan's beside layout the CTAs take smaller K
//     and V rings (kSlotsBeside), one per SM, and the segment kernel's CTAs
//     run next to them.
// A shared page is never a member's last page, so every shared page is full
// and none takes the step's append.  Every wait is bounded: a wait on
// another role's progress by the call's limit (2 s unless the caller set
// another, pkv_set_wait_limit_ns); past it the kernel records
// PKV_DEVERR_TIMEOUT, lets its outstanding copies and MMAs finish (waits
// bounded by the full 2 s), frees its TMEM and returns.
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

constexpr int kTcRows = kSharedMembers * kGroup;  // 64 query rows
constexpr int kTcM = 2 * kTcRows;                 // MMA rows: two copies
constexpr int kTcBatch = 4;                       // pages per S / P batch
constexpr int kTcCols = kTcBatch * kPageSize;     // 64 score columns per S
constexpr int kTcHalfCols = kTcCols / 2;          // a row's share of them
constexpr int kSlotsSequential = 5;  // K (and V) regions in flight, two CTAs per SM
constexpr int kSlotsBeside = 3;      // the same beside a segment CTA (one per SM)
constexpr int kTcSoftmaxWarps = 4;
constexpr int kPvWarp = 4;
constexpr int kSWarp = 5;
constexpr int kKLoadWarp = 6;
constexpr int kVLoadWarp = 7;
constexpr int kTcThreads = 32 * (kTcSoftmaxWarps + 4);
constexpr int kTcCtasPerSm = kSharedCtasPerSm;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemO = 2 * kTcCols;           // X0: 0, X1: 64, O: 128
constexpr uint32_t kTmemQ = kTmemO + kHeadDim;     // Q: 192 (32 columns)
constexpr uint32_t kPLo = kTcHalfCols;             // P lo terms: X + 32
constexpr int kMaxPagesPerItem = 1024;

// Shared memory, from a 1024-byte aligned base.
constexpr int kHalfTileBytes = kPageSize * kRowBytes;    // 2 KiB: one head's K (or V) rows
constexpr int kRegionBytes = kTcBatch * kHalfTileBytes;  // 8 KiB: a batch's K (or V) rows
constexpr int kPrefetchBatches = 4;  // pulled into L2 before the grid dependency wait
constexpr int kXchStride = kHeadDim + 4;  // floats per exchanged row: acc, then (m, l), 16-B aligned

// Shared memory, from a 1024-byte aligned base, for rings of kSlots K and
// kSlots V regions.
template <int kSlots>
struct ShLayout {
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kSlots * kRegionBytes;
  static constexpr int kOffBars = kOffV + kSlots * kRegionBytes;
  // k_full[kSlots], k_empty[kSlots], v_full[kSlots], v_empty[kSlots],
  // s_ready[2], x_free[2], p_ready[2], pv_done, s_fin, pv_fin, q_ready
  static constexpr int kNumBars = 4 * kSlots + 10;
  static constexpr int kOffTmemSlot = kOffBars + 8 * kNumBars;
  static constexpr int kOffPages = kOffTmemSlot + 16;
  static_assert(kTcRows * kXchStride * 4 <= kSlots * kRegionBytes, "end-of-CTA exchange fits");
  static constexpr size_t smem_bytes(int pages) {
    return 1024 /* alignment slack */ + kOffPages + static_cast<size_t>(pages) * 4;
  }
};

static_assert(kTcM == 128 && 32 * kTcSoftmaxWarps == kTcM, "one softmax thread per TMEM lane");
static_assert(kTmemQ + kHeadDim / 2 <= kTmemCols, "X0, X1, O and Q fit the allocation");
// In the sequential layout shared memory alone keeps more than
// kTcCtasPerSm CTAs of this kernel off one SM (228 KiB per SM, 1 KiB
// reserved per CTA), so their TMEM allocations always fit the 512 columns
// and tcgen05.alloc never waits.  Beside a segment CTA the smaller rings
// leave that to registers, which the launch checks (sh_occupancy_ok).
static_assert((kTcCtasPerSm + 1) * (ShLayout<kSlotsSequential>::kOffPages + 1024 + 1024) >
                  228 * 1024,
              "at most kTcCtasPerSm CTAs per SM");
static_assert(kTcCtasPerSm * kTmemCols <= 512, "TMEM columns of the resident CTAs");
static_assert(kTcCtasPerSm * (ShLayout<kSlotsSequential>::kOffPages + 1024 + 1024 + 4 * 64) <=
                  228 * 1024,
              "kTcCtasPerSm CTAs per SM fit for ranges of up to 64 pages");
static_assert(ShLayout<kSlotsBeside>::smem_bytes(kMaxPagesPerItem) + 1024 <= kSharedBesideSmemMax,
              "a beside segment CTA fits next to any beside shared-prefix CTA");

constexpr uint32_t kIdescS = tc_idesc_bf16(kTcM, kTcCols, false);   // K: K-major
constexpr uint32_t kIdescPV = tc_idesc_bf16(kTcM, kHeadDim, true);  // V: MN-major

// Before the grid dependency wait: pull the first kPrefetchBatches batches'
// K and V rows of pages [p_begin, p_begin + n) of the leader's table into
// L2.  The item (plan data) is complete before this grid starts; the
// leader's table entries read here may still be being written by the
// previous grid, so they serve only as prefetch addresses (L1-bypassing
// loads, every index range-checked, nothing recorded), and the kernel reads
// them again after the wait.
__device__ __forceinline__ void prefetch_first_batches(const CUtensorMap* map, const AttnArgs& a,
                                                       int g, int tid, int p_begin, int n,
                                                       int leader) {
  constexpr int kPages = kPrefetchBatches * kTcBatch;
  if (tid >= 2 * kPages) return;
  const int i = tid >> 1;            // page of the range; even tid: K rows, odd: V rows
  if (i < n && leader >= 0 && leader < a.batch && p_begin >= 0 && p_begin + i < a.max_blocks) {
    const int pid = ld_cg(a.block_table + static_cast<int64_t>(leader) * a.max_blocks + p_begin + i);
    if (pid >= 0 && pid < a.num_pages)
      tma_prefetch_l2_3d(map, g * kHeadDim, (tid & 1) ? kPageSize : 0, pid);
  }
}

// Named barrier of the softmax warps (id 1; 0 is __syncthreads).
__device__ __forceinline__ void softmax_warps_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kTcSoftmaxWarps) : "memory");
}

template <int kSlots>
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
    paged_decode_shared_kernel(const __grid_constant__ CUtensorMap half_map, const AttnArgs a) {
  using Ly = ShLayout<kSlots>;
  constexpr int kKSlots = kSlots, kVSlots = kSlots;
  constexpr int kOffK = Ly::kOffK, kOffV = Ly::kOffV, kOffBars = Ly::kOffBars;
  constexpr int kNumBars = Ly::kNumBars, kOffTmemSlot = Ly::kOffTmemSlot;
  constexpr int kOffPages = Ly::kOffPages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_addr(smem);
  const uint32_t bars = sb + kOffBars;
  auto k_full = [&](int b) { return bars + 8u * (b % kKSlots); };
  auto k_empty = [&](int b) { return bars + 8u * (kKSlots + b % kKSlots); };
  auto v_full = [&](int b) { return bars + 8u * (2 * kKSlots + b % kVSlots); };
  auto v_empty = [&](int b) { return bars + 8u * (2 * kKSlots + kVSlots + b % kVSlots); };
  const uint32_t bars2 = bars + 8u * (2 * kKSlots + 2 * kVSlots);
  auto s_ready = [&](int b) { return bars2 + 8u * (b & 1); };
  auto x_free = [&](int b) { return bars2 + 16u + 8u * (b & 1); };
  // One p_ready per S/P buffer, like s_ready and x_free: the softmax may
  // finish batches j and j + 1 (S_{j+1} needs only PV_{j-1}) before the PV
  // issuer looks for batch j, and one barrier for all batches would then be
  // two phases ahead with batch j's parity, so its parity wait would wait
  // for batch j + 2, which needs PV_j.  Per buffer, batch j + 2 needs PV_j
  // first, so a waiter is never more than one phase behind.
  auto p_ready = [&](int j) { return bars2 + 32u + 8u * (j & 1); };
  const uint32_t pv_done = bars2 + 48u;
  const uint32_t s_fin = bars2 + 56u;
  const uint32_t pv_fin = bars2 + 64u;
  const uint32_t q_ready = bars2 + 72u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  int32_t* s_pages = reinterpret_cast<int32_t*>(smem + kOffPages);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g = blockIdx.x;  // kv head
  if (tid == 0) tma_prefetch_desc(&half_map);
  // ---- the item: {members, p_begin, n, 0, seq[16], slot[16]} (plan data,
  // complete before this grid starts)
  const int32_t* it = reinterpret_cast<const int32_t*>(a.plan_shared) +
                      static_cast<int64_t>(blockIdx.y) * kPlanSharedWords;
  const int members = it[0], p_begin = it[1], n = it[2];
  const int leader = it[4];
  const int nb = (n + kTcBatch - 1) / kTcBatch;
  prefetch_first_batches(&half_map, a, g, tid, p_begin, n, leader);
  // The barriers and the TMEM allocation before the grid wait, so this CTA
  // holds its columns before it lets a dependent grid launch: a dependent
  // grid's CTAs on this SM (the next layer's, beside a segment grid that
  // waits for this one) can then never take columns this CTA still needs.
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const uint32_t bar = bars + 8u * i;  // the softmax rows arrive on two
      mbar_init(bar, (bar == p_ready(0) || bar == p_ready(1) || bar == q_ready) ? kTcM : 1);
    }
    fence_barrier_init();
  }
  if (warp == kPvWarp) {
    __syncwarp();
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  wait_for_prior_grids();
  allow_dependent_grids();

  // page ids: the leader's table (every member's holds the same ones here)
  for (int i = tid; i < n; i += kTcThreads) {
    int32_t pid = a.block_table[static_cast<int64_t>(leader) * a.max_blocks + p_begin + i];
    if (pid < 0 || pid >= a.num_pages) {
      record_error(a.dev_err, kErrPage);
      pid = -1;
    }
    s_pages[i] = pid;
  }
  // Q rows into registers now, into TMEM once it is allocated: MMA row L
  // holds query row (L mod 64) = 4 m + i, query row i of head g of member m
  // (absent members: zeros), 64 dims as 32 packed columns
  uint32_t qw[2][16];
  if (warp < kTcSoftmaxWarps) {
    const int qr = tid & (kTcRows - 1), m = qr >> 2;
    const uint4* src = m < members
                           ? reinterpret_cast<const uint4*>(
                                 a.q + (static_cast<int64_t>(it[4 + m]) * kNumQHeads + g * kGroup +
                                        (qr & 3)) * kHeadDim)
                           : nullptr;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = src != nullptr ? src[c] : make_uint4(0u, 0u, 0u, 0u);
      qw[c >> 2][4 * (c & 3) + 0] = v.x;
      qw[c >> 2][4 * (c & 3) + 1] = v.y;
      qw[c >> 2][4 * (c & 3) + 2] = v.z;
      qw[c >> 2][4 * (c & 3) + 3] = v.w;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (warp < kTcSoftmaxWarps) {
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    tmem_st16(t_lane + kTmemQ, qw[0]);
    tmem_st16(t_lane + kTmemQ + 16, qw[1]);
    tmem_wait_st();
    tc_fence_before_sync();
    mbar_arrive(q_ready);  // S_0 may read Q
  }

  // The plan says every member's table holds the leader's page ids over
  // [p_begin, p_begin + n) in this layer; a member whose table says
  // otherwise (a plan built from another layer's tables, or tables changed
  // since) would silently attend the leader's K/V.  The softmax threads
  // compare the entries batch by batch, off the S -> P path: after handing
  // P(j) over, thread t loads member 1 + t / 4's entry for page t mod 4 of
  // batch j, and compares it after handing P(j + 1) over (the load's latency
  // hides in the wait for S(j + 1)).  A difference is reported as
  // PKV_DEVERR_PLAN.  (The
  // whole check before the first batch put a row of table loads in front of
  // it: the first scores reached the softmax 2.3 us after S(0) was issued,
  // against 0.35 us for later batches.)
  int32_t chk_pid = 0;
  int chk_i = -1;        // page of the entry in flight, -1: none
  bool chk_differs = false;
  auto check_load = [&](int j) {
    const int m = 1 + tid / kTcBatch, i = j * kTcBatch + tid % kTcBatch;
    if (m < members && i < n) {
      chk_i = i;
      chk_pid = a.block_table[static_cast<int64_t>(it[4 + m]) * a.max_blocks + p_begin + i];
    }
  };
  auto check_compare = [&]() {
    if (chk_i >= 0 && s_pages[chk_i] >= 0 && chk_pid != s_pages[chk_i]) chk_differs = true;
    chk_i = -1;
  };
  static_assert((kSharedMembers - 1) * kTcBatch <= 32 * kTcSoftmaxWarps,
                "one member entry per softmax thread and batch");

  auto page_live = [&](int k) { return k < n && s_pages[k] >= 0; };
  auto batch_live = [&](int b) {
    int live = 0;
    for (int p = 0; p < kTcBatch; ++p) live += page_live(b * kTcBatch + p) ? 1 : 0;
    return live;
  };
  int issued = 0;  // batches whose copies this producer issued
  // softmax state (warps 0..3: thread = TMEM lane = MMA row), kept past the
  // role loops for the epilogue
  const int L = tid;
  const int h = (L / kTcRows) & 1;  // 0: pages 0, 1 of each batch; 1: pages 2, 3
  const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  float m_ref = -INFINITY, l_run = 0.f;
  bool o_live = false;  // a PV MMA has been issued (O initialised)
  bool ok = true;       // no wait of this softmax row timed out

  if (warp == kKLoadWarp || warp == kVLoadWarp) {
    // ----------------------------------------------------- TMA producers
    if (lane == 0) {
      const bool is_k = warp == kKLoadWarp;
      const int slots = is_k ? kKSlots : kVSlots;
      const uint64_t policy = l2_policy_evict_first();
      for (int b = 0; b < nb; ++b) {
        const uint32_t empty = is_k ? k_empty(b) : v_empty(b);
        const uint32_t full = is_k ? k_full(b) : v_full(b);
        if (b >= slots && !mbar_wait_bounded(empty, ((b / slots) - 1) & 1, a.wait_ns)) {
          record_error(a.dev_err, kErrTimeout);
          break;
        }
        const int live = batch_live(b);
        if (live > 0)
          mbar_arrive_expect_tx(full, live * kHalfTileBytes);
        else
          mbar_arrive(full);
        const uint32_t region =
            sb + (is_k ? kOffK + (b % kKSlots) * kRegionBytes : kOffV + (b % kVSlots) * kRegionBytes);
        for (int p = 0; p < kTcBatch; ++p) {
          const int k = b * kTcBatch + p;
          if (page_live(k))
            tma_load_3d(region + p * kHalfTileBytes, &half_map, full, g * kHeadDim,
                        is_k ? 0 : kPageSize, s_pages[k], policy);
        }
        issued = b + 1;
      }
    }
  } else if (warp == kSWarp) {
    // -------------------------------------------- S = Q K^T, 64 tokens
    if (lane == 0) {
      bool ok = mbar_wait_bounded(q_ready, 0, a.wait_ns);
      tc_fence_after_sync();
      for (int b = 0; b < nb && ok; ++b) {
        if (b >= 2) {  // PV_{b-2} has read P_{b-2} out of X(b mod 2)
          if (!mbar_wait_bounded(x_free(b), ((b - 2) >> 1) & 1, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
        }
        if (!mbar_wait_bounded(k_full(b), (b / kKSlots) & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        if (batch_live(b) > 0) {  // else the softmax masks every column
          const uint32_t kr = sb + kOffK + (b % kKSlots) * kRegionBytes;
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            tc_mma_bf16_ta(tmem + (b & 1) * kTcCols, tmem + kTmemQ + 8 * kk,
                           sw128_desc(kr + 32 * kk), kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(s_ready(b));
        tc_commit(k_empty(b));  // the K region may be refilled
      }
      if (!ok) record_error(a.dev_err, kErrTimeout);
      tc_commit(s_fin);
      if (!mbar_wait_bounded(s_fin, 0)) record_error(a.dev_err, kErrTimeout);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------- O += P V
    if (lane == 0) {
      bool ok = true;
      uint32_t o_init = 0;
      for (int j = 0; j < nb; ++j) {
        if (!mbar_wait_bounded(p_ready(j), (j >> 1) & 1, a.wait_ns) ||
            !mbar_wait_bounded(v_full(j), (j / kVSlots) & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t vr = sb + kOffV + (j % kVSlots) * kRegionBytes;
        const uint32_t x = tmem + (j & 1) * kTcCols;
        for (int p = 0; p < kTcBatch; ++p) {
          if (!page_live(j * kTcBatch + p)) continue;
          const uint64_t v_op = sw128_desc(vr + p * kHalfTileBytes);
          tc_mma_bf16_ta(tmem + kTmemO, x + 8 * p, v_op, kIdescPV, o_init);
          o_init = 1;
          tc_mma_bf16_ta(tmem + kTmemO, x + kPLo + 8 * p, v_op, kIdescPV, 1u);
        }
        tc_commit(pv_done);     // O holds batches 0..j
        tc_commit(x_free(j));   // X(j mod 2) may take S_{j+2}
        tc_commit(v_empty(j));  // the V region may be refilled
      }
      if (!ok) record_error(a.dev_err, kErrTimeout);
      tc_commit(pv_fin);
      if (!mbar_wait_bounded(pv_fin, 0)) record_error(a.dev_err, kErrTimeout);
    }
  } else {
    // --------------------------------------------------------- softmax
    const float c = a.scale_log2;
    const uint32_t zero16[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    for (int j = 0; j < nb; ++j) {
      const bool ready = mbar_wait_bounded(s_ready(j), (j >> 1) & 1, a.wait_ns);
      if (!__all_sync(kFullMask, ready)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t x = t_lane + (j & 1) * kTcCols;
      uint32_t sr[2][16];  // this row's 32 scores: pages 2h, 2h + 1
      tmem_ld16(x + h * kTcHalfCols, sr[0]);
      tmem_ld16(x + h * kTcHalfCols + 16, sr[1]);
      tmem_wait_ld();
      reg_after_wait(sr[0]);
      reg_after_wait(sr[1]);
      bool live[2], any_live = false;
#pragma unroll
      for (int q = 0; q < 2; ++q) live[q] = page_live(j * kTcBatch + 2 * h + q);
#pragma unroll
      for (int p = 0; p < kTcBatch; ++p) any_live = any_live || page_live(j * kTcBatch + p);
      // row maximum as a tree (independent chains)
      float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (live[q])
#pragma unroll
          for (int t = 0; t < kPageSize; ++t)
            mxs[t & 3] = fmaxf(mxs[t & 3], __uint_as_float(sr[q][t]));
      const float mx = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])) * c;
      // (branch-free: the TMEM accesses below are warp-collective)
      const bool grow = mx > m_ref + kRescaleLog2;
      const float m_new = grow ? fmaxf(m_ref, mx) : m_ref;
      const float alpha = grow ? fast_exp2(m_ref - m_new) : 1.f;  // 0 on the first live page
      m_ref = m_new;
      // P = 2^(s c - m_ref) as hi + lo bf16 terms; word w of page q packs
      // tokens 2w, 2w + 1
      uint32_t hi[16], lo[16];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          float x0 = 0.f, x1 = 0.f;
          if (live[q]) {
            x0 = fast_exp2(fmaf(__uint_as_float(sr[q][2 * w]), c, -m_ref));
            x1 = fast_exp2(fmaf(__uint_as_float(sr[q][2 * w + 1]), c, -m_ref));
          }
          ls[w & 3] += x0 + x1;
          const uint32_t hw = pack_bf16x2(x0, x1);
          hi[8 * q + w] = hw;
          lo[8 * q + w] = pack_bf16x2(x0 - __uint_as_float(hw << 16),
                                      x1 - __uint_as_float(hw & 0xFFFF0000u));
        }
      l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      if (__any_sync(kFullMask, grow && o_live)) {
        // O row *= alpha, once PV_{j-1} is done (every lane takes part in the
        // collective TMEM accesses; rows that did not move multiply by 1).
        // S_j needed PV_{j-2} done and PV_j needs this row's P_j, so pv_done
        // is within one phase of j - 1 here and its parity is unambiguous.
        const bool done = j == 0 || mbar_wait_bounded(pv_done, (j - 1) & 1, a.wait_ns);
        if (!__all_sync(kFullMask, done)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int q = 0; q < kHeadDim / 16; ++q) {
          uint32_t o[16];
          tmem_ld16(t_lane + kTmemO + 16 * q, o);
          tmem_wait_ld();
          reg_after_wait(o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st16(t_lane + kTmemO + 16 * q, o);
        }
      }
      // P over S: hi in X + 16h, lo in X + 32 + 16h; the other half's
      // columns of this row are zero
      tmem_st16(x + h * 16, hi);
      tmem_st16(x + (1 - h) * 16, zero16);
      tmem_st16(x + kPLo + h * 16, lo);
      tmem_st16(x + kPLo + (1 - h) * 16, zero16);
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(p_ready(j));
      check_compare();  // the entry loaded after P(j - 1), landed long since
      check_load(j);
      o_live = o_live || any_live;
    }
    check_compare();  // the last batch's entry
    if (chk_differs) record_error(a.dev_err, kErrPlan);
  }

  // ---- drain.  After a timeout a producer's copies may still be in flight:
  // wait for the last batch each ring slot was given (a slot is refilled only
  // after its previous batch was consumed, so that is the only one that can
  // be pending), by the full limit.  Past the barrier below no copy and no
  // MMA of this CTA is in flight (the issuers waited for their last commits,
  // s_fin and pv_fin), so the epilogue may read O from TMEM and reuse the K
  // ring for the row exchange.
  if ((warp == kKLoadWarp || warp == kVLoadWarp) && lane == 0) {
    const bool is_k = warp == kKLoadWarp;
    const int slots = is_k ? kKSlots : kVSlots;
    for (int s = 0; s < slots && s < issued; ++s) {
      const int last_b = s + ((issued - 1 - s) / slots) * slots;
      if (!mbar_wait_bounded(is_k ? k_full(last_b) : v_full(last_b), (last_b / slots) & 1))
        record_error(a.dev_err, kErrTimeout);
    }
  }
  tc_fence_before_sync();
  __syncthreads();

  if (warp < kTcSoftmaxWarps) {
    // ---- epilogue: combine the two copies of each query row, then write
    // the row's partial (max, sum, acc) to its member's slot
    if (!ok && lane == 0) record_error(a.dev_err, kErrTimeout);
    uint32_t o[kHeadDim / 16][16];
    tc_fence_after_sync();
#pragma unroll
    for (int q = 0; q < kHeadDim / 16; ++q) tmem_ld16(t_lane + kTmemO + 16 * q, o[q]);
    tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < kHeadDim / 16; ++q) reg_after_wait(o[q]);
    if (!o_live) {
#pragma unroll
      for (int q = 0; q < kHeadDim / 16; ++q)
#pragma unroll
        for (int e = 0; e < 16; ++e) o[q][e] = 0u;
      l_run = 0.f;
    }
    // the lower copies hand (acc, m, l) to the upper ones through the K ring
    // (every S, the only reader of it, has completed): [64 rows][68 floats]
    float4* xch = reinterpret_cast<float4*>(smem + kOffK);
    const int qr = L & (kTcRows - 1);
    float4* xrow = xch + qr * (kXchStride / 4);
    if (h == 1) {
#pragma unroll
      for (int q = 0; q < kHeadDim / 16; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          xrow[4 * q + e] = make_float4(__uint_as_float(o[q][4 * e]), __uint_as_float(o[q][4 * e + 1]),
                                        __uint_as_float(o[q][4 * e + 2]),
                                        __uint_as_float(o[q][4 * e + 3]));
      xrow[kHeadDim / 4] = make_float4(m_ref, l_run, 0.f, 0.f);
    }
    softmax_warps_sync();
    const int m = qr >> 2;
    if (h == 0 && m < members) {
      const float4 ml = xrow[kHeadDim / 4];
      const float m1 = ml.x, l1 = ml.y;
      const float M = fmaxf(m_ref, m1);
      const float w0 = M == -INFINITY ? 0.f : fast_exp2(m_ref - M);
      const float w1 = M == -INFINITY ? 0.f : fast_exp2(m1 - M);
      const int64_t part =
          static_cast<int64_t>(it[4 + kSharedMembers + m]) * kNumQHeads + g * kGroup + (qr & 3);
      float4* dst = reinterpret_cast<float4*>(a.part_acc + part * kHeadDim);
#pragma unroll
      for (int q = 0; q < kHeadDim / 16; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 u = xrow[4 * q + e];
          dst[4 * q + e] = make_float4(__uint_as_float(o[q][4 * e]) * w0 + u.x * w1,
                                       __uint_as_float(o[q][4 * e + 1]) * w0 + u.y * w1,
                                       __uint_as_float(o[q][4 * e + 2]) * w0 + u.z * w1,
                                       __uint_as_float(o[q][4 * e + 3]) * w0 + u.w * w1);
        }
      *reinterpret_cast<float2*>(a.part_ml + part * 2) = make_float2(M, l_run * w0 + l1 * w1);
    }
  }

  // ---- teardown: every TMEM read is done, so the columns go back
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kPvWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Sets the kernel's shared-memory limit and checks that no more CTAs of it
// fit on one SM than TMEM holds allocations for (kTcCtasPerSm x 256 of 512
// columns), whatever else shares the SM: with that, tcgen05.alloc never
// waits.  The sequential layout's rings guarantee it by shared memory; the
// beside layout's smaller rings leave it to the registers (about 100 per
// thread: two CTAs of 256 threads per SM).
template <int kSlots>
cudaError_t configure_sh_once(int device) {
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (device & 63);
  if (configured.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(
      paged_decode_shared_kernel<kSlots>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      static_cast<int>(ShLayout<kSlots>::smem_bytes(kMaxPagesPerItem)));
  if (err != cudaSuccess) return err;
  if (kSlots == kSlotsBeside) {
    // CTAs of two kernels share an SM only under one L1 / shared-memory
    // split: ask for the largest shared part, which the segment CTAs that
    // run beside these need (they ask for the same)
    err = cudaFuncSetAttribute(paged_decode_shared_kernel<kSlots>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
  }
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, paged_decode_shared_kernel<kSlots>, kTcThreads, ShLayout<kSlots>::smem_bytes(1));
  if (err != cudaSuccess) return err;
  if (per_sm > static_cast<int>(512 / kTmemCols)) return cudaErrorInvalidConfiguration;
  configured.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <int kSlots>
cudaError_t launch_sh(const CUtensorMap& pool_map, const AttnArgs& args, int num_shared,
                      int range_pages, cudaStream_t stream) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  err = configure_sh_once<kSlots>(device);
  if (err != cudaSuccess) return err;
  return launch_pdl(paged_decode_shared_kernel<kSlots>, dim3(kNumKvHeads, num_shared),
                    dim3(kTcThreads), ShLayout<kSlots>::smem_bytes(range_pages), stream, pool_map,
                    args);
}

}  // namespace

cudaError_t launch_shared_prefix_attention(const CUtensorMap& pool_map, const AttnArgs& args,
                                           int num_shared, int range_pages, cudaStream_t stream,
                                           bool beside) {
  if (num_shared < 1 || range_pages < 1 || range_pages > kMaxPagesPerItem)
    return cudaErrorInvalidValue;
  return beside ? launch_sh<kSlotsBeside>(pool_map, args, num_shared, range_pages, stream)
                : launch_sh<kSlotsSequential>(pool_map, args, num_shared, range_pages, stream);
}

}  // namespace pkv
