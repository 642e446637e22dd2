// pkv_internal.h -- launchers shared between the C-ABI layer and the kernels
// of libpkv (not part of the public interface).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Fixed model geometry (Llama 3.2 1B as used by the Tiny-vLLM engine).
constexpr int kHeadDim = 64;
constexpr int kPageSize = 16;
constexpr int kNumKvHeads = 8;
constexpr int kNumQHeads = 32;
constexpr int kGroup = kNumQHeads / kNumKvHeads;  // 4 query rows per kv head

// Default limit of a kernel's wait on its own progress (a page copy, an MMA,
// another role's hand-off), in nanoseconds: 2 s (pkv_set_wait_limit_ns).
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

// Device error bits (mirror PKV_DEVERR_* in pkv.h).
constexpr int kErrPage = 1;
constexpr int kErrSeqLen = 2;
constexpr int kErrPosition = 4;
constexpr int kErrTimeout = 8;
constexpr int kErrOffsets = 16;
constexpr int kErrPlan = 32;

// Work plans (include/pkv.h): header words, item and merge entry sizes.
constexpr int kPlanHeaderWords = 12;
constexpr int kPlanItemWords = 16;
constexpr int kPlanMergeWords = 4;
constexpr int kPlanKindRange = 0;   // 4 warps share pages [p_begin, p_begin + n) of one sequence
constexpr int kPlanKindPacked = 1;  // one whole sequence per warp
constexpr int kPackPages = 16;      // most pages a packed sequence may have
constexpr int kPlanWarps = 4;       // warps per attention CTA: one packed sequence each
// Shared-prefix items (a plan's last section): one CTA per (item, kv head)
// attends pages [p_begin, p_begin + n) that the item's members' tables all
// hold, for the 4 query rows of every member at once: {members, p_begin, n,
// 0, seq[16], slot[16]}.  The planner sizes their ranges for one wave of
// kSharedCtasPerSm CTAs per SM.
constexpr int kSharedMembers = 16;
constexpr int kSharedCtasPerSm = 2;
constexpr int kPlanSharedWords = 4 + 2 * kSharedMembers;
// Segment plans (the plan's segment section, header word 10 = its count):
// one CTA per item of kind kPlanKindSegments {2, first segment, segments,
// pages, 0 ...} streams the pages of up to kSegMax segments {b, L, p_begin,
// n, slot, fold, fold_slot, 0} in order through one ring of whole-page boxes,
// all 8 kv heads at once (paged_decode_segments_kernel); slot -1: the
// segment writes its sequence's output, else a partial for the merge.  With
// fold > 0 the output also takes in the partials of slots [fold_slot,
// fold_slot + fold), which the shared-prefix kernel launched before it wrote.
// The planner packs the layer's pages into one wave of kSegCtasPerSm CTAs
// per SM of near-equal pages.
constexpr int kPlanKindSegments = 2;
constexpr int kPlanSegWords = 8;
constexpr int kSegMax = 4;
constexpr int kSegCtasPerSm = 2;
constexpr int kSegMaxPages = 1024;  // pages of one segment CTA (its page list)
// Header word 11, the plan's layout.  kPlanLayoutBeside (a shared-prefix
// plan whose shared-prefix CTAs fit one per SM): the other attention CTAs
// run beside them -- segment CTAs, one per SM (deeper rings), or
// per-(item, kv head) CTAs, two per SM next to each shared-prefix CTA --
// each streaming its own pages as soon as it starts and waiting for the
// shared-prefix grid only before it folds that grid's partials and before
// it ends.
constexpr int kPlanLayoutSequential = 0;
constexpr int kPlanLayoutBeside = 1;
constexpr int kSegBesideCtasPerSm = 1;
constexpr int kSharedBesideCtasPerSm = 1;
// Shared memory of one beside shared-prefix CTA with the SM's 1 KiB reserve
// per CTA, at most (any page list): what a beside segment CTA leaves free.
constexpr int kSharedBesideSmemMax = 55 * 1024;

// Host side of the work plans (planner.cpp): an upper bound on a plan's
// bytes, and the plan itself from host lengths (PKV_* status).
size_t plan_bytes(int batch, int max_blocks);
int build_plan(const int32_t* lens, int batch, int max_blocks, int num_sms, int32_t* out,
               size_t out_bytes);
// The same with shared prefixes: runs of consecutive sequences whose host
// block tables start with the same min_shared_pages or more entries get
// those pages as shared-prefix items (PKV_* status).
int build_plan_shared(const int32_t* lens, const int32_t* block_tables, int batch,
                      int max_blocks, int num_sms, int min_shared_pages, int32_t* out,
                      size_t out_bytes);

// Positions covered by the per-device cos/sin table (the 2048-token context).
constexpr int kRopeTablePositions = 2048;

// RoPE parameters passed by value to the kernels: inv_freq[i] =
// theta^(-2i/64) for the 32 rotation pairs, and this device's cos/sin table
// of angle pos * inv_freq[i] for pos < kRopeTablePositions.  A kernel uses the
// table only while *table_theta == theta; otherwise it evaluates sincos
// itself (same arithmetic, same values).
struct RopeFreqs {
  double inv_freq[32];
  double theta;
  const float2* table32;     // [pos][i] (cos, sin) rounded to float
  const double2* table64;    // [pos][i] (cos, sin)
  const double* table_theta; // theta the table holds
};

// Fill `f` for theta and, when this device's table holds another theta,
// enqueue its rebuild on `stream`.
cudaError_t prepare_rope(double theta, RopeFreqs* f, cudaStream_t stream);

// Launch `kernel` with programmatic stream serialization allowed (see
// wait_for_prior_grids in pkv_device.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same, launched in thread-block clusters of cluster_x CTAs along x (the
// kernel uses no cluster feature: the cluster only makes its CTAs start
// together, on one GPC).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Split plan of one attention call.
struct SplitPlan {
  int num_splits;       // grid extent of the split dimension (S)
  int pages_per_split;  // logical pages per range
};

cudaError_t launch_kv_append(const uint16_t* k_new, const uint16_t* v_new,
                             uint16_t* pool, int64_t num_pages,
                             const int32_t* block_table, int max_blocks,
                             const int32_t* positions, int batch,
                             const RopeFreqs& freqs, const uint16_t* q_in,
                             uint16_t* q_out, int32_t* dev_err,
                             cudaStream_t stream);

cudaError_t launch_kv_write_prefill(const uint16_t* k, const uint16_t* v, int num_tokens,
                                    const int32_t* token_offsets,
                                    const int32_t* start_positions, uint16_t* pool,
                                    int64_t num_pages, const int32_t* block_table,
                                    int max_blocks, int batch, const RopeFreqs& freqs,
                                    int32_t* dev_err, unsigned long long wait_ns,
                                    cudaStream_t stream);

struct AttnArgs {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  uint16_t* out;
  float* part_acc;  // [B][Hq][S][D] fp32, unnormalised
  float* part_ml;   // [B][Hq][S][2] fp32, (max in log2 units, sum)
  const int4* plan_items;   // work plan items (kPlanItemWords words each), or nullptr
  const int4* plan_merges;  // work plan merge entries (b, first slot, ranges, 0)
  const int4* plan_shared;  // work plan shared-prefix items (kPlanSharedWords words each)
  const int4* plan_segs;    // work plan segments (kPlanSegWords words each)
  int32_t* dev_err;
  int64_t num_pages;
  int max_blocks;
  int batch;
  float scale_log2;  // softmax scale * log2(e)
  SplitPlan plan;
  unsigned long long wait_ns;  // limit of each wait on the kernel's progress
};

// The calling thread's wait limit (pkv_set_wait_limit_ns), for the launches.
unsigned long long wait_limit_ns();

// Extra inputs of the fused decode step: the new token of every sequence is
// appended at position seq_lens[b] - 1 by the attention kernel itself.
struct AppendArgs {
  const uint16_t* k_new;  // [B][Hkv][D]
  const uint16_t* v_new;  // [B][Hkv][D]
  uint16_t* pool;         // the pool, writable
  RopeFreqs freqs;
};

// Attention only (append == nullptr) or the fused append + attention step.
cudaError_t launch_paged_decode_attention(const CUtensorMap& pool_map,
                                          const AttnArgs& args,
                                          cudaStream_t stream,
                                          const AppendArgs* append = nullptr);

// The same under a work plan: grid (Hkv, num_items), then the merge of the
// num_merges split sequences.  range_pages sizes the shared page list.
// beside: the plan's layout is kPlanLayoutBeside (launched right after the
// shared-prefix grid, whose CTAs it runs next to).
cudaError_t launch_planned_decode_attention(const CUtensorMap& pool_map,
                                            const AttnArgs& args, int num_items,
                                            int num_merges, int range_pages,
                                            cudaStream_t stream,
                                            const AppendArgs* append = nullptr,
                                            bool beside = false);

// The same attention (fixed plan: args.plan_items == nullptr, grid (S, B);
// work plan: range items only, grid (num_items)) with one CTA per (sequence,
// range) covering all kv heads, each page fetched as one 32 KiB box through
// page_map (decode_pagebox.cu).  The caller launches the split merge.
cudaError_t launch_pagebox_attention(const CUtensorMap& page_map, const AttnArgs& args,
                                     int num_items, int range_pages, cudaStream_t stream,
                                     const AppendArgs* append = nullptr);
int pagebox_max_range_pages();

// A segment plan's CTAs (decode_segments.cu): grid (num_items), each CTA
// streaming its segments' pages (at most max_pages) through whole-page boxes
// of page_map.  beside: the plan's layout is kPlanLayoutBeside (launched
// right after the shared-prefix grid, whose CTAs it runs beside).  The
// caller launches the merge.
cudaError_t launch_segments_attention(const CUtensorMap& page_map, const AttnArgs& args,
                                      int num_items, int max_pages, cudaStream_t stream,
                                      const AppendArgs* append = nullptr, bool beside = false);

// Launch the split merge of a plan (fixed: merge_splits_kernel when S > 1;
// work plan: merge_plan_kernel over num_merges sequences).
cudaError_t launch_split_merge(const AttnArgs& args, int num_merges, cudaStream_t stream);

// Shared-prefix items of a work plan: grid (Hkv, num_shared), each CTA
// writing its members' partials (decode_shared.cu).  beside: the plan's
// layout is kPlanLayoutBeside (smaller rings, to leave room for a segment CTA).
cudaError_t launch_shared_prefix_attention(const CUtensorMap& pool_map, const AttnArgs& args,
                                           int num_shared, int range_pages, cudaStream_t stream,
                                           bool beside = false);

// Largest logical page range one attention CTA handles.
int max_pages_per_split();

// Workspace bytes for a plan (0 when nothing is split).
size_t workspace_bytes_for(int batch, int num_q_heads, int head_dim,
                           const SplitPlan& plan);

}  // namespace pkv
