// pkv_api.cu -- the extern "C" boundary of libpkv (declared in include/pkv.h):
// argument checks, the split plan, TMA descriptor encoding, and launches.
// No entry point allocates, frees or synchronizes; everything is enqueued on
// the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "pkv.h"
#include "pkv_internal.h"

using pkv::kHeadDim;
using pkv::kNumKvHeads;
using pkv::kNumQHeads;
using pkv::kPageSize;

namespace pkv {

// The calling thread's limit on each in-kernel wait (pkv_set_wait_limit_ns).
unsigned long long& t_wait_ns_ref() {
  thread_local unsigned long long ns = kDefaultWaitNs;
  return ns;
}

unsigned long long wait_limit_ns() { return t_wait_ns_ref(); }

}  // namespace pkv

namespace {

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// SM count of the current device, cached per device (-1 when unavailable).
int current_sm_count() {
  static std::atomic<int> cache[64] = {};  // 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (dev < 0 || dev >= 64) return -1;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Split plan: S logical page ranges of pages_per_split pages per sequence,
// one CTA each.  Explicit S is honoured (capped by the table width); S = 0
// aims for about four CTAs per SM across (sequence, kv head, range) while
// keeping at least eight pages per range (measured on one 2048-token
// sequence: 8 pages per range 114.7 us per 16 layers, 4 pages 135.9 us).
bool make_plan(int batch, int max_blocks, int num_splits, pkv::SplitPlan* plan) {
  int S;
  if (num_splits > 0) {
    S = num_splits;
  } else {
    const int sms = current_sm_count();
    if (sms <= 0) return false;
    const long long units = static_cast<long long>(batch) * kNumKvHeads;
    const long long target = 4LL * sms;
    S = static_cast<int>((target + units - 1) / units);
    const int cap = (max_blocks + 7) / 8;
    if (S > cap) S = cap;
    if (S < 1) S = 1;
  }
  if (S > max_blocks) S = max_blocks;
  int pps = (max_blocks + S - 1) / S;
  if (pps > pkv::max_pages_per_split()) pps = pkv::max_pages_per_split();
  plan->pages_per_split = pps;
  plan->num_splits = (max_blocks + pps - 1) / pps;
  return true;
}

size_t plan_workspace(int batch, const pkv::SplitPlan& plan) {
  return pkv::workspace_bytes_for(batch, kNumQHeads, kHeadDim, plan);
}

bool supported_dims(int num_q_heads, int num_kv_heads, int head_dim, int page_size) {
  return num_q_heads == kNumQHeads && num_kv_heads == kNumKvHeads &&
         head_dim == kHeadDim && page_size == kPageSize;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// TMA descriptor of the pool viewed as [num_pages][32 rows (K|V x slot)][512]
// bf16, 128-byte swizzled, with a box of one kv head's rows of one page:
// box_rows = 32 takes its K and V rows (a 4 KiB tile), box_rows = 16 its K
// rows (row coordinate 0) or its V rows (row coordinate 16), 2 KiB each.
// Cached per thread for the last (device, pool, pages) of each box height.
bool pool_tensor_map(const void* pool, int64_t num_pages, CUtensorMap* out,
                     int box_rows = 2 * kPageSize) {
  struct Entry {
    int device = -1;
    const void* pool = nullptr;
    int64_t num_pages = 0;
    CUtensorMap map;
  };
  thread_local Entry cached[2];
  if (box_rows != kPageSize && box_rows != 2 * kPageSize) return false;
  Entry& c = cached[box_rows == kPageSize ? 1 : 0];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (c.device == dev && c.pool == pool && c.num_pages == num_pages) {
    *out = c.map;
    return true;
  }
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kNumKvHeads * kHeadDim),
                              static_cast<cuuint64_t>(2 * kPageSize),
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[2] = {
      static_cast<cuuint64_t>(kNumKvHeads * kHeadDim * 2),
      static_cast<cuuint64_t>(2 * kPageSize * kNumKvHeads * kHeadDim * 2)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim),
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap m;
  const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  c.device = dev;
  c.pool = pool;
  c.num_pages = num_pages;
  c.map = m;
  *out = m;
  return true;
}

// TMA descriptor of the pool as the 4-D tensor (dim 64, row 32, kv head 8,
// page) with strides (2 B, 1 KiB, 128 B, 32 KiB) and a box of one whole page:
// the box lands in shared memory as [head][32 rows][64], 128-byte swizzled,
// i.e. each head's 4 KiB tile laid out as in pool_tensor_map's box.
bool pool_page_map(const void* pool, int64_t num_pages, CUtensorMap* out) {
  struct Entry {
    int device = -1;
    const void* pool = nullptr;
    int64_t num_pages = 0;
    CUtensorMap map;
  };
  thread_local Entry cached;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cached.device == dev && cached.pool == pool && cached.num_pages == num_pages) {
    *out = cached.map;
    return true;
  }
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim),
                              static_cast<cuuint64_t>(2 * kPageSize),
                              static_cast<cuuint64_t>(kNumKvHeads),
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {
      static_cast<cuuint64_t>(kNumKvHeads * kHeadDim * 2),  // next row (slot, K|V)
      static_cast<cuuint64_t>(kHeadDim * 2),                 // next kv head
      static_cast<cuuint64_t>(2 * kPageSize * kNumKvHeads * kHeadDim * 2)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(kHeadDim),
                             static_cast<cuuint32_t>(2 * kPageSize),
                             static_cast<cuuint32_t>(kNumKvHeads), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMap m;
  const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  cached.device = dev;
  cached.pool = pool;
  cached.num_pages = num_pages;
  cached.map = m;
  *out = m;
  return true;
}

// Whole-page boxes pay off once the CTAs (one per sequence range, all heads)
// fill every SM at least once.
bool use_pagebox(long long ctas, int range_pages) {
  const int sms = current_sm_count();
  return sms > 0 && ctas >= sms && range_pages <= pkv::pagebox_max_range_pages();
}

// Launch attention (append == nullptr) or the fused step under `plan`: the
// whole-page kernel when the batch fills the SMs, else the per-(sequence,
// kv head) kernel; then the split merge.
cudaError_t launch_attention(const pkv::SplitPlan& plan, const void* pool, int64_t num_pages,
                             const pkv_bf16* q, const int32_t* block_table, int max_blocks,
                             const int32_t* seq_lens, int batch, float scale, pkv_bf16* out,
                             void* workspace, int32_t* dev_err, cudaStream_t stream,
                             const pkv::AppendArgs* append) {
  pkv::AttnArgs args = {};
  args.q = q;
  args.block_table = block_table;
  args.seq_lens = seq_lens;
  args.out = out;
  const size_t need = pkv::workspace_bytes_for(batch, kNumQHeads, kHeadDim, plan);
  float* ws = static_cast<float*>(workspace);
  const size_t acc_elems = static_cast<size_t>(batch) * kNumQHeads * plan.num_splits * kHeadDim;
  args.part_acc = need > 0 ? ws : nullptr;
  args.part_ml = need > 0 ? ws + acc_elems : nullptr;
  args.dev_err = dev_err;
  args.num_pages = num_pages;
  args.max_blocks = max_blocks;
  args.batch = batch;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.plan = plan;
  args.wait_ns = pkv::wait_limit_ns();
  CUtensorMap map;
  if (use_pagebox(static_cast<long long>(batch) * plan.num_splits, plan.pages_per_split)) {
    if (!pool_page_map(pool, num_pages, &map)) return cudaErrorInvalidValue;
    const cudaError_t err =
        pkv::launch_pagebox_attention(map, args, 0, plan.pages_per_split, stream, append);
    if (err != cudaSuccess) return err;
    return pkv::launch_split_merge(args, 0, stream);
  }
  if (!pool_tensor_map(pool, num_pages, &map)) return cudaErrorInvalidValue;
  return pkv::launch_paged_decode_attention(map, args, stream, append);
}

}  // namespace

extern "C" {

PKV_API int pkv_abi_version(void) { return 1; }

PKV_API unsigned long long pkv_set_wait_limit_ns(unsigned long long ns) {
  const unsigned long long prev = pkv::t_wait_ns_ref();
  pkv::t_wait_ns_ref() = ns;
  return prev;
}

PKV_API const char* pkv_strerror(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument (null pointer, bad size or bad scale/theta)";
    case PKV_EUNSUPPORTED: return "unsupported geometry (needs 32 q heads, 8 kv heads, head dim 64, page size 16)";
    case PKV_EWORKSPACE: return "workspace missing or smaller than pkv_workspace_bytes()";
    case PKV_ECUDA: return "CUDA runtime error (launch failed or no usable device)";
    case PKV_EALIGN: return "pointer alignment requirement violated";
    case 7: return "request rejected: its page budget exceeds the whole pool";
    case 8: return "unknown or already finished request id";
    case PKV_ESCRATCH: return "split partials would exceed the static scratch buffer (PKV_STATIC_SCRATCH_BYTES); use fewer splits";
    default: return "unknown status";
  }
}

PKV_API int pkv_plan_splits(int batch, int num_kv_heads, int max_blocks, int num_splits) {
  if (batch < 1 || max_blocks < 1 || num_splits < 0 || num_kv_heads != kNumKvHeads) return -1;
  pkv::SplitPlan plan;
  if (!make_plan(batch, max_blocks, num_splits, &plan)) return -1;
  return plan.num_splits;
}

PKV_API size_t pkv_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                   int head_dim, int max_blocks, int num_splits) {
  if (batch < 0 || max_blocks < 1 || num_splits < 0 ||
      !supported_dims(num_q_heads, num_kv_heads, head_dim, kPageSize))
    return static_cast<size_t>(-1);
  if (batch == 0) return 0;
  pkv::SplitPlan plan;
  if (!make_plan(batch, max_blocks, num_splits, &plan)) return static_cast<size_t>(-1);
  return plan_workspace(batch, plan);
}

PKV_API int pkv_kv_append(const pkv_bf16* k_new, const pkv_bf16* v_new, pkv_bf16* pool,
                          int64_t num_pages, const int32_t* block_table, int max_blocks,
                          const int32_t* positions, int batch, int num_kv_heads,
                          int head_dim, int page_size, double rope_theta,
                          const pkv_bf16* q_in, pkv_bf16* q_out, int num_q_heads,
                          int32_t* dev_err, pkv_stream_t stream) {
  if (!k_new || !v_new || !pool || !block_table || !positions) return PKV_EINVAL;
  if (batch < 0 || num_pages < 1 || num_pages > INT32_MAX || max_blocks < 1) return PKV_EINVAL;
  if ((q_in == nullptr) != (q_out == nullptr)) return PKV_EINVAL;
  if (!(rope_theta > 0.0) || !isfinite(rope_theta)) return PKV_EINVAL;
  if (num_kv_heads != kNumKvHeads || head_dim != kHeadDim || page_size != kPageSize)
    return PKV_EUNSUPPORTED;
  if (q_in != nullptr && num_q_heads != kNumQHeads) return PKV_EUNSUPPORTED;
  if (batch > INT32_MAX / 2) return PKV_EINVAL;
  if (!aligned(pool, 16) || !aligned(v_new, 4) || !aligned(k_new, 2) || !aligned(q_in, 2) ||
      !aligned(q_out, 2) || !aligned(dev_err, 4))
    return PKV_EALIGN;
  if (batch == 0) return PKV_OK;
  pkv::RopeFreqs freqs;
  if (pkv::prepare_rope(rope_theta, &freqs, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PKV_ECUDA;
  const cudaError_t err = pkv::launch_kv_append(
      k_new, v_new, pool, num_pages, block_table, max_blocks, positions, batch, freqs, q_in,
      q_out, dev_err, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

PKV_API int pkv_kv_write_prefill(const pkv_bf16* k, const pkv_bf16* v, int num_tokens,
                                 const int32_t* token_offsets, const int32_t* start_positions,
                                 pkv_bf16* pool, int64_t num_pages, const int32_t* block_table,
                                 int max_blocks, int batch, int num_kv_heads, int head_dim,
                                 int page_size, double rope_theta, int32_t* dev_err,
                                 pkv_stream_t stream) {
  if (!k || !v || !token_offsets || !start_positions || !pool || !block_table) return PKV_EINVAL;
  if (num_tokens < 0 || batch < 1 || num_pages < 1 || num_pages > INT32_MAX || max_blocks < 1 ||
      max_blocks > (INT32_MAX / kPageSize))
    return PKV_EINVAL;
  if (!(rope_theta > 0.0) || !isfinite(rope_theta)) return PKV_EINVAL;
  if (num_kv_heads != kNumKvHeads || head_dim != kHeadDim || page_size != kPageSize)
    return PKV_EUNSUPPORTED;
  if (!aligned(pool, 16) || !aligned(v, 16) || !aligned(k, 16) || !aligned(dev_err, 4))
    return PKV_EALIGN;
  if (num_tokens == 0) return PKV_OK;
  pkv::RopeFreqs freqs;
  if (pkv::prepare_rope(rope_theta, &freqs, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PKV_ECUDA;
  const cudaError_t err = pkv::launch_kv_write_prefill(
      k, v, num_tokens, token_offsets, start_positions, pool, num_pages, block_table, max_blocks,
      batch, freqs, dev_err, pkv::wait_limit_ns(), reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

PKV_API int pkv_paged_decode_attention(const pkv_bf16* q, const pkv_bf16* pool,
                                       int64_t num_pages, const int32_t* block_table,
                                       int max_blocks, const int32_t* seq_lens, int batch,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int page_size, float scale, pkv_bf16* out,
                                       void* workspace, size_t workspace_bytes,
                                       int num_splits, int32_t* dev_err,
                                       pkv_stream_t stream) {
  if (!q || !pool || !block_table || !seq_lens || !out) return PKV_EINVAL;
  if (batch < 0 || batch > 65535 || num_pages < 1 || num_pages > INT32_MAX ||
      max_blocks < 1 || max_blocks > (INT32_MAX / kPageSize) || num_splits < 0)
    return PKV_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return PKV_EINVAL;
  if (!supported_dims(num_q_heads, num_kv_heads, head_dim, page_size)) return PKV_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(out, 4) || !aligned(workspace, 16) ||
      !aligned(dev_err, 4))
    return PKV_EALIGN;
  if (batch == 0) return PKV_OK;
  pkv::SplitPlan plan;
  if (!make_plan(batch, max_blocks, num_splits, &plan)) return PKV_ECUDA;
  const size_t need = plan_workspace(batch, plan);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PKV_EWORKSPACE;
  const cudaError_t err =
      launch_attention(plan, pool, num_pages, q, block_table, max_blocks, seq_lens, batch, scale,
                       out, workspace, dev_err, reinterpret_cast<cudaStream_t>(stream), nullptr);
  return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

PKV_API int pkv_decode_step(const pkv_bf16* q, const pkv_bf16* k_new, const pkv_bf16* v_new,
                            pkv_bf16* pool, int64_t num_pages, const int32_t* block_table,
                            int max_blocks, const int32_t* seq_lens, int batch, int num_q_heads,
                            int num_kv_heads, int head_dim, int page_size, double rope_theta,
                            float scale, pkv_bf16* out, void* workspace, size_t workspace_bytes,
                            int num_splits, int32_t* dev_err, pkv_stream_t stream) {
  if (!q || !k_new || !v_new || !pool || !block_table || !seq_lens || !out) return PKV_EINVAL;
  if (batch < 0 || batch > 65535 || num_pages < 1 || num_pages > INT32_MAX ||
      max_blocks < 1 || max_blocks > (INT32_MAX / kPageSize) || num_splits < 0)
    return PKV_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return PKV_EINVAL;
  if (!(rope_theta > 0.0) || !isfinite(rope_theta)) return PKV_EINVAL;
  if (!supported_dims(num_q_heads, num_kv_heads, head_dim, page_size)) return PKV_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(out, 4) || !aligned(workspace, 16) ||
      !aligned(dev_err, 4) || !aligned(v_new, 4) || !aligned(k_new, 2))
    return PKV_EALIGN;
  if (batch == 0) return PKV_OK;
  pkv::SplitPlan plan;
  if (!make_plan(batch, max_blocks, num_splits, &plan)) return PKV_ECUDA;
  const size_t need = plan_workspace(batch, plan);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PKV_EWORKSPACE;
  pkv::AppendArgs app;
  app.k_new = k_new;
  app.v_new = v_new;
  app.pool = pool;
  if (pkv::prepare_rope(rope_theta, &app.freqs, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PKV_ECUDA;
  const cudaError_t err =
      launch_attention(plan, pool, num_pages, q, block_table, max_blocks, seq_lens, batch, scale,
                       out, workspace, dev_err, reinterpret_cast<cudaStream_t>(stream), &app);
  return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Attention without a caller workspace: the split-K partials live in a fixed
// device buffer owned by the library (see pkv_paged_decode_attention_static_ws
// in pkv.h for who needs this and the rules of sharing it).

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch, looked up once per device (with that
// device current) and cached.  In host code the symbol itself is only a
// stand-in for the device object, so its address must never be passed to a
// kernel directly.
void* static_scratch_address(int device) {
  static std::atomic<void*> cache[64] = {};
  if (device < 0 || device >= 64) return nullptr;
  void* p = cache[device].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  cache[device].store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" PKV_API int pkv_paged_decode_attention_static_ws(
    const pkv_bf16* q, const pkv_bf16* pool, int64_t num_pages, const int32_t* block_table,
    int max_blocks, const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
    int head_dim, int page_size, float scale, pkv_bf16* out, int num_splits,
    int32_t* dev_err, pkv_stream_t stream) {
  if (!q || !pool || !block_table || !seq_lens || !out) return PKV_EINVAL;
  if (batch < 0 || batch > 65535 || num_pages < 1 || num_pages > INT32_MAX ||
      max_blocks < 1 || max_blocks > (INT32_MAX / kPageSize) || num_splits < 0)
    return PKV_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return PKV_EINVAL;
  if (!supported_dims(num_q_heads, num_kv_heads, head_dim, page_size)) return PKV_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(out, 4) || !aligned(dev_err, 4))
    return PKV_EALIGN;
  if (batch == 0) return PKV_OK;
  pkv::SplitPlan plan;
  if (!make_plan(batch, max_blocks, num_splits, &plan)) return PKV_ECUDA;
  const size_t need = plan_workspace(batch, plan);
  if (need > PKV_STATIC_SCRATCH_BYTES) return PKV_ESCRATCH;
  float* ws = nullptr;
  if (need > 0) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return PKV_ECUDA;
    ws = static_cast<float*>(static_scratch_address(device));
    if (ws == nullptr) return PKV_ECUDA;
  }
  const cudaError_t err =
      launch_attention(plan, pool, num_pages, q, block_table, max_blocks, seq_lens, batch, scale,
                       out, ws, dev_err, reinterpret_cast<cudaStream_t>(stream), nullptr);
  return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

// ---------------------------------------------------------------------------
// Work plans (include/pkv.h): built on the host by planner.cpp, run by the
// attention kernel's planned instances.

namespace {

struct PlanHeader {
  int32_t magic, batch, max_blocks, num_items, num_merges, num_slots, range_pages, bytes_used;
  int32_t num_shared, shared_pages, num_segs, layout;
};
static_assert(sizeof(PlanHeader) == 4 * pkv::kPlanHeaderWords, "plan header layout");

// True when every index a kernel takes from the plan's body stays inside the
// buffers it addresses: sequences in [0, batch), page ranges inside the table
// and within the page list the launch sizes (range_pages, shared_pages),
// partial slots in [0, num_slots), shared items with 1..16 members.  A plan
// from pkv_plan_build / pkv_plan_build_shared always passes; a hand-made or
// damaged one is refused before anything is launched.
bool plan_body_valid(const PlanHeader& h) {
  const int32_t* w = reinterpret_cast<const int32_t*>(&h) + pkv::kPlanHeaderWords;
  auto seq_ok = [&](int32_t b) { return b >= 0 && b < h.batch; };
  auto range_ok = [&](int32_t p, int32_t n, int32_t cap) {
    return p >= 0 && n >= 0 && n <= cap && static_cast<int64_t>(p) + n <= h.max_blocks;
  };
  const int64_t lmax = static_cast<int64_t>(h.max_blocks) * kPageSize;
  const int32_t* segs = w + static_cast<int64_t>(h.num_items) * pkv::kPlanItemWords +
                        static_cast<int64_t>(h.num_merges) * pkv::kPlanMergeWords +
                        static_cast<int64_t>(h.num_shared) * pkv::kPlanSharedWords;
  for (int i = 0; i < h.num_items; ++i, w += pkv::kPlanItemWords) {
    if (h.num_segs > 0) {
      // a segment plan: every item is a segment CTA, its segments inside the
      // section, their pages summing to the item's, at most range_pages
      if (w[0] != pkv::kPlanKindSegments || w[1] < 0 || w[2] < 1 || w[2] > pkv::kSegMax ||
          static_cast<int64_t>(w[1]) + w[2] > h.num_segs || w[3] < 0 || w[3] > h.range_pages)
        return false;
      int64_t pages = 0;
      for (int k = 0; k < w[2]; ++k) {
        const int32_t* sg = segs + static_cast<int64_t>(w[1] + k) * pkv::kPlanSegWords;
        const int64_t live = (static_cast<int64_t>(sg[1]) + kPageSize - 1) / kPageSize;
        if (!seq_ok(sg[0]) || sg[1] < 0 || sg[1] > lmax || !range_ok(sg[2], sg[3], h.range_pages) ||
            sg[2] + sg[3] > live || (sg[4] != -1 && (sg[4] < 0 || sg[4] >= h.num_slots)))
          return false;
        // partials folded into the output: slots [sg[6], sg[6] + sg[5])
        if (sg[5] < 0 || sg[7] != 0 ||
            (sg[5] == 0 ? sg[6] != 0
                        : (sg[4] != -1 || sg[6] < 0 ||
                           static_cast<int64_t>(sg[6]) + sg[5] > h.num_slots)))
          return false;
        pages += sg[3];
      }
      if (pages != w[3]) return false;
      continue;
    }
    if (w[0] == pkv::kPlanKindRange) {
      if (!seq_ok(w[4]) || !range_ok(w[2], w[3], h.range_pages)) return false;
      if (w[1] != -1 && (w[1] < 0 || w[1] >= h.num_slots)) return false;
    } else if (w[0] == pkv::kPlanKindPacked) {
      if (w[1] != -1) return false;
      for (int k = 0; k < pkv::kPlanWarps; ++k)
        if (w[4 + k] != -1 && (!seq_ok(w[4 + k]) || w[8 + k] < 0 || w[8 + k] > lmax))
          return false;
    } else {
      return false;
    }
  }
  for (int i = 0; i < h.num_merges; ++i, w += pkv::kPlanMergeWords)
    if (!seq_ok(w[0]) || w[1] < 0 || w[2] < 1 ||
        static_cast<int64_t>(w[1]) + w[2] > h.num_slots)
      return false;
  for (int i = 0; i < h.num_shared; ++i, w += pkv::kPlanSharedWords) {
    const int members = w[0];
    if (members < 1 || members > pkv::kSharedMembers || w[2] < 1 ||
        !range_ok(w[1], w[2], h.shared_pages))
      return false;
    for (int m = 0; m < members; ++m)
      if (!seq_ok(w[4 + m]) || w[4 + pkv::kSharedMembers + m] < 0 ||
          w[4 + pkv::kSharedMembers + m] >= h.num_slots)
        return false;
  }
  return true;
}

// The plan's header when it is well formed for this batch and table, else nullptr.
const PlanHeader* plan_header(const void* plan, int batch, int max_blocks) {
  if (plan == nullptr || !aligned(plan, 16)) return nullptr;
  const PlanHeader* h = static_cast<const PlanHeader*>(plan);
  if (h->magic != static_cast<int32_t>(PKV_PLAN_MAGIC) || h->batch != batch ||
      h->max_blocks != max_blocks || h->num_items < 1 || h->num_items > 65535 ||
      h->num_merges < 0 || h->num_merges > batch || h->num_slots < 0 ||
      h->range_pages < 1 || h->range_pages > 1024 || h->num_shared < 0 ||
      h->num_shared > 65535 || h->num_segs < 0 ||
      (h->num_shared > 0 && (h->shared_pages < 1 || h->shared_pages > 1024)))
    return nullptr;
  // the beside layout is for shared-prefix plans only
  if (h->layout != pkv::kPlanLayoutSequential &&
      (h->layout != pkv::kPlanLayoutBeside || h->num_shared < 1))
    return nullptr;
  // bytes_used is exactly the header and the three sections the counts imply
  const int64_t words = pkv::kPlanHeaderWords +
                        static_cast<int64_t>(h->num_items) * pkv::kPlanItemWords +
                        static_cast<int64_t>(h->num_merges) * pkv::kPlanMergeWords +
                        static_cast<int64_t>(h->num_shared) * pkv::kPlanSharedWords +
                        static_cast<int64_t>(h->num_segs) * pkv::kPlanSegWords;
  if (static_cast<int64_t>(h->bytes_used) != 4 * words) return nullptr;
  if (!plan_body_valid(*h)) return nullptr;
  return h;
}

size_t plan_slots_bytes(const PlanHeader& h) {
  return static_cast<size_t>(h.num_slots) * kNumQHeads * (kHeadDim + 2) * sizeof(float);
}

// True when every item of the plan is a range (no packed sequences).
bool plan_has_only_ranges(const PlanHeader& h) {
  const int32_t* item = reinterpret_cast<const int32_t*>(&h) + pkv::kPlanHeaderWords;
  for (int i = 0; i < h.num_items; ++i, item += pkv::kPlanItemWords)
    if (item[0] != pkv::kPlanKindRange) return false;
  return true;
}

// Launch a planned call: the whole-page kernel when the plan is all ranges
// and fills the SMs, else the per-(item, kv head) kernel; then the merge.
cudaError_t launch_planned(const PlanHeader& h, const void* pool, int64_t num_pages,
                           const pkv_bf16* q, const int32_t* block_table, int max_blocks,
                           const int32_t* seq_lens, int batch, float scale, pkv_bf16* out,
                           const void* plan_dev, void* workspace, int32_t* dev_err,
                           cudaStream_t stream, const pkv::AppendArgs* append) {
  pkv::AttnArgs args = {};
  args.q = q;
  args.block_table = block_table;
  args.seq_lens = seq_lens;
  args.out = out;
  float* ws = static_cast<float*>(workspace);
  const size_t slots = static_cast<size_t>(h.num_slots) * kNumQHeads;
  args.part_acc = h.num_slots > 0 ? ws : nullptr;
  args.part_ml = h.num_slots > 0 ? ws + slots * kHeadDim : nullptr;
  const int32_t* words = static_cast<const int32_t*>(plan_dev);
  args.plan_items = reinterpret_cast<const int4*>(words + pkv::kPlanHeaderWords);
  args.plan_merges = reinterpret_cast<const int4*>(
      words + pkv::kPlanHeaderWords + static_cast<size_t>(h.num_items) * pkv::kPlanItemWords);
  args.plan_shared = reinterpret_cast<const int4*>(
      words + pkv::kPlanHeaderWords + static_cast<size_t>(h.num_items) * pkv::kPlanItemWords +
      static_cast<size_t>(h.num_merges) * pkv::kPlanMergeWords);
  args.plan_segs = reinterpret_cast<const int4*>(
      reinterpret_cast<const int32_t*>(args.plan_shared) +
      static_cast<size_t>(h.num_shared) * pkv::kPlanSharedWords);
  args.dev_err = dev_err;
  args.num_pages = num_pages;
  args.max_blocks = max_blocks;
  args.batch = batch;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.plan.num_splits = 1;
  args.plan.pages_per_split = h.range_pages;
  args.wait_ns = pkv::wait_limit_ns();
  CUtensorMap map;
  if (h.num_shared > 0) {
    // shared prefixes first: their partials join the members' own ones in
    // the merge that follows the attention kernel
    if (!pool_tensor_map(pool, num_pages, &map, kPageSize)) return cudaErrorInvalidValue;
    const cudaError_t err =
        pkv::launch_shared_prefix_attention(map, args, h.num_shared, h.shared_pages, stream,
                                            h.layout == pkv::kPlanLayoutBeside);
    if (err != cudaSuccess) return err;
  }
  if (h.num_segs > 0) {
    if (!pool_page_map(pool, num_pages, &map)) return cudaErrorInvalidValue;
    const cudaError_t err =
        pkv::launch_segments_attention(map, args, h.num_items, h.range_pages, stream, append,
                                       h.layout == pkv::kPlanLayoutBeside);
    if (err != cudaSuccess) return err;
    return pkv::launch_split_merge(args, h.num_merges, stream);
  }
  const bool beside = h.layout == pkv::kPlanLayoutBeside;
  if (!beside && use_pagebox(h.num_items, h.range_pages) && plan_has_only_ranges(h)) {
    if (!pool_page_map(pool, num_pages, &map)) return cudaErrorInvalidValue;
    const cudaError_t err = pkv::launch_pagebox_attention(map, args, h.num_items, h.range_pages,
                                                          stream, append);
    if (err != cudaSuccess) return err;
    return pkv::launch_split_merge(args, h.num_merges, stream);
  }
  if (!pool_tensor_map(pool, num_pages, &map)) return cudaErrorInvalidValue;
  return pkv::launch_planned_decode_attention(map, args, h.num_items, h.num_merges,
                                              h.range_pages, stream, append, beside);
}

}  // namespace

extern "C" {

PKV_API const char* pkv_attention_kernels(int batch, int max_blocks, int num_splits,
                                          const void* plan) {
  if (batch < 1 || max_blocks < 1 || num_splits < 0) return nullptr;
  if (plan != nullptr) {
    const PlanHeader* h = plan_header(plan, batch, max_blocks);
    if (h == nullptr) return nullptr;
    if (h->num_segs > 0) {
      if (h->num_shared > 0)
        return h->num_merges > 0
                   ? "paged_decode_shared_kernel+paged_decode_segments_kernel+merge_plan_kernel"
                   : "paged_decode_shared_kernel+paged_decode_segments_kernel";
      return h->num_merges > 0 ? "paged_decode_segments_kernel+merge_plan_kernel"
                               : "paged_decode_segments_kernel";
    }
    const bool pb = h->layout != pkv::kPlanLayoutBeside &&
                    use_pagebox(h->num_items, h->range_pages) && plan_has_only_ranges(*h);
    if (h->num_shared > 0)  // a plan with shared groups always merges
      return pb ? "paged_decode_shared_kernel+paged_decode_pagebox_kernel+merge_plan_kernel"
                : "paged_decode_shared_kernel+paged_decode_kernel+merge_plan_kernel";
    if (h->num_merges > 0)
      return pb ? "paged_decode_pagebox_kernel+merge_plan_kernel"
                : "paged_decode_kernel+merge_plan_kernel";
    return pb ? "paged_decode_pagebox_kernel" : "paged_decode_kernel";
  }
  pkv::SplitPlan p;
  if (!make_plan(batch, max_blocks, num_splits, &p)) return nullptr;
  const bool pb = use_pagebox(static_cast<long long>(batch) * p.num_splits, p.pages_per_split);
  if (p.num_splits > 1)
    return pb ? "paged_decode_pagebox_kernel+merge_splits_kernel"
              : "paged_decode_kernel+merge_splits_kernel";
  return pb ? "paged_decode_pagebox_kernel" : "paged_decode_kernel";
}

PKV_API size_t pkv_plan_bytes(int batch, int max_blocks) {
  return pkv::plan_bytes(batch, max_blocks);
}

PKV_API int pkv_plan_build(const int32_t* seq_lens_host, int batch, int max_blocks, int num_sms,
                           void* plan, size_t plan_bytes) {
  if (num_sms < 0) return PKV_EINVAL;
  if (num_sms == 0) {
    num_sms = current_sm_count();
    if (num_sms <= 0) return PKV_ECUDA;
  }
  return pkv::build_plan(seq_lens_host, batch, max_blocks, num_sms, static_cast<int32_t*>(plan),
                         plan_bytes);
}

PKV_API int pkv_plan_build_shared(const int32_t* seq_lens_host, const int32_t* block_tables_host,
                                  int batch, int max_blocks, int num_sms, int min_shared_pages,
                                  void* plan, size_t plan_bytes) {
  if (num_sms < 0) return PKV_EINVAL;
  if (num_sms == 0) {
    num_sms = current_sm_count();
    if (num_sms <= 0) return PKV_ECUDA;
  }
  return pkv::build_plan_shared(seq_lens_host, block_tables_host, batch, max_blocks, num_sms,
                                min_shared_pages, static_cast<int32_t*>(plan), plan_bytes);
}

PKV_API size_t pkv_plan_workspace_bytes(const void* plan) {
  if (plan == nullptr || !aligned(plan, 16)) return static_cast<size_t>(-1);
  const PlanHeader* h = static_cast<const PlanHeader*>(plan);
  if (h->magic != static_cast<int32_t>(PKV_PLAN_MAGIC) || h->num_slots < 0)
    return static_cast<size_t>(-1);
  return plan_slots_bytes(*h);
}

PKV_API int pkv_paged_decode_attention_planned(
    const pkv_bf16* q, const pkv_bf16* pool, int64_t num_pages, const int32_t* block_table,
    int max_blocks, const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
    int head_dim, int page_size, float scale, pkv_bf16* out, const void* plan_host,
    const void* plan_dev, void* workspace, size_t workspace_bytes, int32_t* dev_err,
    pkv_stream_t stream) {
  if (!q || !pool || !block_table || !seq_lens || !out || !plan_host || !plan_dev)
    return PKV_EINVAL;
  if (batch < 1 || batch > 65535 || num_pages < 1 || num_pages > INT32_MAX || max_blocks < 1 ||
      max_blocks > (INT32_MAX / kPageSize))
    return PKV_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return PKV_EINVAL;
  if (!supported_dims(num_q_heads, num_kv_heads, head_dim, page_size)) return PKV_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(out, 4) || !aligned(workspace, 16) ||
      !aligned(dev_err, 4) || !aligned(plan_dev, 16) || !aligned(plan_host, 16))
    return PKV_EALIGN;
  const PlanHeader* h = plan_header(plan_host, batch, max_blocks);
  if (h == nullptr) return PKV_EINVAL;
  const size_t need = plan_slots_bytes(*h);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PKV_EWORKSPACE;
  const cudaError_t err =
      launch_planned(*h, pool, num_pages, q, block_table, max_blocks, seq_lens, batch, scale, out,
                     plan_dev, workspace, dev_err, reinterpret_cast<cudaStream_t>(stream),
                     nullptr);
  return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

PKV_API int pkv_decode_step_planned(
    const pkv_bf16* q, const pkv_bf16* k_new, const pkv_bf16* v_new, pkv_bf16* pool,
    int64_t num_pages, const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
    int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
    double rope_theta, float scale, pkv_bf16* out, const void* plan_host, const void* plan_dev,
    void* workspace, size_t workspace_bytes, int32_t* dev_err, pkv_stream_t stream) {
  if (!q || !k_new || !v_new || !pool || !block_table || !seq_lens || !out || !plan_host ||
      !plan_dev)
    return PKV_EINVAL;
  if (batch < 1 || batch > 65535 || num_pages < 1 || num_pages > INT32_MAX || max_blocks < 1 ||
      max_blocks > (INT32_MAX / kPageSize))
    return PKV_EINVAL;
  if (!(scale > 0.f) || !isfinite(scale)) return PKV_EINVAL;
  if (!(rope_theta > 0.0) || !isfinite(rope_theta)) return PKV_EINVAL;
  if (!supported_dims(num_q_heads, num_kv_heads, head_dim, page_size)) return PKV_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(out, 4) || !aligned(workspace, 16) ||
      !aligned(dev_err, 4) || !aligned(v_new, 4) || !aligned(k_new, 2) ||
      !aligned(plan_dev, 16) || !aligned(plan_host, 16))
    return PKV_EALIGN;
  const PlanHeader* h = plan_header(plan_host, batch, max_blocks);
  if (h == nullptr) return PKV_EINVAL;
  const size_t need = plan_slots_bytes(*h);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PKV_EWORKSPACE;
  pkv::AppendArgs app;
  app.k_new = k_new;
  app.v_new = v_new;
  app.pool = pool;
  if (pkv::prepare_rope(rope_theta, &app.freqs, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PKV_ECUDA;
  const cudaError_t err =
      launch_planned(*h, pool, num_pages, q, block_table, max_blocks, seq_lens, batch, scale, out,
                     plan_dev, workspace, dev_err, reinterpret_cast<cudaStream_t>(stream), &app);
  return err == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

PKV_API int pkv_decode_steps_planned(
    int layers, const pkv_bf16* q, const pkv_bf16* k_new, const pkv_bf16* v_new, pkv_bf16* pool,
    int64_t num_pages, const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
    int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size, double rope_theta,
    float scale, pkv_bf16* out, const void* plan_host, const void* plan_dev, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, pkv_stream_t stream) {
  if (layers < 1) return PKV_EINVAL;
  // layer 0 through the single-layer call checks every argument (the layer
  // strides keep each array's alignment: whole rows of 64 elements) and
  // prepares the RoPE table; the other layers only launch
  const int rc = pkv_decode_step_planned(q, k_new, v_new, pool, num_pages, block_tables,
                                         max_blocks, seq_lens, batch, num_q_heads, num_kv_heads,
                                         head_dim, page_size, rope_theta, scale, out, plan_host,
                                         plan_dev, workspace, workspace_bytes, dev_err, stream);
  if (rc != PKV_OK || layers == 1) return rc;
  const PlanHeader* h = plan_header(plan_host, batch, max_blocks);
  pkv::AppendArgs app;
  app.pool = pool;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (pkv::prepare_rope(rope_theta, &app.freqs, st) != cudaSuccess) return PKV_ECUDA;
  const size_t q_stride = static_cast<size_t>(batch) * kNumQHeads * kHeadDim;
  const size_t kv_stride = static_cast<size_t>(batch) * kNumKvHeads * kHeadDim;
  const size_t bt_stride = static_cast<size_t>(batch) * static_cast<size_t>(max_blocks);
  for (int l = 1; l < layers; ++l) {
    app.k_new = k_new + l * kv_stride;
    app.v_new = v_new + l * kv_stride;
    const cudaError_t err =
        launch_planned(*h, pool, num_pages, q + l * q_stride, block_tables + l * bt_stride,
                       max_blocks, seq_lens, batch, scale, out + l * q_stride, plan_dev,
                       workspace, dev_err, st, &app);
    if (err != cudaSuccess) return PKV_ECUDA;
  }
  return PKV_OK;
}

PKV_API int pkv_kv_write_prefill_layers(int layers, const pkv_bf16* k, const pkv_bf16* v,
                                        int num_tokens, const int32_t* token_offsets,
                                        const int32_t* start_positions, pkv_bf16* pool,
                                        int64_t num_pages, const int32_t* block_tables,
                                        int max_blocks, int batch, int num_kv_heads,
                                        int head_dim, int page_size, double rope_theta,
                                        int32_t* dev_err, pkv_stream_t stream) {
  if (layers < 1) return PKV_EINVAL;
  const int rc = pkv_kv_write_prefill(k, v, num_tokens, token_offsets, start_positions, pool,
                                      num_pages, block_tables, max_blocks, batch, num_kv_heads,
                                      head_dim, page_size, rope_theta, dev_err, stream);
  if (rc != PKV_OK || layers == 1 || num_tokens == 0) return rc;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  pkv::RopeFreqs freqs;
  if (pkv::prepare_rope(rope_theta, &freqs, st) != cudaSuccess) return PKV_ECUDA;
  const size_t kv_stride = static_cast<size_t>(num_tokens) * kNumKvHeads * kHeadDim;
  const size_t bt_stride = static_cast<size_t>(batch) * static_cast<size_t>(max_blocks);
  for (int l = 1; l < layers; ++l) {
    const cudaError_t err = pkv::launch_kv_write_prefill(
        k + l * kv_stride, v + l * kv_stride, num_tokens, token_offsets, start_positions, pool,
        num_pages, block_tables + l * bt_stride, max_blocks, batch, freqs, dev_err,
        pkv::wait_limit_ns(), st);
    if (err != cudaSuccess) return PKV_ECUDA;
  }
  return PKV_OK;
}

}  // extern "C"
