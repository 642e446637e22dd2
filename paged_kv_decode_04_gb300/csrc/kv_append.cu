// kv_append.cu -- KV writes with rotate-half RoPE: the one-token decode append
// and the multi-token prefill write, plus the per-device cos/sin table they
// (and the fused decode step) read.
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗", KV page pool item: each
// decode step adds one new token per sequence at its absolute RoPE position
// into the sequence's page slot of the shared BF16 pool; prefill fills the
// prompt's pages.
//
// The stored key is rotate_pair's value: the rotation evaluated in FP64 with
// separately rounded products and one rounding to bf16.  rotate_pair_rope
// reaches the same bits with FP32 arithmetic plus an FP64 redo of the rare
// elements that land next to a bf16 rounding midpoint, and the (cos, sin)
// pairs come from a table built once per rope_theta instead of an FP64
// sincos per element, since FP64 is slow on this part.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kAppendThreads = 256;
constexpr int kHalf = kHeadDim / 2;
constexpr int kRopeEntries = kRopeTablePositions * kHalf;

// This device's cos/sin tables: kRopeSlots slots, each built once for one
// rope_theta and tagged with it afterwards (a tag of 0 = not built yet; a
// valid theta is > 0).  A slot that holds a theta is never rewritten, so a
// kernel that has read its tag can read its table while calls with other
// thetas run on other streams; once every slot is taken, calls with a new
// theta evaluate sincos in the kernels (the same values).
constexpr int kRopeSlots = 4;
__device__ __align__(16) float2 g_rope32[kRopeSlots][kRopeEntries];
__device__ __align__(16) double2 g_rope64[kRopeSlots][kRopeEntries];
__device__ double g_rope_theta[kRopeSlots];

__global__ void rope_tag_kernel(int slot, double value) { g_rope_theta[slot] = value; }

__global__ void __launch_bounds__(256) rope_table_kernel(RopeFreqs f, int slot) {
  const int e = blockIdx.x * 256 + threadIdx.x;
  if (e >= kRopeEntries) return;
  const int pos = e / kHalf, i = e % kHalf;
  double sn, cs;
  sincos(__dmul_rn(static_cast<double>(pos), f.inv_freq[i]), &sn, &cs);
  g_rope64[slot][e] = make_double2(cs, sn);
  g_rope32[slot][e] = make_float2(static_cast<float>(cs), static_cast<float>(sn));
}

// One CTA per sequence, thread (h, i) rotates pair i of kv head h (and of
// query heads h, h + 8, h + 16, h + 24 when asked); V is copied one word per
// thread.  Every load that does not depend on the position is issued first.
__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(const uint16_t* __restrict__ k_new,
                     const uint16_t* __restrict__ v_new,
                     uint16_t* __restrict__ pool, int64_t num_pages,
                     const int32_t* __restrict__ block_table, int max_blocks,
                     const int32_t* __restrict__ positions, RopeFreqs freqs,
                     const uint16_t* __restrict__ q_in,
                     uint16_t* __restrict__ q_out, int32_t* dev_err) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int h = tid / kHalf, i = tid % kHalf;
  const int64_t row = kNumKvHeads * kHeadDim;  // elements per (kv, slot)
  const int64_t src = static_cast<int64_t>(b) * row;
  wait_for_prior_grids();
  allow_dependent_grids();

  const uint16_t k1 = k_new[src + h * kHeadDim + i];
  const uint16_t k2 = k_new[src + h * kHeadDim + i + kHalf];
  const uint32_t vw = reinterpret_cast<const uint32_t*>(v_new + src)[tid];
  const bool table_ok = rope_table_ready(freqs);
  const int32_t pos = positions[b];
  const bool pos_ok = pos >= 0 && pos < max_blocks * kPageSize;
  const int32_t page =
      pos_ok ? block_table[static_cast<int64_t>(b) * max_blocks + pos / kPageSize] : -1;
  RopeCS cs = rope_cs(freqs, table_ok, pos, i);

  // Optional out-of-place query rotation: 32 heads x 32 pairs, 4 per thread.
  if (q_in != nullptr) {
    const int64_t qbase = static_cast<int64_t>(b) * kNumQHeads * kHeadDim;
    uint16_t x1[4], x2[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = h + 8 * k;
      x1[k] = q_in[qbase + j * kHeadDim + i];
      x2[k] = q_in[qbase + j * kHeadDim + i + kHalf];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t o = qbase + (h + 8 * k) * kHeadDim + i;
      uint16_t y1, y2;
      rotate_pair_rope(freqs, table_ok, pos, i, cs, x1[k], x2[k], &y1, &y2);
      q_out[o] = y1;
      q_out[o + kHalf] = y2;
    }
  }

  if (!pos_ok) {
    if (tid == 0) record_error(dev_err, kErrPosition);
    return;
  }
  if (page < 0 || page >= num_pages) {
    if (tid == 0) record_error(dev_err, kErrPage);
    return;
  }
  const int slot = pos % kPageSize;
  uint16_t* k_dst = pool + ((static_cast<int64_t>(page) * 2 + 0) * kPageSize + slot) * row;
  uint16_t* v_dst = pool + ((static_cast<int64_t>(page) * 2 + 1) * kPageSize + slot) * row;
  uint16_t y1, y2;
  rotate_pair_rope(freqs, table_ok, pos, i, cs, k1, k2, &y1, &y2);
  k_dst[h * kHeadDim + i] = y1;
  k_dst[h * kHeadDim + i + kHalf] = y2;
  reinterpret_cast<uint32_t*>(v_dst)[tid] = vw;
}

// Prefill write.  Token t of the flat prompt batch (sequence b with
// token_offsets[b] <= t < token_offsets[b + 1], position start_positions[b] +
// t - token_offsets[b]) has a 1 KiB K row and a 1 KiB V row, [8 kv][64]
// bf16, contiguous in k and v; its pool rows are as contiguous.  The kernel
// is persistent: each CTA walks chunks of kPfChunk consecutive tokens,
// staging a chunk's K and V rows (one bulk copy each) in a ring of
// kPfStages shared-memory stages so that the next chunks stream in while
// the current one is rotated and written out.  Warp w writes tokens w,
// w + kPfWarps, ... of the chunk; within a row, each lane holds whole
// rotation pairs, so no data moves between lanes.
constexpr int kPfChunk = 16;
constexpr int kPfStages = 2;
constexpr int kPfWarps = 8;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kRowBytes = kNumKvHeads * kHeadDim * 2;       // 1 KiB
constexpr int kPfHalfStage = kPfChunk * kRowBytes;          // the chunk's K (or V) rows
constexpr int kPfStageBytes = 2 * kPfHalfStage;

// Batches up to this size search token_offsets in shared memory.
constexpr int kPrefillSmemBatch = 2048;
constexpr size_t kPfSmemBytes =
    static_cast<size_t>(kPfStages) * kPfStageBytes + 8 * kPfStages +
    sizeof(int32_t) * (kPrefillSmemBatch + 1) + 2 * sizeof(int32_t) * kPfStages;

// Where token t goes: its pool page (-1: skip), slot and position.
struct PfDest {
  int32_t page, slot, pos;
};

__device__ __forceinline__ PfDest prefill_dest(int t, const int32_t* off, int batch,
                                               const int32_t* __restrict__ start_positions,
                                               const int32_t* __restrict__ block_table,
                                               int max_blocks, int64_t num_pages,
                                               int32_t* dev_err) {
  // largest b with off[b] <= t
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int32_t first = off[b];
  PfDest d{-1, 0, 0};
  if (t < first || t >= off[b + 1]) {
    record_error(dev_err, kErrOffsets);
    return d;
  }
  const int32_t pos = start_positions[b] + (t - first);
  if (pos < 0 || pos >= max_blocks * kPageSize) {
    record_error(dev_err, kErrPosition);
    return d;
  }
  const int32_t page = block_table[static_cast<int64_t>(b) * max_blocks + pos / kPageSize];
  if (page < 0 || page >= num_pages) {
    record_error(dev_err, kErrPage);
    return d;
  }
  d.page = page;
  d.slot = pos % kPageSize;
  d.pos = pos;
  return d;
}

// Rotation of the lane's 8 pairs (x1, x2) = dims (8 q + p, 32 + 8 q + p),
// p < 8, of one kv head of a K row in shared memory, stored to the pool row.
// a_src / b_src hold the lane's x1 and x2 values, in that order for even
// heads and swapped for odd ones; with sigma = -1 (x1 first) or +1 (x2
// first) the FP32 rotation of each pair is
//   y_a = a c + fl(b sigma s),   y_b = b c - fl(a sigma s),
// i.e. fma(x1, c, -fl(x2 s)) and fma(x2, c, fl(x1 s)), whose distance from
// the FP64 value is at most 2^-23 (|x1| + |x2| + |y|) (see
// rotate_pair_rope).  y - A and y + A, A = 2^-22 (|x1| + |x2| + |y|), each
// with one rounding, bracket both; when they round to the same bf16, no
// rounding midpoint lies between them and, rounding being monotone, y and
// the FP64 value round alike.  Pairs where that fails, or where |x1| + |x2|
// is outside [2^-100, 2^100] (zeros, subnormals, huge values, inf, NaN),
// come back as bits of the result for rope_redo_pairs.
__device__ __forceinline__ uint32_t rope_row_pairs(const RopeFreqs& f, bool table_ok, int pos,
                                                   uint32_t a_src, uint32_t b_src,
                                                   uint8_t* a_dst, uint8_t* b_dst, int lane_q,
                                                   bool head_odd) {
  const uint4 A4 = lds128(a_src);
  const uint4 B4 = lds128(b_src);
  const uint32_t aw[4] = {A4.x, A4.y, A4.z, A4.w};
  const uint32_t bw[4] = {B4.x, B4.y, B4.z, B4.w};
  const int i0 = 8 * lane_q;
  float c[8], sn[8];
  if (table_ok) {
    const float4* t = reinterpret_cast<const float4*>(f.table32 + pos * kHalf + i0);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 cs = t[e];
      c[2 * e] = cs.x;
      sn[2 * e] = cs.y;
      c[2 * e + 1] = cs.z;
      sn[2 * e + 1] = cs.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      double s64, c64;
      sincos(__dmul_rn(static_cast<double>(pos), f.inv_freq[i0 + e]), &s64, &c64);
      c[e] = static_cast<float>(c64);
      sn[e] = static_cast<float>(s64);
    }
  }
  const uint32_t sigma = head_odd ? 0u : 0x80000000u;
  uint32_t oa[4], ob[4];
  uint32_t bad = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float ya[2], yb[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int p = 2 * e + h;
      const float a = __uint_as_float(h ? (aw[e] & 0xFFFF0000u) : (aw[e] << 16));
      const float b = __uint_as_float(h ? (bw[e] & 0xFFFF0000u) : (bw[e] << 16));
      const float ss = __uint_as_float(__float_as_uint(sn[p]) ^ sigma);
      ya[h] = fmaf(a, c[p], b * ss);
      yb[h] = fmaf(b, c[p], -(a * ss));
      const float s0 = fabsf(a) + fabsf(b);
      const float sa = s0 + fabsf(ya[h]);
      const float sb = s0 + fabsf(yb[h]);
      const uint32_t lo = cvt_bf16x2_rn(fmaf(sa, -0x1p-22f, ya[h]), fmaf(sb, -0x1p-22f, yb[h]));
      const uint32_t hi = cvt_bf16x2_rn(fmaf(sa, 0x1p-22f, ya[h]), fmaf(sb, 0x1p-22f, yb[h]));
      // 2^-100 <= s0 <= 2^100 (binary32 patterns 0x0D800000 .. 0x71800000)
      const bool in_range = __float_as_uint(s0) - 0x0D800000u <= 0x71800000u - 0x0D800000u;
      if (lo != hi || !in_range) bad |= 1u << p;
    }
    oa[e] = cvt_bf16x2_rn(ya[0], ya[1]);
    ob[e] = cvt_bf16x2_rn(yb[0], yb[1]);
  }
  *reinterpret_cast<uint4*>(a_dst) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *reinterpret_cast<uint4*>(b_dst) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  return bad;
}

// rotate_pair's FP64 evaluation of the pairs flagged in `bad`, read back
// from the K row in shared memory (x1_src: the lane's x1 dims; its x2 dims
// are 64 bytes on) and stored over the values rope_row_pairs wrote.
__device__ __forceinline__ void rope_redo_pairs(const RopeFreqs& f, bool table_ok, int pos,
                                                uint32_t bad, uint32_t x1_src, uint8_t* x1_dst,
                                                int lane_q) {
  while (bad != 0) {
    const int p = __ffs(bad) - 1;
    bad &= bad - 1;
    const int i = 8 * lane_q + p;
    const uint16_t h1 = lds16(x1_src + 2 * p);
    const uint16_t h2 = lds16(x1_src + 64 + 2 * p);
    double c64, s64;
    if (table_ok) {
      const double2 t = f.table64[pos * kHalf + i];
      c64 = t.x;
      s64 = t.y;
    } else {
      sincos(__dmul_rn(static_cast<double>(pos), f.inv_freq[i]), &s64, &c64);
    }
    uint16_t o1, o2;
    rotate_pair(h1, h2, c64, s64, &o1, &o2);
    *reinterpret_cast<uint16_t*>(x1_dst + 2 * p) = o1;
    *reinterpret_cast<uint16_t*>(x1_dst + 64 + 2 * p) = o2;
  }
}

__global__ void __launch_bounds__(kPfThreads)
    kv_write_prefill_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                            int num_tokens, const int32_t* __restrict__ token_offsets,
                            const int32_t* __restrict__ start_positions,
                            uint16_t* __restrict__ pool, int64_t num_pages,
                            const int32_t* __restrict__ block_table, int max_blocks, int batch,
                            RopeFreqs freqs, int32_t* dev_err, unsigned long long wait_ns) {
  extern __shared__ __align__(16) uint8_t pf_smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(pf_smem + kPfStages * kPfStageBytes);
  int32_t* s_off = reinterpret_cast<int32_t*>(bars + kPfStages);
  int32_t* done = s_off + kPrefillSmemBatch + 1;  // warps finished with each stage
  int32_t* last_issued = done + kPfStages;       // the last chunk each stage was given
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nchunks = (num_tokens + kPfChunk - 1) / kPfChunk;
  const int my_chunks =
      static_cast<int>(blockIdx.x) < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const uint32_t bar0 = smem_addr(bars);
  const uint32_t stage0 = smem_addr(pf_smem);
  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(bar0 + 8 * s, 1);
      done[s] = 0;
      last_issued[s] = -1;
    }
    fence_barrier_init();
  }
  wait_for_prior_grids();
  allow_dependent_grids();

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int it) {  // one thread: chunk number `it` of this CTA
    const int t0 = (blockIdx.x + it * gridDim.x) * kPfChunk;
    const uint32_t bytes = static_cast<uint32_t>(min(kPfChunk, num_tokens - t0)) * kRowBytes;
    const int st = it % kPfStages;
    const uint32_t bar = bar0 + 8 * st;
    const uint32_t dst = stage0 + st * kPfStageBytes;
    const int64_t src = static_cast<int64_t>(t0) * (kRowBytes / 2);
    last_issued[st] = it;
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_load(dst, k + src, bytes, bar, policy);
    bulk_load(dst + kPfHalfStage, v + src, bytes, bar, policy);
  };
  __syncthreads();  // barriers initialised
  if (tid == 0)
    for (int it = 0; it < kPfStages && it < my_chunks; ++it) issue(it);

  const bool smem_offsets = batch <= kPrefillSmemBatch;
  if (smem_offsets)
    for (int i = tid; i <= batch; i += kPfThreads) s_off[i] = token_offsets[i];
  const int32_t* off = smem_offsets ? s_off : token_offsets;
  const bool tag_ok = rope_table_ready(freqs);
  __syncthreads();  // offsets staged

  // K: lane l rotates dims 8 (l % 4) .. + 8 of both halves of kv head l / 4.
  // The half read and written first alternates with the head (x1 half for
  // even heads, x2 half for odd ones) so that every 8-lane phase of a
  // 16-byte shared-memory access covers all 32 banks.  V: lane l copies
  // bytes [16 l, 16 l + 16) and [512 + 16 l, 512 + 16 l + 16) of the row.
  const int lane_q = lane & 3;
  const int head = lane >> 2;
  const bool head_odd = (head & 1) != 0;
  const int x1_off = head * 128 + 16 * lane_q;  // byte offset of my x1 dims
  const int a_off = x1_off + (head_odd ? 64 : 0);
  const int b_off = x1_off + (head_odd ? 0 : 64);
  const int v_off = 16 * lane;
  for (int it = 0; it < my_chunks; ++it) {
    const int t0 = (blockIdx.x + it * gridDim.x) * kPfChunk;
    const int n = min(kPfChunk, num_tokens - t0);
    // destinations of this warp's tokens, one per lane, while the copy lands
    PfDest dst{-1, 0, 0};
    const int my_j = warp + kPfWarps * lane;
    if (lane < kPfChunk / kPfWarps && my_j < n)
      dst = prefill_dest(t0 + my_j, off, batch, start_positions, block_table, max_blocks,
                         num_pages, dev_err);
    const int st = it % kPfStages;
    const bool ready = mbar_wait_bounded(bar0 + 8 * st, (it / kPfStages) & 1, wait_ns);
    if (!__all_sync(0xFFFFFFFFu, ready)) {
      // stop; the copies still in flight are drained below
      if (lane == 0) record_error(dev_err, kErrTimeout);
      break;
    }
    const uint32_t kst = stage0 + st * kPfStageBytes;
    for (int q = 0; q < kPfChunk / kPfWarps; ++q) {
      const int j = warp + kPfWarps * q;
      const int page = __shfl_sync(0xFFFFFFFFu, dst.page, q);
      const int slot = __shfl_sync(0xFFFFFFFFu, dst.slot, q);
      const int pos = __shfl_sync(0xFFFFFFFFu, dst.pos, q);
      if (j >= n || page < 0) continue;  // warp-uniform
      const int64_t row_el = (static_cast<int64_t>(page) * 2 * kPageSize + slot) * (kRowBytes / 2);
      uint8_t* kd = reinterpret_cast<uint8_t*>(pool + row_el);
      uint8_t* vd = kd + kPageSize * kRowBytes;
      const uint32_t ks = kst + j * kRowBytes;
      const uint32_t vs = ks + kPfHalfStage;
      *reinterpret_cast<uint4*>(vd + v_off) = lds128(vs + v_off);
      *reinterpret_cast<uint4*>(vd + 512 + v_off) = lds128(vs + 512 + v_off);
      const bool table_ok = tag_ok && pos < kRopeTablePositions;
      const uint32_t bad =
          rope_row_pairs(freqs, table_ok, pos, ks + a_off, ks + b_off, kd + a_off, kd + b_off,
                         lane_q, head_odd);
      if (__any_sync(0xFFFFFFFFu, bad != 0))
        rope_redo_pairs(freqs, table_ok, pos, bad, ks + x1_off, kd + x1_off, lane_q);
    }
    // release the stage; the last of the warps refills it, so no warp waits
    // for the others (one may be redoing a rotation in FP64)
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(done + st, 1) == kPfWarps - 1) {
        done[st] = 0;
        __threadfence_block();
        if (it + kPfStages < my_chunks) {
          fence_proxy_async_smem();
          issue(it + kPfStages);
        }
      }
    }
  }
  // before the CTA exits, every copy it issued has landed: after a timeout
  // the phase of the last chunk each stage was given may still be pending (a
  // stage is refilled only once every warp released its previous chunk, so
  // it is the only one), waited for by the full limit
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < kPfStages; ++s)
      if (last_issued[s] >= 0) mbar_wait_bounded(bar0 + 8 * s, (last_issued[s] / kPfStages) & 1);
}

// Device addresses of this device's table slots (looked up once per device)
// and the theta each slot was given (NaN: free).
struct RopeTableAddrs {
  float2* t32 = nullptr;
  double2* t64 = nullptr;
  double* theta = nullptr;
  double slot_theta[kRopeSlots] = {NAN, NAN, NAN, NAN};
};

std::mutex g_rope_mutex;
RopeTableAddrs g_rope_addrs[64];

}  // namespace

cudaError_t prepare_rope(double theta, RopeFreqs* f, cudaStream_t stream) {
  for (int i = 0; i < kHalf; ++i)
    f->inv_freq[i] = pow(theta, -(2.0 * i) / static_cast<double>(kHeadDim));
  f->theta = theta;
  f->table32 = nullptr;
  f->table64 = nullptr;
  f->table_theta = nullptr;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaSuccess;  // no table: kernels evaluate sincos
  std::lock_guard<std::mutex> lock(g_rope_mutex);
  RopeTableAddrs& a = g_rope_addrs[dev];
  if (a.t32 == nullptr) {
    void *p32 = nullptr, *p64 = nullptr, *pt = nullptr;
    if ((err = cudaGetSymbolAddress(&p32, g_rope32)) != cudaSuccess) return err;
    if ((err = cudaGetSymbolAddress(&p64, g_rope64)) != cudaSuccess) return err;
    if ((err = cudaGetSymbolAddress(&pt, g_rope_theta)) != cudaSuccess) return err;
    a.t32 = static_cast<float2*>(p32);
    a.t64 = static_cast<double2*>(p64);
    a.theta = static_cast<double*>(pt);
  }
  int slot = -1;
  for (int s = 0; s < kRopeSlots && slot < 0; ++s)
    if (a.slot_theta[s] == theta) slot = s;
  if (slot < 0) {
    for (int s = 0; s < kRopeSlots && slot < 0; ++s)
      if (isnan(a.slot_theta[s])) slot = s;
    if (slot < 0) return cudaSuccess;  // every slot holds another theta: sincos
    // build, then tag -- in stream order; readers on any stream use the slot
    // only once they read the tag
    rope_table_kernel<<<(kRopeEntries + 255) / 256, 256, 0, stream>>>(*f, slot);
    rope_tag_kernel<<<1, 1, 0, stream>>>(slot, theta);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    a.slot_theta[slot] = theta;
  }
  f->table32 = a.t32 + static_cast<size_t>(slot) * kRopeEntries;
  f->table64 = a.t64 + static_cast<size_t>(slot) * kRopeEntries;
  f->table_theta = a.theta + slot;
  return cudaSuccess;
}

cudaError_t launch_kv_write_prefill(const uint16_t* k, const uint16_t* v, int num_tokens,
                                    const int32_t* token_offsets,
                                    const int32_t* start_positions, uint16_t* pool,
                                    int64_t num_pages, const int32_t* block_table,
                                    int max_blocks, int batch, const RopeFreqs& freqs,
                                    int32_t* dev_err, unsigned long long wait_ns,
                                    cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  // per device: opt in to the stage ring's shared memory, then size the
  // persistent grid from the resident CTAs per SM
  static std::atomic<int> grid_cap[64];
  const int slot = device & 63;
  int cap = grid_cap[slot].load(std::memory_order_acquire);
  if (cap == 0) {
    err = cudaFuncSetAttribute(kv_write_prefill_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kPfSmemBytes));
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cap, kv_write_prefill_kernel,
                                                        kPfThreads, kPfSmemBytes);
    if (err != cudaSuccess) return err;
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (err != cudaSuccess) return err;
    cap = (cap < 1 ? 1 : cap) * sms;
    grid_cap[slot].store(cap, std::memory_order_release);
  }
  const int nchunks = (num_tokens + kPfChunk - 1) / kPfChunk;
  const int ctas = nchunks < cap ? nchunks : cap;
  return launch_pdl(kv_write_prefill_kernel, dim3(ctas), dim3(kPfThreads), kPfSmemBytes, stream,
                    k, v, num_tokens, token_offsets, start_positions, pool, num_pages,
                    block_table, max_blocks, batch, freqs, dev_err, wait_ns);
}

cudaError_t launch_kv_append(const uint16_t* k_new, const uint16_t* v_new,
                             uint16_t* pool, int64_t num_pages,
                             const int32_t* block_table, int max_blocks,
                             const int32_t* positions, int batch,
                             const RopeFreqs& freqs, const uint16_t* q_in,
                             uint16_t* q_out, int32_t* dev_err,
                             cudaStream_t stream) {
  return launch_pdl(kv_append_kernel, dim3(batch), dim3(kAppendThreads), 0, stream, k_new,
                    v_new, pool, num_pages, block_table, max_blocks, positions, freqs, q_in,
                    q_out, dev_err);
}

}  // namespace pkv
