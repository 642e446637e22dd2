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

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kAppendThreads = 256;
constexpr int kHalf = kHeadDim / 2;
constexpr int kRopeEntries = kRopeTablePositions * kHalf;

// This device's cos/sin table and the theta it holds (NaN = none).
__device__ __align__(16) float2 g_rope32[kRopeEntries];
__device__ __align__(16) double2 g_rope64[kRopeEntries];
__device__ double g_rope_theta;

__global__ void rope_tag_kernel(double value) { g_rope_theta = value; }

__global__ void __launch_bounds__(256) rope_table_kernel(RopeFreqs f) {
  const int e = blockIdx.x * 256 + threadIdx.x;
  if (e >= kRopeEntries) return;
  const int pos = e / kHalf, i = e % kHalf;
  double sn, cs;
  sincos(__dmul_rn(static_cast<double>(pos), f.inv_freq[i]), &sn, &cs);
  g_rope64[e] = make_double2(cs, sn);
  g_rope32[e] = make_float2(static_cast<float>(cs), static_cast<float>(sn));
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

// Prefill write: one warp per token.  The token's sequence is found by a
// binary search over token_offsets.  Lane l holds bf16 elements
// [16l, 16l + 16) of the token's 512-element K row (kv head l / 4, dims
// 16 (l % 4) ..) and of its V row, loaded and stored 16 bytes at a time; the
// rotation partner of dims 0..31 is dims 32..63, i.e. lane l ^ 2, reached
// with shuffles.  Lanes holding dims < 32 produce x1*c - x2*s, the others
// x2*c + x1*s, for 16 pairs each.
constexpr int kPrefillTokensPerCta = 8;

// Batches up to this size search token_offsets in shared memory.
constexpr int kPrefillSmemBatch = 2048;

__global__ void __launch_bounds__(kPrefillTokensPerCta * 32, 4)
    kv_write_prefill_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                            int num_tokens, const int32_t* __restrict__ token_offsets,
                            const int32_t* __restrict__ start_positions,
                            uint16_t* __restrict__ pool, int64_t num_pages,
                            const int32_t* __restrict__ block_table, int max_blocks, int batch,
                            RopeFreqs freqs, int32_t* dev_err) {
  __shared__ int32_t s_off[kPrefillSmemBatch + 1];
  wait_for_prior_grids();
  allow_dependent_grids();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kPrefillTokensPerCta + (threadIdx.x >> 5);
  const bool smem_offsets = batch <= kPrefillSmemBatch;
  if (smem_offsets) {
    for (int i = threadIdx.x; i <= batch; i += blockDim.x) s_off[i] = token_offsets[i];
    __syncthreads();
  }
  if (t >= num_tokens) return;
  const int32_t* off = smem_offsets ? s_off : token_offsets;
  const int64_t row = kNumKvHeads * kHeadDim;
  const int64_t src = static_cast<int64_t>(t) * row;
  // position-independent loads first: this lane's 16 K and 16 V elements
  const uint4* ks = reinterpret_cast<const uint4*>(k + src) + 2 * lane;
  const uint4* vs = reinterpret_cast<const uint4*>(v + src) + 2 * lane;
  const uint4 k0 = ks[0], k1 = ks[1];
  const uint4 v0 = vs[0], v1 = vs[1];
  // largest b with token_offsets[b] <= t
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int32_t first = off[b];
  if (t < first || t >= off[b + 1]) {
    if (lane == 0) record_error(dev_err, kErrOffsets);
    return;
  }
  const int32_t pos = start_positions[b] + (t - first);
  if (pos < 0 || pos >= max_blocks * kPageSize) {
    if (lane == 0) record_error(dev_err, kErrPosition);
    return;
  }
  const int32_t page = block_table[static_cast<int64_t>(b) * max_blocks + pos / kPageSize];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) record_error(dev_err, kErrPage);
    return;
  }
  const int slot = pos % kPageSize;
  uint16_t* k_dst = pool + ((static_cast<int64_t>(page) * 2 + 0) * kPageSize + slot) * row;
  uint16_t* v_dst = pool + ((static_cast<int64_t>(page) * 2 + 1) * kPageSize + slot) * row;
  reinterpret_cast<uint4*>(v_dst)[2 * lane] = v0;
  reinterpret_cast<uint4*>(v_dst)[2 * lane + 1] = v1;

  const bool first_half = (lane & 2) == 0;  // my dims are the x1 side of their pairs
  const bool table_ok = rope_table_ready(freqs) && pos < kRopeTablePositions;
  uint4* kd = reinterpret_cast<uint4*>(k_dst) + 2 * lane;
#pragma unroll
  for (int part = 0; part < 2; ++part) {  // 8 pairs at a time
    const uint4 mine4 = part ? k1 : k0;
    const uint32_t mine[4] = {mine4.x, mine4.y, mine4.z, mine4.w};
    uint32_t other[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) other[e] = __shfl_xor_sync(0xFFFFFFFFu, mine[e], 2);
    const int i0 = 16 * (lane & 1) + 8 * part;  // pair index of element 0 of this part
    float c32[8], s32[8];
    if (table_ok) {
      const float4* tc = reinterpret_cast<const float4*>(freqs.table32 + pos * kHalf + i0);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 q = tc[e];
        c32[2 * e] = q.x;
        s32[2 * e] = q.y;
        c32[2 * e + 1] = q.z;
        s32[2 * e + 1] = q.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        double sn, cs;
        sincos(__dmul_rn(static_cast<double>(pos), freqs.inv_freq[i0 + e]), &sn, &cs);
        c32[e] = static_cast<float>(cs);
        s32[e] = static_cast<float>(sn);
      }
    }
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint16_t r[2];
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int el = 2 * e + hlf;
        const uint16_t a = static_cast<uint16_t>(hlf ? mine[e] >> 16 : mine[e] & 0xFFFFu);
        const uint16_t o = static_cast<uint16_t>(hlf ? other[e] >> 16 : other[e] & 0xFFFFu);
        r[hlf] = rope_one(freqs, table_ok, pos, i0 + el, first_half, c32[el], s32[el],
                          first_half ? a : o, first_half ? o : a);
      }
      out[e] = static_cast<uint32_t>(r[0]) | (static_cast<uint32_t>(r[1]) << 16);
    }
    kd[part] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// Device addresses of this device's table, looked up once per device.
struct RopeTableAddrs {
  float2* t32 = nullptr;
  double2* t64 = nullptr;
  double* theta = nullptr;
  double built_for = NAN;  // theta of the last rebuild enqueued on this device
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
  if (!(a.built_for == theta)) {
    // invalidate, rebuild, then publish the theta -- in stream order
    rope_tag_kernel<<<1, 1, 0, stream>>>(NAN);
    rope_table_kernel<<<(kRopeEntries + 255) / 256, 256, 0, stream>>>(*f);
    rope_tag_kernel<<<1, 1, 0, stream>>>(theta);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    a.built_for = theta;
  }
  f->table32 = a.t32;
  f->table64 = a.t64;
  f->table_theta = a.theta;
  return cudaSuccess;
}

cudaError_t launch_kv_write_prefill(const uint16_t* k, const uint16_t* v, int num_tokens,
                                    const int32_t* token_offsets,
                                    const int32_t* start_positions, uint16_t* pool,
                                    int64_t num_pages, const int32_t* block_table,
                                    int max_blocks, int batch, const RopeFreqs& freqs,
                                    int32_t* dev_err, cudaStream_t stream) {
  const int ctas = (num_tokens + kPrefillTokensPerCta - 1) / kPrefillTokensPerCta;
  return launch_pdl(kv_write_prefill_kernel, dim3(ctas), dim3(kPrefillTokensPerCta * 32), 0,
                    stream, k, v, num_tokens, token_offsets, start_positions, pool, num_pages,
                    block_table, max_blocks, batch, freqs, dev_err);
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
