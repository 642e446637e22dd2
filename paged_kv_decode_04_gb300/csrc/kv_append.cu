// kv_append.cu -- decode-time KV append with rotate-half RoPE.
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗", KV page pool item: each
// decode step adds one new token per sequence at its absolute RoPE position
// into the sequence's page slot of the shared BF16 pool.
//
// One CTA per sequence.  Warp 0 evaluates the 32 (cos, sin) pairs of the
// token's position in FP64 once; all 256 threads then rotate the 8 kv heads'
// keys (one thread per (head, frequency) pair), copy the values, and, when
// asked, rotate the 32 query heads out of place.  The rotation is FP64 with
// separately rounded products (no contraction) and one rounding to bf16, so
// the stored keys are a deterministic function of the inputs.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kAppendThreads = 256;
constexpr int kHalf = kHeadDim / 2;

__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(const uint16_t* __restrict__ k_new,
                     const uint16_t* __restrict__ v_new,
                     uint16_t* __restrict__ pool, int64_t num_pages,
                     const int32_t* __restrict__ block_table, int max_blocks,
                     const int32_t* __restrict__ positions, RopeFreqs freqs,
                     const uint16_t* __restrict__ q_in,
                     uint16_t* __restrict__ q_out, int32_t* dev_err) {
  __shared__ double s_cos[kHalf];
  __shared__ double s_sin[kHalf];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int h = tid / kHalf, i = tid % kHalf;
  const int64_t row = kNumKvHeads * kHeadDim;  // elements per (kv, slot)
  const int64_t src = static_cast<int64_t>(b) * row;

  // Everything that does not depend on the position is fetched first so that
  // its latency overlaps the position -> page lookup and the FP64 sincos.
  const uint16_t k1 = k_new[src + h * kHeadDim + i];
  const uint16_t k2 = k_new[src + h * kHeadDim + i + kHalf];
  const uint32_t vw = reinterpret_cast<const uint32_t*>(v_new + src)[tid];
  const int32_t pos = positions[b];
  const bool pos_ok = pos >= 0 && pos < max_blocks * kPageSize;
  const int32_t page =
      pos_ok ? block_table[static_cast<int64_t>(b) * max_blocks + pos / kPageSize] : -1;

  if (tid < kHalf) {
    const double angle = __dmul_rn(static_cast<double>(pos), freqs.inv_freq[tid]);
    double sn, cs;
    sincos(angle, &sn, &cs);
    s_cos[tid] = cs;
    s_sin[tid] = sn;
  }
  __syncthreads();

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
      rotate_pair(x1[k], x2[k], s_cos[i], s_sin[i], &y1, &y2);
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
  // Keys: thread (h, i) rotates pair i of kv head h.
  uint16_t y1, y2;
  rotate_pair(k1, k2, s_cos[i], s_sin[i], &y1, &y2);
  k_dst[h * kHeadDim + i] = y1;
  k_dst[h * kHeadDim + i + kHalf] = y2;
  // Values: 512 bf16 = 256 words, one per thread.
  reinterpret_cast<uint32_t*>(v_dst)[tid] = vw;
}

// Prefill write: one warp per token.  The token's sequence is found by a
// binary search over token_offsets; lane i evaluates the (cos, sin) pair i of
// the token's position in FP64 and rotates pair i of all 8 kv heads; the 512
// value elements are copied as 8 words per lane.
constexpr int kPrefillTokensPerCta = 8;

__global__ void __launch_bounds__(kPrefillTokensPerCta * 32)
    kv_write_prefill_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                            int num_tokens, const int32_t* __restrict__ token_offsets,
                            const int32_t* __restrict__ start_positions,
                            uint16_t* __restrict__ pool, int64_t num_pages,
                            const int32_t* __restrict__ block_table, int max_blocks, int batch,
                            RopeFreqs freqs, int32_t* dev_err) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kPrefillTokensPerCta + (threadIdx.x >> 5);
  if (t >= num_tokens) return;
  // largest b with token_offsets[b] <= t
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (token_offsets[mid] <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int32_t first = token_offsets[b];
  if (t < first || t >= token_offsets[b + 1]) {
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
  const int64_t row = kNumKvHeads * kHeadDim;
  const int64_t src = static_cast<int64_t>(t) * row;
  uint16_t* k_dst = pool + ((static_cast<int64_t>(page) * 2 + 0) * kPageSize + slot) * row;
  uint16_t* v_dst = pool + ((static_cast<int64_t>(page) * 2 + 1) * kPageSize + slot) * row;
  double sn, cs;
  sincos(__dmul_rn(static_cast<double>(pos), freqs.inv_freq[lane]), &sn, &cs);
#pragma unroll
  for (int h = 0; h < kNumKvHeads; ++h) {
    uint16_t y1, y2;
    rotate_pair(k[src + h * kHeadDim + lane], k[src + h * kHeadDim + lane + kHalf], cs, sn,
                &y1, &y2);
    k_dst[h * kHeadDim + lane] = y1;
    k_dst[h * kHeadDim + lane + kHalf] = y2;
  }
  const uint32_t* vs = reinterpret_cast<const uint32_t*>(v + src);
  uint32_t* vd = reinterpret_cast<uint32_t*>(v_dst);
#pragma unroll
  for (int j = 0; j < static_cast<int>(row / 2) / 32; ++j) vd[lane + 32 * j] = vs[lane + 32 * j];
}

}  // namespace

cudaError_t launch_kv_write_prefill(const uint16_t* k, const uint16_t* v, int num_tokens,
                                    const int32_t* token_offsets,
                                    const int32_t* start_positions, uint16_t* pool,
                                    int64_t num_pages, const int32_t* block_table,
                                    int max_blocks, int batch, const RopeFreqs& freqs,
                                    int32_t* dev_err, cudaStream_t stream) {
  const int ctas = (num_tokens + kPrefillTokensPerCta - 1) / kPrefillTokensPerCta;
  kv_write_prefill_kernel<<<ctas, kPrefillTokensPerCta * 32, 0, stream>>>(
      k, v, num_tokens, token_offsets, start_positions, pool, num_pages, block_table,
      max_blocks, batch, freqs, dev_err);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const uint16_t* k_new, const uint16_t* v_new,
                             uint16_t* pool, int64_t num_pages,
                             const int32_t* block_table, int max_blocks,
                             const int32_t* positions, int batch,
                             const RopeFreqs& freqs, const uint16_t* q_in,
                             uint16_t* q_out, int32_t* dev_err,
                             cudaStream_t stream) {
  kv_append_kernel<<<batch, kAppendThreads, 0, stream>>>(
      k_new, v_new, pool, num_pages, block_table, max_blocks, positions, freqs,
      q_in, q_out, dev_err);
  return cudaGetLastError();
}

}  // namespace pkv
