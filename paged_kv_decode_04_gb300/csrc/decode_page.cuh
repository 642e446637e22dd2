// decode_page.cuh -- the per-page arithmetic of paged decode attention, shared
// by every decomposition of the work (one warp, one page of one kv head, the
// group's 4 query rows), plus the fused append of the step's new token.
//
// Tiny-vLLM README ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here"), section "これまでの進捗", paged decode attention
// item: each query head streams its sequence's pages and accumulates
// softmax-weighted values with an FP32 online softmax.
//
// Tensor-core formulation (mma.sync m16n8k16, bf16 inputs, FP32 accumulators):
//   S^T = K Q^T   tokens as M (16 per page), query rows as N (4, padded to 8)
//   O^T += V^T P^T  head dims as M (4 tiles of 16), query rows as N
// K comes from the 128-byte-swizzled tile through ldmatrix, V through
// ldmatrix.trans.  The softmax keeps a lazily updated reference maximum per
// row: the accumulators are rescaled only when a score exceeds it by more
// than kRescaleLog2 (weights stay <= 2^kRescaleLog2); the final division by
// the running sum makes the result independent of the reference.  P enters
// the second product as two bf16 terms, hi = bf16(P) and lo = bf16(P - hi),
// so every weight keeps about 16 significant bits.
#pragma once

#include <math.h>
#include <stdint.h>

#include "pkv_device.cuh"

namespace pkv {

constexpr int kRowBytes = kHeadDim * 2;                // 128 B: one head's row
constexpr int kTileBytes = 2 * kPageSize * kRowBytes;  // 4 KiB: 16 K rows, 16 V rows
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned kFullMask = 0xFFFFFFFFu;

// Per-lane fragment coordinates and swizzled ldmatrix row offsets.
struct LaneGeom {
  int fg;           // fragment group: token (S^T) / head-dim (O^T) row
  int ft;           // thread in group: query rows 2ft, 2ft + 1
  int lr;           // ldmatrix: row inside an 8x8 matrix
  uint32_t k_row;   // K: byte offset of this lane's row (tokens 8*(li & 1) + lr)
  int k_chunk;      // K: 16-byte chunk offset within a k-step (li >> 1)
  uint32_t v_row;   // V: byte offset of this lane's row (tokens 8*(li >> 1) + lr)
  int v_chunk;      // V: chunk offset within a 16-dim slice (li & 1)
  int src_a, src_b; // lanes holding this lane's P^T entries in the S^T layout
  bool odd_row;     // this lane's P^T column is an odd query row

  __device__ __forceinline__ explicit LaneGeom(int lane) {
    fg = lane >> 2;
    ft = lane & 3;
    lr = lane & 7;
    const int li = lane >> 3;
    k_row = static_cast<uint32_t>((lr + 8 * (li & 1)) * kRowBytes);
    k_chunk = li >> 1;
    v_row = static_cast<uint32_t>((lr + 8 * (li >> 1)) * kRowBytes);
    v_chunk = li & 1;
    src_a = 8 * ft + (fg >> 1);
    src_b = src_a + 4;
    odd_row = (fg & 1) != 0;
  }
};

// Online-softmax state of one warp for the 4 query rows of one kv head.
struct AttnState {
  float m_ref[2];    // reference maxima of rows 2ft, 2ft+1 (log2 units)
  float l_run[2];    // this lane's share of the row sums
  float oacc[4][4];  // O^T fragments: dims 16mt + fg (+8) x rows 2ft (+1)

  __device__ __forceinline__ void reset() {
    m_ref[0] = m_ref[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
  }
};

// Q^T as the B operand of S^T = K Q^T for the 4 query rows starting at
// `qrow0` ([4][64] bf16): columns 0..3 are the rows, 4..7 zero padding.
__device__ __forceinline__ void load_q_frags(const uint16_t* qrow0, const LaneGeom& G,
                                             uint32_t (&qb)[4][2]) {
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(qrow0 + (G.fg & 3) * kHeadDim);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    qb[kk][0] = G.fg < kGroup ? qw[kk * 8 + G.ft] : 0u;
    qb[kk][1] = G.fg < kGroup ? qw[kk * 8 + 4 + G.ft] : 0u;
  }
}

// Fold one page (tile at shared address kt, `valid` live tokens) into S.
// c = softmax scale * log2(e).  Tokens at or past `valid` get no weight and
// their V rows are zeroed in the tile first (they may hold any bytes).
__device__ __forceinline__ void attend_page(uint32_t kt, int valid, const uint32_t (&qb)[4][2],
                                            float c, const LaneGeom& G, int lane,
                                            AttnState& S) {
  const uint32_t vt = kt + kPageSize * kRowBytes;
  float s[4] = {0.f, 0.f, 0.f, 0.f};  // tokens fg | fg+8 x rows 2ft, 2ft+1
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t ka[4];
    ldsm_x4(kt + G.k_row + (static_cast<uint32_t>((2 * kk + G.k_chunk) ^ G.lr) << 4), ka);
    mma_16816_bf16(s, ka, qb[kk][0], qb[kk][1]);
  }
  if (valid < kPageSize) {
    if (G.fg >= valid) s[0] = s[1] = -INFINITY;
    if (G.fg + 8 >= valid) s[2] = s[3] = -INFINITY;
    for (int idx = lane; idx < (kPageSize - valid) * 8; idx += 32)
      sts128_zero(vt + (valid + (idx >> 3)) * kRowBytes + ((idx & 7) << 4));
    __syncwarp();
  }
  float mx0 = fmaxf(s[0], s[2]) * c;
  float mx1 = fmaxf(s[1], s[3]) * c;
  const bool grow = mx0 > S.m_ref[0] + kRescaleLog2 || mx1 > S.m_ref[1] + kRescaleLog2;
  if (__any_sync(kFullMask, grow)) {
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, x));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, x));
    }
    const float mx[2] = {mx0, mx1};
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const float m_new = fmaxf(S.m_ref[rr], mx[rr]);
      const float alpha = fast_exp2(S.m_ref[rr] - m_new);  // 0 on the first page
      S.l_run[rr] *= alpha;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        S.oacc[mt][rr] *= alpha;
        S.oacc[mt][2 + rr] *= alpha;
      }
      S.m_ref[rr] = m_new;
    }
  }
  float p[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) p[e] = fast_exp2(fmaf(s[e], c, -S.m_ref[e & 1]));
  S.l_run[0] += p[0] + p[2];
  S.l_run[1] += p[1] + p[3];

  // P^T fragments, hi and lo bf16 terms: words (row 2ft | row 2ft+1) x
  // (token fg in the low half, token fg+8 in the high half).
  const uint32_t eh = pack_bf16x2(p[0], p[2]);
  const uint32_t oh = pack_bf16x2(p[1], p[3]);
  const uint32_t el = pack_bf16x2(p[0] - __uint_as_float(eh << 16),
                                  p[2] - __uint_as_float(eh & 0xFFFF0000u));
  const uint32_t ol = pack_bf16x2(p[1] - __uint_as_float(oh << 16),
                                  p[3] - __uint_as_float(oh & 0xFFFF0000u));
  uint32_t pb[2][2];
  {
    const uint32_t w_even[2] = {eh, el};
    const uint32_t w_odd[2] = {oh, ol};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t ea = __shfl_sync(kFullMask, w_even[h], G.src_a);
      const uint32_t oa = __shfl_sync(kFullMask, w_odd[h], G.src_a);
      const uint32_t eb = __shfl_sync(kFullMask, w_even[h], G.src_b);
      const uint32_t ob = __shfl_sync(kFullMask, w_odd[h], G.src_b);
      const uint32_t wa = G.odd_row ? oa : ea;  // tokens 2ft (lo), 2ft+8 (hi)
      const uint32_t wb = G.odd_row ? ob : eb;  // tokens 2ft+1 (lo), 2ft+9 (hi)
      pb[h][0] = prmt(wa, wb, 0x5410u);
      pb[h][1] = prmt(wa, wb, 0x7632u);
    }
  }
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    uint32_t va[4];
    ldsm_x4_trans(vt + G.v_row + (static_cast<uint32_t>((2 * mt + G.v_chunk) ^ G.lr) << 4), va);
    mma_16816_bf16(S.oacc[mt], va, pb[0][0], pb[0][1]);
    mma_16816_bf16(S.oacc[mt], va, pb[1][0], pb[1][1]);
  }
}

// Sum the lanes' shares of the row sums (lanes with the same ft).
__device__ __forceinline__ void reduce_row_sums(AttnState& S) {
#pragma unroll
  for (int x = 4; x <= 16; x <<= 1) {
    S.l_run[0] += __shfl_xor_sync(kFullMask, S.l_run[0], x);
    S.l_run[1] += __shfl_xor_sync(kFullMask, S.l_run[1], x);
  }
}

// The step's new token for kv head g of one sequence at position `pos`:
// lane i rotates pair (i, i + 32) of K (FP64, one rounding to bf16) and takes
// dims 2i, 2i + 1 of V.
struct AppendRow {
  uint16_t k1, k2;  // rotated K dims lane, lane + 32
  uint32_t v;       // V dims 2*lane, 2*lane + 1
};

__device__ __forceinline__ AppendRow make_append_row(const uint16_t* k_src,
                                                     const uint16_t* v_src, int pos,
                                                     const RopeFreqs& f, int lane) {
  AppendRow r;
  const uint16_t x1 = k_src[lane];
  const uint16_t x2 = k_src[lane + 32];
  r.v = reinterpret_cast<const uint32_t*>(v_src)[lane];
  const bool table_ok = rope_table_ready(f);
  RopeCS cs = rope_cs(f, table_ok, pos, lane);
  rotate_pair_rope(f, table_ok, pos, lane, cs, x1, x2, &r.k1, &r.k2);
  return r;
}

// Write the row into the pool slot (head g's 128 bytes of K and of V).
__device__ __forceinline__ void store_append_row(uint16_t* pool, int64_t page, int slot, int g,
                                                 const AppendRow& r, int lane) {
  const int64_t row = kNumKvHeads * kHeadDim;
  uint16_t* kd = pool + ((page * 2 + 0) * kPageSize + slot) * row + g * kHeadDim;
  uint16_t* vd = pool + ((page * 2 + 1) * kPageSize + slot) * row + g * kHeadDim;
  kd[lane] = r.k1;
  kd[lane + 32] = r.k2;
  reinterpret_cast<uint32_t*>(vd)[lane] = r.v;
}

// Put the row into the swizzled tile at shared address kt (row `slot`).
__device__ __forceinline__ void patch_append_row(uint32_t kt, int slot, const AppendRow& r,
                                                 int lane) {
  const uint32_t sw = static_cast<uint32_t>(slot & 7);
  const uint32_t kr = kt + slot * kRowBytes;
  const uint32_t vr = kt + (kPageSize + slot) * kRowBytes;
  const uint32_t ln = static_cast<uint32_t>(lane);
  sts16(kr + (((ln >> 3) ^ sw) << 4) + ((ln & 7) << 1), r.k1);
  sts16(kr + (((4u + (ln >> 3)) ^ sw) << 4) + ((ln & 7) << 1), r.k2);
  sts32(vr + (((ln >> 2) ^ sw) << 4) + ((ln & 3) << 2), r.v);
  __syncwarp();
}

}  // namespace pkv
