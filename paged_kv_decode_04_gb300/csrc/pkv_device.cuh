// pkv_device.cuh -- sm_103a device helpers for libpkv: shared-memory
// mbarriers, TMA tensor copies, packed FP32 arithmetic and bf16 bit tricks.
// Everything here is inline PTX or plain integer/float code; no library
// kernels are used on the decode path.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

// Upper bound for one in-kernel wait on a page copy: past it the kernel
// records kErrTimeout and stops waiting instead of spinning forever.  The
// waits on a kernel's progress take the per-call limit (AttnArgs::wait_ns,
// this value unless the caller set another); the drains after a timeout
// always take this one.
constexpr unsigned long long kWaitLimitNs = kDefaultWaitNs;

// Programmatic dependent launch.  Every library kernel is launched allowed to
// start before the previous kernel on its stream has finished; it calls
// wait_for_prior_grids() (which returns once the prior grids have completed
// and their writes are visible, and at once when there is no such dependency)
// before it reads anything it uses, and allow_dependent_grids() so that the
// next kernel may be scheduled in turn.  Before the wait, the attention
// kernels only prefetch into L2 (the addresses read there serve as hints).
__device__ __forceinline__ void wait_for_prior_grids() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_grids() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void record_error(int32_t* dev_err, int bits) {
  if (dev_err != nullptr) atomicOr(dev_err, bits);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking look at phase `parity` of a barrier.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` of a barrier, giving up after limit_ns nanoseconds
// (0: a single non-blocking look, so a phase that has not completed by then
// counts as a timeout).  The kernels' waits on their own progress take the
// caller's limit (pkv_set_wait_limit_ns, 2 s by default); the waits that
// drain a CTA's own copies and MMAs after a timeout always take
// kWaitLimitNs, so nothing the CTA started is still running when it exits.
//
// The time waited is the sum of the forward steps of %globaltimer between
// looks, each counted up to kTimerStepCapNs: the global timer is kept in step
// with the host clock, and a step back (which an unsigned difference from a
// start time would read as an enormous wait) or a jump forward must not end a
// wait early.
constexpr unsigned long long kTimerStepCapNs = 1000000ull;  // 1 ms

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (limit_ns == 0) return mbar_test_wait(bar, parity);
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long last = global_timer_ns(), waited = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 0u) {
      const unsigned long long now = global_timer_ns();
      if (now > last) waited += min(now - last, kTimerStepCapNs);
      last = now;
      if (waited > limit_ns) return false;
    }
  }
}

// ----------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Loads that bypass L1 (cached in L2 only).  The attention kernels use them
// for the reads they make before griddepcontrol.wait: the previous grid may
// still be writing those words, and a stale line must not stay in L1 for the
// reads made after the wait.
__device__ __forceinline__ int ld_cg(const int32_t* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int4 ld_cg(const int4* p) {
  int4 v;
  asm volatile("ld.global.cg.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Prefetch of one tensor-map box into L2 (no shared memory, no barrier).  L2
// is coherent for every SM, so a prefetch can never make a later read stale:
// a write that lands after it updates the same L2 lines.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int x, int y, int z,
                                                   int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   map),
               "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

// 3-D tiled tensor copy global -> shared, completion signalled on `bar`
// (transaction bytes).  Coordinates are element indices, innermost first.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int x, int y, int z,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// Contiguous global -> shared copy of `bytes` bytes (a multiple of 16; both
// addresses 16-byte aligned), completion signalled on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once per step (the K/V pages).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------- shared memory I/O --

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// ------------------------------------------------------- packed FP32 ops --

// d = a * b + c on two FP32 lanes at once (sm_100+ packed FMA).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

// 2^x on the special-function unit (relative error ~2^-22; ex2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// --------------------------------------------------------------- bf16 --

// Two bf16 packed in one 32-bit word -> two floats (low half first).
// A bf16 is the upper half of a binary32, so widening is a shift / mask.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float bf16_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// binary32 -> bf16, round to nearest even (NaN stays a quiet NaN).
__device__ __forceinline__ uint16_t float_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Two floats -> packed bf16 pair (lo in the low half), each rounded to
// nearest even by the conversion instruction.
__device__ __forceinline__ uint32_t cvt_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// binary64 -> bf16 in ONE rounding step (round to nearest even), done on the
// bit pattern: keep the sign, rebias the exponent from 1023 to 127, keep 7
// mantissa bits and round on the 45 discarded ones; values below the bf16
// normal range are shifted into the subnormal grid (spacing 2^-133) first.
__device__ __forceinline__ uint16_t double_to_bf16_rne(double x) {
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(x));
  const uint16_t sign = static_cast<uint16_t>((u >> 48) & 0x8000u);
  const uint64_t a = u & 0x7FFFFFFFFFFFFFFFull;
  if (a > 0x7FF0000000000000ull) return sign | 0x7FC0u;  // NaN
  if (a == 0x7FF0000000000000ull) return sign | 0x7F80u;  // inf
  const int e = static_cast<int>(a >> 52) - 1023;         // unbiased exponent
  if (e > 127) return sign | 0x7F80u;                      // overflow
  if (e >= -126) {
    // bits [51:0] mantissa; rebias exponent into a 60-bit field so that the
    // bf16 pattern is (r >> 45) and a carry runs into the exponent (or inf).
    uint64_t r = (static_cast<uint64_t>(e + 127) << 52) | (a & 0x000FFFFFFFFFFFFFull);
    r += 0x00000FFFFFFFFFFFull + ((r >> 45) & 1ull);
    return sign | static_cast<uint16_t>(r >> 45);
  }
  if ((a >> 52) == 0) return sign;  // binary64 subnormal: far below 2^-134
  // subnormal bf16: value = sig * 2^(e-52), grid spacing 2^-133
  const uint64_t sig = (a & 0x000FFFFFFFFFFFFFull) | (1ull << 52);
  const int shift = -e - 81;  // = 52 - (e + 133)
  if (shift >= 54) return sign;
  uint64_t q = sig >> shift;
  const uint64_t rem = sig & ((1ull << shift) - 1ull);
  const uint64_t half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (q & 1ull))) ++q;
  return sign | static_cast<uint16_t>(q);
}


// Rotate-half RoPE of one pair: (x1, x2) -> (x1*c - x2*s, x2*c + x1*s), each
// product and the sum rounded in FP64 (no contraction), then one rounding to
// bf16.  This is the defining evaluation; rotate_pair_rope reaches the same
// bits faster.
__device__ __forceinline__ void rotate_pair(uint16_t h1, uint16_t h2, double c,
                                            double s, uint16_t* o1,
                                            uint16_t* o2) {
  const double x1 = static_cast<double>(bf16_to_float(h1));
  const double x2 = static_cast<double>(bf16_to_float(h2));
  const double y1 = __dsub_rn(__dmul_rn(x1, c), __dmul_rn(x2, s));
  const double y2 = __dadd_rn(__dmul_rn(x2, c), __dmul_rn(x1, s));
  *o1 = double_to_bf16_rne(y1);
  *o2 = double_to_bf16_rne(y2);
}

// True when every value within `err` of y rounds to the same bf16 as y: y is
// farther than err from both bf16 rounding midpoints around it.
__device__ __forceinline__ bool bf16_rounding_stable(float y, float err) {
  const float ay = fabsf(y);
  if (!(ay >= 0x1p-100f) || !(ay < 0x1p+126f)) return false;  // tiny, huge, NaN
  const uint32_t hi = __float_as_uint(ay) & 0xFFFF0000u;
  const float m_hi = __uint_as_float(hi | 0x8000u);               // above (or at) ay's bf16
  const float m_lo = __uint_as_float((hi - 0x10000u) | 0x8000u);  // below it
  return fabsf(ay - m_hi) > err && fabsf(ay - m_lo) > err;
}

// cos/sin of pair i at position pos: from the device table when it holds
// this theta, else evaluated here (identical values either way).
struct RopeCS {
  float c32, s32;    // the double values rounded to float
  double c64, s64;   // valid when have64
  bool have64;
};

__device__ __forceinline__ RopeCS rope_cs(const RopeFreqs& f, bool table_ok, int pos, int i) {
  RopeCS r;
  if (table_ok && pos >= 0 && pos < kRopeTablePositions) {
    const float2 t = f.table32[pos * 32 + i];
    r.c32 = t.x;
    r.s32 = t.y;
    r.c64 = r.s64 = 0.0;
    r.have64 = false;
  } else {
    sincos(__dmul_rn(static_cast<double>(pos), f.inv_freq[i]), &r.s64, &r.c64);
    r.c32 = static_cast<float>(r.c64);
    r.s32 = static_cast<float>(r.s64);
    r.have64 = true;
  }
  return r;
}

// Error allowance of the FP32 rotation (see rotate_pair_rope).
__device__ __forceinline__ float rope_fp32_allowance(float x1, float x2, float y) {
  return 0x1p-22f * (fabsf(x1) + fabsf(x2) + fabsf(y));
}

// The result of rotate_pair with c, s = cos/sin of pair i at pos, computed
// in FP32 whenever that is provably the same bf16.  With c32 = float(c),
// s32 = float(s), y = fma(x1, c32, -float(x2*s32)) differs from the FP64
// value by at most 2^-24 * (2|x1| + 2|x2| + |y|) plus about 2^-51 * (|x1| +
// |x2|), which is at most half of rope_fp32_allowance; if y is farther than
// the allowance from both bf16 rounding midpoints around it, both values
// round to the same bf16.  Otherwise (about one element in a thousand,
// mostly under cancellation) the element is redone by rotate_pair's FP64
// arithmetic.
__device__ __forceinline__ void rotate_pair_rope(const RopeFreqs& f, bool table_ok, int pos,
                                                 int i, RopeCS& cs, uint16_t h1, uint16_t h2,
                                                 uint16_t* o1, uint16_t* o2) {
  const float x1 = bf16_to_float(h1);
  const float x2 = bf16_to_float(h2);
  const float y1 = fmaf(x1, cs.c32, -(x2 * cs.s32));
  const float y2 = fmaf(x2, cs.c32, x1 * cs.s32);
  const bool ok1 = bf16_rounding_stable(y1, rope_fp32_allowance(x1, x2, y1));
  const bool ok2 = bf16_rounding_stable(y2, rope_fp32_allowance(x1, x2, y2));
  if (ok1 && ok2) {
    *o1 = float_to_bf16_rne(y1);
    *o2 = float_to_bf16_rne(y2);
    return;
  }
  if (!cs.have64) {
    if (table_ok && pos >= 0 && pos < kRopeTablePositions) {
      const double2 t = f.table64[pos * 32 + i];
      cs.c64 = t.x;
      cs.s64 = t.y;
    } else {
      sincos(__dmul_rn(static_cast<double>(pos), f.inv_freq[i]), &cs.s64, &cs.c64);
    }
    cs.have64 = true;
  }
  uint16_t e1, e2;
  rotate_pair(h1, h2, cs.c64, cs.s64, &e1, &e2);
  *o1 = ok1 ? float_to_bf16_rne(y1) : e1;
  *o2 = ok2 ? float_to_bf16_rne(y2) : e2;
}

// One output element of rotate_pair for pair i at pos: first ? x1*c - x2*s
// : x2*c + x1*s, with the same FP32 fast path and FP64 redo as
// rotate_pair_rope (c32, s32: the float cos/sin of the pair).
__device__ __forceinline__ uint16_t rope_one(const RopeFreqs& f, bool table_ok, int pos, int i,
                                             bool first, float c32, float s32, uint16_t h1,
                                             uint16_t h2) {
  const float x1 = bf16_to_float(h1);
  const float x2 = bf16_to_float(h2);
  const float y = first ? fmaf(x1, c32, -(x2 * s32)) : fmaf(x2, c32, x1 * s32);
  if (bf16_rounding_stable(y, rope_fp32_allowance(x1, x2, y))) return float_to_bf16_rne(y);
  double c64, s64;
  if (table_ok && pos >= 0 && pos < kRopeTablePositions) {
    const double2 t = f.table64[pos * 32 + i];
    c64 = t.x;
    s64 = t.y;
  } else {
    sincos(__dmul_rn(static_cast<double>(pos), f.inv_freq[i]), &s64, &c64);
  }
  uint16_t e1, e2;
  rotate_pair(h1, h2, c64, s64, &e1, &e2);
  return first ? e1 : e2;
}

__device__ __forceinline__ bool rope_table_ready(const RopeFreqs& f) {
  return f.table_theta != nullptr && *f.table_theta == f.theta;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ------------------------------------------------ warp-level tensor ops --

// Four 8x8 b16 matrices from shared memory; lane l supplies the row address
// of row (l & 7) of matrix (l >> 3); register i receives matrix i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// As ldsm_x4, each matrix transposed on the way into registers.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, FP32 accumulators.
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Byte permute of two words (PTX prmt, default mode).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}


// ------------------------------------------------------------- tcgen05 --
// Fifth-generation tensor cores: one thread issues an MMA for the whole CTA,
// operands come from shared memory through 64-bit matrix descriptors and the
// FP32 accumulator lives in tensor memory (TMEM: 128 lanes x 512 columns of
// 32 bits per SM), which warps read and write with tcgen05.ld / tcgen05.st
// (warp w reaches lanes 32 (w mod 4) .. + 31).

// Allocate `ncols` TMEM columns (a power of two >= 32); the warp-collective
// instruction writes the TMEM address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_alloc_permit() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Order tcgen05 operations around a thread synchronisation (barrier or
// mbarrier): `before` on the signalling side, `after` on the waiting side.
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand whose rows
// are 128 bytes (the pattern TMA's 128B swizzle writes: 16-byte chunk c of
// row r sits at chunk c ^ (r mod 8); groups of 8 rows are 1024 bytes apart).
// Bits: start address >> 4 [0,14), leading byte offset >> 4 [16,30), stride
// byte offset >> 4 [32,46), descriptor version 1 at bit 46, base offset 0
// (every tile starts on a 1024-byte boundary; a start advanced by a multiple
// of 32 bytes inside the first row selects a K slice), swizzle mode 2
// (128 bytes) at [61,64).  Both offsets are 1024 bytes: for a K-major operand
// only the 8-row group stride is used; for an MN-major operand 64 bf16 wide
// (one swizzle row) the group stride along K is the only one used either way.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1024 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma.kind::f16 with bf16 A and B and an
// FP32 accumulator: D format [4,6) = 1 (f32), A format [7,10) = 1 (bf16),
// B format [10,13) = 1, A major bit 15 (0: K-major), B major bit 16
// (1: MN-major), N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.  A sits in TMEM
// row r in lane r, its K elements packed two bf16 per 32-bit column (the
// lower-indexed one in the low half): a K = 16 slice is 8 columns.
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread has
// issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Registers written by tcgen05.ld hold their values only after
// tcgen05.wait::ld: passing them through an empty volatile statement placed
// after the wait keeps every use of them behind it.
__device__ __forceinline__ void reg_after_wait(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace pkv
