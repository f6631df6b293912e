// fp8q_device.cuh -- device-side building blocks of the fused row kernels (sm_103a).
//
// Packed-type conversions are single PTX instructions:
//   cvt.rn.bf16x2.f32           two fp32 -> two bf16, round-to-nearest-even
//   cvt.rn.satfinite.e4m3x2.f32 two fp32 -> two E4M3 codes, RNE, saturating to +-448
//   fma.rn.bf16x2               two single-rounded bf16 fused multiply-adds
// Double-float ("dd") helpers form the LayerNorm row constants at ~2^-45 relative precision
// with fp32 arithmetic only (GB300's fp64 rate is far too low for a per-element path). They
// follow the error-free transformations of Knuth (TwoSum), Dekker (FastTwoSum) and the
// FMA-based TwoProduct; all operations use explicit _rn intrinsics so the compiler can
// neither contract nor reassociate them.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8q {

// ------------------------------------------------------------------------------------------
// bf16 / e4m3 packing
// ------------------------------------------------------------------------------------------

// Low / high bf16 of a packed pair as fp32 (exact: bf16 is the top half of a binary32).
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Pack two fp32 into bf16x2 with RNE: `lo` goes to bits 0..15, `hi` to bits 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> two E4M3 codes (RNE, satfinite): `lo` in bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Elementwise single-rounded bf16 FMA on packed pairs: a * b + c.
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Programmatic dependent launch: wait until the grids this launch depends on have completed
// and their memory is visible (returns at once when there is no such grid).
__device__ __forceinline__ void wait_for_producers() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream (launched with programmatic serialization) be scheduled
// onto SMs this grid frees; it still waits in griddepcontrol.wait for this grid to complete.
// Only for persistent grids whose CTAs are all resident from the start, so waiting dependents
// never hold resources one of our own CTAs still needs.
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Streaming 16-byte global accesses (data touched once).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint2* p, uint2 v) { __stcs(p, v); }

// ------------------------------------------------------------------------------------------
// double-float arithmetic
// ------------------------------------------------------------------------------------------

struct dd {
  float hi, lo;
};

// Knuth TwoSum: s = RN(a + b), e exact error (any magnitudes).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
}

// Dekker FastTwoSum: exact when |a| >= |b| (or a == 0).
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// TwoProduct with FMA: p = RN(a * b), e exact error.
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
  p = __fmul_rn(a, b);
  e = __fmaf_rn(a, b, -p);
}

__device__ __forceinline__ dd dd_add(dd a, dd b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  dd r;
  fast_two_sum(s, e, r.hi, r.lo);
  return r;
}

__device__ __forceinline__ dd dd_neg(dd a) { return dd{-a.hi, -a.lo}; }

// a / c for a positive integer c < 2^16 (the row width) given rc = RN(1/c): q1 = RN(a.hi * rc)
// lies within two ulps of a.hi / c, so the remainder a.hi - q1 c (at most 2 ulp(q1) c, on the
// grid of ulp(q1) times the lowest set bit of c) is exact in one FMA while q1 is normal; the
// second quotient digit comes from it. No division instruction sits on the row's critical path.
__device__ __forceinline__ dd dd_div_f(dd a, float c, float rc) {
  const float q1 = __fmul_rn(a.hi, rc);
  const float rem = __fadd_rn(__fmaf_rn(-q1, c, a.hi), a.lo);
  const float q2 = __fmul_rn(rem, rc);
  dd r;
  fast_two_sum(q1, q2, r.hi, r.lo);
  return r;
}

__device__ __forceinline__ dd dd_sqr(dd a) {
  float p, pe;
  two_prod(a.hi, a.hi, p, pe);
  pe = __fmaf_rn(__fmul_rn(2.0f, a.hi), a.lo, pe);
  dd r;
  fast_two_sum(p, pe, r.hi, r.lo);
  return r;
}

// 1 / sqrt(w) for w > 0 as a double-float: correctly rounded fp32 seed, then one Newton
// step r <- r0 + r0 * (1 - w r0^2) / 2 evaluated with the residual 1 - w r0^2 in exact
// arithmetic up to the w.lo term (relative error ~2^-46).
__device__ __forceinline__ dd dd_rsqrt(dd w) {
  const float r0 = __frsqrt_rn(w.hi);
  float a, b;
  two_prod(r0, r0, a, b);          // r0^2 = a + b exactly
  float p, pe;
  two_prod(w.hi, a, p, pe);        // w.hi * a = p + pe exactly
  const float rest = __fadd_rn(pe, __fmaf_rn(w.hi, b, __fmul_rn(w.lo, a)));
  const float h = __fsub_rn(__fsub_rn(1.0f, p), rest);  // 1 - p is exact (p ~ 1)
  const float corr = __fmul_rn(__fmul_rn(r0, h), 0.5f);
  dd r;
  fast_two_sum(r0, corr, r.hi, r.lo);
  return r;
}

// Row constants of the LayerNorm, from exact-ish row sums sum(x) and sum(x^2).
struct RowConst {
  float mu_hi;     // mean, high part
  float mu_lo;     // mean, low part
  float r_hi;      // 1/sqrt(var + eps), high part
  float r_lo;      // low part
  float c;         // RN(-mu_lo * r_hi): folds the low part of the mean into one FMA
  float t_small;   // |t| below this goes to the exact path (absolute error dominates there)
};

// rcols = RN(1 / cols).
__device__ __forceinline__ RowConst row_constants(dd sum, dd sumsq, float cols, float rcols,
                                                  float eps) {
  const dd mu = dd_div_f(sum, cols, rcols);
  const dd e2 = dd_div_f(sumsq, cols, rcols);
  dd var = dd_add(e2, dd_neg(dd_sqr(mu)));
  if (!(var.hi > 0.0f)) var = dd{0.0f, 0.0f};  // exact zero for constant rows; no negatives
  float ws, we;
  two_sum(var.hi, eps, ws, we);
  dd w;
  fast_two_sum(ws, __fadd_rn(we, var.lo), w.hi, w.lo);
  const dd r = dd_rsqrt(w);
  RowConst k;
  k.mu_hi = mu.hi;
  k.mu_lo = mu.lo;
  k.r_hi = r.hi;
  k.r_lo = r.lo;
  k.c = -__fmul_rn(mu.lo, r.hi);
  // Absolute error of the fast path is below ~2^-45 * r * |mu|; require |t| >= 2^-20 r |mu|
  // so that it stays under a quarter of an fp32 ulp of t.
  k.t_small = __fmul_rn(__fmul_rn(fabsf(mu.hi), r.hi), 0x1p-20f);
  return k;
}

// True when no bf16 value lies within 2^-18 |mu| of the mean, so |x - mu| is never small
// enough for the absolute error term to matter and the per-element |t| < t_small test can be
// skipped for the whole row (the usual case: one row in thousands fails this).
__device__ __forceinline__ bool mean_far_from_bf16_grid(float mu_hi) {
  const uint32_t u = __float_as_uint(mu_hi);
  const float lo = __uint_as_float(u & 0xFFFF0000u);            // bf16 value toward zero
  const float hi = __uint_as_float((u & 0xFFFF0000u) + 0x10000u);  // next bf16 away from zero
  const float d = fminf(fabsf(__fsub_rn(mu_hi, lo)), fabsf(__fsub_rn(hi, mu_hi)));
  return d > __fmul_rn(fabsf(mu_hi), 0x1p-18f);
}

// ------------------------------------------------------------------------------------------
// normalised value n = RN_bf16((x - mu) * rstd)
// ------------------------------------------------------------------------------------------

// Fast path: t = RN(RN(x - mu_hi) * r_hi + c), c = RN(-mu_lo * r_hi). Against the exact
// (x - mu) r its error is below 2.5 fp32 ulps of t: the rounding of x - mu_hi and the
// neglected r_lo each move it by at most 2^-24 |t| (under one ulp), the fused multiply-add
// rounds once (half an ulp); c's rounding and the row statistics' relative error (about
// 2^-34 on the workload rows, far below 2^-24 on any bf16 row) add a small fraction of an ulp,
// and the absolute error terms are bounded through t_small. The bf16 rounding of t is
// therefore certain unless the low 16 bits of t are within kGuard = 3 of the midpoint
// pattern 0x8000 (otherwise t is at least 4 ulps from the midpoint), or |t| < t_small. The
// QKV epilogue's fast value (within one ulp) uses the same test.
constexpr uint32_t kGuard = 3;
constexpr uint32_t kGuardAdd = ((kGuard - 0x8000u) & 0xFFFFu) << 16;
constexpr uint32_t kGuardMax = (2u * kGuard) << 16;

__device__ __forceinline__ float norm_fast(float x, const RowConst& k) {
  return __fmaf_rn(__fsub_rn(x, k.mu_hi), k.r_hi, k.c);
}

__device__ __forceinline__ bool near_bf16_midpoint(float t) {
  return ((__float_as_uint(t) << 16) + kGuardAdd) <= kGuardMax;
}

__device__ __forceinline__ bool norm_uncertain(float t, const RowConst& k) {
  return near_bf16_midpoint(t) | (fabsf(t) < k.t_small);
}

// Exact path: t = (x - mu) * r in double-float, then RN_bf16 of (t_hi + t_lo): t_hi decides
// unless it sits exactly on a bf16 midpoint, where the sign of t_lo breaks the tie (t_lo is
// below half an fp32 ulp, far below half a bf16 quantum). Returns the bf16 bits of n.
__device__ __forceinline__ uint32_t norm_exact_bits(float x, const RowConst& k) {
  float s, e;
  two_sum(x, -k.mu_hi, s, e);
  float d_hi, d_lo;
  two_sum(s, __fsub_rn(e, k.mu_lo), d_hi, d_lo);
  float p, pe;
  two_prod(d_hi, k.r_hi, p, pe);
  pe = __fadd_rn(pe, __fmaf_rn(d_hi, k.r_lo, __fmul_rn(d_lo, k.r_hi)));
  float t_hi, t_lo;
  fast_two_sum(p, pe, t_hi, t_lo);
  const uint32_t u = __float_as_uint(t_hi);
  if ((u & 0xFFFFu) == 0x8000u && t_lo != 0.0f) {
    const bool mag_up = (t_lo > 0.0f) == (t_hi > 0.0f);
    return (u >> 16) + (mag_up ? 1u : 0u);
  }
  return pack_bf16x2(t_hi, 0.0f) & 0xFFFFu;
}

// ------------------------------------------------------------------------------------------
// per-element epilogue: modulate, quantise
// ------------------------------------------------------------------------------------------

// y = RN_bf16(fma(n, one_plus_scale, shift)) for two elements (n given as fp32 values of
// bf16 numbers); returns the packed bf16 pair.
__device__ __forceinline__ uint32_t modulate2(float n0, float n1, float ops0, float ops1,
                                              float sh0, float sh1) {
  return pack_bf16x2(__fmaf_rn(n0, ops0, sh0), __fmaf_rn(n1, ops1, sh1));
}

// q for a packed bf16 pair y: E4M3(RN(y * inv)); returns 16 bits (two codes).
__device__ __forceinline__ uint32_t quant2(uint32_t ypair, float inv) {
  return pack_e4m3x2(__fmul_rn(bf_lo(ypair), inv), __fmul_rn(bf_hi(ypair), inv));
}

}  // namespace fp8q

namespace fp8q {

// ------------------------------------------------------------------------------------------
// packed fp32 pairs (sm_100+ f32x2 instructions: one issue slot for two lanes of work)
// ------------------------------------------------------------------------------------------

// ptxas may fuse a mul.rn.f32x2 whose result feeds an add.rn.f32x2 into one fused
// multiply-add (observed on sm_103a, unlike the scalar _rn intrinsics): where a product must
// be rounded on its own before a sum, use __fmul_rn / __fadd_rn instead.
struct f2 {
  unsigned long long v;
};

__device__ __forceinline__ f2 f2_make(float lo, float hi) {
  return f2{(static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo)};
}
__device__ __forceinline__ float f2_lo(f2 a) { return __uint_as_float(uint32_t(a.v)); }
__device__ __forceinline__ float f2_hi(f2 a) { return __uint_as_float(uint32_t(a.v >> 32)); }
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}

// bf16x2 word -> (lo, hi) fp32 pair.
__device__ __forceinline__ f2 bf2_to_f2(uint32_t u) { return f2_make(bf_lo(u), bf_hi(u)); }

// Dekker FastTwoSum on both lanes: s + e == a + b exactly when exponent(a) >= exponent(b).
__device__ __forceinline__ void fast_two_sum2(f2 a, f2 b, f2& s, f2& e) {
  s = add2(a, b);
  e = sub2(b, sub2(s, a));
}

// Lane-wise max of two packed u16 pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Lane-wise max(|a|, |b|) of two bf16 pairs (sign = xor of the signs, not used): the
// magnitude bits of the result are the larger magnitude of each lane, in one instruction.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Knuth TwoSum on both lanes: s + e == a + b exactly.
__device__ __forceinline__ void two_sum2(f2 a, f2 b, f2& s, f2& e) {
  s = add2(a, b);
  const f2 bv = sub2(s, a);
  const f2 av = sub2(s, bv);
  e = add2(sub2(a, av), sub2(b, bv));
}

// ------------------------------------------------------------------------------------------
// asynchronous global -> shared copies (cp.async, completion by wait_group: no spin loops)
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// 16-byte shared-memory load kept as one instruction (four fp32 lanes).
__device__ __forceinline__ float4 lds128(const float4* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace fp8q

namespace fp8q {

// ------------------------------------------------------------------------------------------
// device error word, mbarriers and bulk (TMA) copies
// ------------------------------------------------------------------------------------------

// Bits set by a kernel that gave up on a wait (a wait only runs out when a phase it depends
// on never completes, i.e. on a defect): the kernel records the bit, stops taking work and
// returns. The host reads and clears the word with fp8q_device_error().
constexpr unsigned kDevErrWaitTimeout = 1u;
__device__ unsigned int g_device_error = 0u;

__device__ __forceinline__ void report_device_error(unsigned bits) {
  atomicOr(&g_device_error, bits);
}

// Upper bound of every mbarrier wait, in SM clock cycles (about two seconds at 2 GHz).
constexpr long long kWaitLimitCycles = 1ll << 32;

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes initialised mbarriers visible to the other threads and to the bulk-copy unit.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One arrival that also adds `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// True once the phase with parity `parity` has completed (the thread may be suspended for a
// hardware-chosen time inside the instruction while it is pending).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for a phase: false when it has not completed within kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitLimitCycles) return false;
  return true;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to this
// CTA's shared memory, completing as transactions on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// One bulk copy shared -> global (TMA, bulk-group completion), its commit, and the waits for
// the committed groups: `.read` returns once at most N groups still read shared memory, the
// plain form once at most N groups are incomplete. Both addresses 16-byte aligned, size a
// multiple of 16.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(gmem_dst), "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// The next index of a shared counter for the whole warp (lane 0 increments, all lanes get it).
__device__ __forceinline__ int ws_claim(int* ctr) {
  int k = 0;
  if ((threadIdx.x & 31) == 0) k = atomicAdd(ctr, 1);
  return __shfl_sync(0xffffffffu, k, 0);
}

// The stage's row word: written with release semantics by the producer once the stage's
// previous use has been released, read with acquire semantics by the consumers.
__device__ __forceinline__ void ws_set_row(int* rowid, int k) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(rowid)), "r"(k)
               : "memory");
}
__device__ __forceinline__ int ws_get_row(const int* rowid) {
  int k;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(k) : "r"(smem_addr(rowid))
               : "memory");
  return k;
}

// Wait for phase u of `bar` for row k in stage s. From the second use of a stage on, first
// (bounded) until the producer has written k into the stage's row word.
__device__ __forceinline__ bool ws_wait_row(uint64_t* bar, const int* rowid, int s, int k,
                                            int u) {
  if (u > 0 && ws_get_row(rowid + s) != k) {
    const long long t0 = clock64();
    while (ws_get_row(rowid + s) != k) {
      if (clock64() - t0 > kWaitLimitCycles) return false;
      __nanosleep(100);
    }
  }
  return mbar_wait(bar, u & 1);
}


// Four E4M3 codes E4M3(RN(y * inv)) of two bf16 pairs, as one 32-bit word (y0 low pair in
// bytes 0-1, y1 in bytes 2-3): two packed multiplies, two conversions, one byte permute.
// Four E4M3 codes of the y values already rounded to bf16 and held as fp32 pairs (as quant4,
// without unpacking packed words).
__device__ __forceinline__ uint32_t quant4f(f2 y0, f2 y1, f2 inv2) {
  const f2 a = mul2(y0, inv2), b = mul2(y1, inv2);
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 a0, a1, b0, b1;\n\t"
      "mov.b64 {a0, a1}, %1;\n\tmov.b64 {b0, b1}, %2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, a1, a0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, b1, b0;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ uint32_t quant4(uint32_t y0, uint32_t y1, unsigned long long inv2) {
  unsigned long long a, b;
  asm("{\n\t.reg .b64 v;\n\tmov.b64 v, {%1, %2};\n\tmul.rn.f32x2 %0, v, %3;\n\t}"
      : "=l"(a) : "r"(y0 << 16), "r"(y0 & 0xFFFF0000u), "l"(inv2));
  asm("{\n\t.reg .b64 v;\n\tmov.b64 v, {%1, %2};\n\tmul.rn.f32x2 %0, v, %3;\n\t}"
      : "=l"(b) : "r"(y1 << 16), "r"(y1 & 0xFFFF0000u), "l"(inv2));
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 a0, a1, b0, b1;\n\t"
      "mov.b64 {a0, a1}, %1;\n\tmov.b64 {b0, b1}, %2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, a1, a0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, b1, b0;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "l"(a), "l"(b));
  return r;
}

// RN_bf16(t) as an fp32 value: the bf16 lands in the high half, the low half is zero.
__device__ __forceinline__ float round_bf16(float t) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(t), "f"(0.0f));
  return __uint_as_float(r);
}

}  // namespace fp8q
