// qkv_kernels.cuh -- attention-input epilogue after the packed QKV GEMM, for sm_103a.
//
// "sglang #37123 - Qwen-Image FP8 QKV fusion" (implementation breakdown item 3, key source
// snippets) and "sglang #37162 - FLUX.2 FP8 LayerNorm/quant/QKV fusions" (implementation
// breakdown item 3): per token of two streams (text, image) and per head of 128 values,
//   Q, K:  n_j = RN_bf16(x_j * w_j / sqrt(mean(x^2) + eps))         (exact value, one rounding)
//          o[2i]   = RN_bf16(RN(RN(n[2i] c_i) - RN(n[2i+1] s_i)))  (interleaved RoPE, fp32
//          o[2i+1] = RN_bf16(RN(RN(n[2i+1] c_i) + RN(n[2i] s_i)))   products and sum)
//   V:     copied,
// written to joint [text tokens + image tokens, heads, 128] buffers, text first.
//
// Two kernels: qkv_ws_kernel (up to 64 heads; warp-specialised, whole tokens streamed through
// a shared-memory ring by bulk copies, four lanes per head, described below) and
// qkv_epilogue_kernel (any head count: one CTA per joint token, 6 warps, two per kind; 8 lanes
// per head with one 32-byte load each, so a lane's 8 packed BF16 words are exactly its 8 RoPE
// pairs; a Q/K warp loads all its heads before computing any).
//
// Exactness of n: sum(x^2) per head is formed without rounding error that matters. Squares
// of BF16 values are exact in fp32. They are accumulated from an offset K2 = 2^(2E+9) >= 128
// max x^2 (E the exponent of the head's max |x|), so every partial sum lies in [K2, 2 K2)
// with one fixed ulp u: s = fma(v, v, S) and e = fma(v, v, S - s) give the exact rounding
// error; the e are added to a second offset accumulator 48u (one binade, ulp u 2^-18) with
// the FastTwoSum error kept, and those second-level errors summed in fp32 (their rounding is
// ~2^-53 of the total). Accumulator offsets come off as exact integers of their ulps, which
// the lanes of a head add as integers. 1/sqrt(mean + eps) is a double-float (~2^-45). The
// fast path (per-token kernel t = fma(p, r_hi, p r_lo), warp-specialised kernel t = RN(p r_hi);
// p = x w exact) is within 1.5 fp32 ulps of the exact value; only values whose low 16 bits lie
// within 3 of the BF16 midpoint pattern take the exact path (TwoProduct + the tie broken by the
// low part).
#pragma once

#include "fp8q_device.cuh"

namespace fp8q {

constexpr int kQkvWarps = 6;       // per CTA: 2 x (Q, K, V)
constexpr int kQkvBatch = 3;       // heads-of-four loaded ahead per Q/K warp
constexpr int kQkvMinCtas = 4;     // resident CTAs per SM the register budget must allow
constexpr int kHeadDim = 128;

struct QkvStream {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const uint16_t* wq;       // [128] RMSNorm weight of Q
  const uint16_t* wk;       // [128] RMSNorm weight of K
  const float* cos_sin;     // [tokens, 128]: cos of pair i at i, sin at 64 + i
  int64_t ld;               // row stride of q, k, v in elements
  int64_t tokens;
  float eps;
};

struct QkvParams {
  uint16_t* jq;
  uint16_t* jk;
  uint16_t* jv;
  QkvStream txt, img;
  int heads;
};

__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(uint32_t(e + 127) << 23); }

__device__ __forceinline__ void ld_nc32(const void* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

// Integer-valued float c (|c| < 2^31) times the power of two `scale`, as a double-float.
__device__ __forceinline__ dd int_to_dd(int c, float scale) {
  const float hi = __int2float_rn(c);
  const float lo = __int2float_rn(c - __float2int_rz(hi));
  return dd{__fmul_rn(hi, scale), __fmul_rn(lo, scale)};
}

// 1 / sqrt(sum(x^2) / 128 + eps) for the head held by this lane's group of 8 lanes.
__device__ __forceinline__ dd head_rrms(const uint32_t (&w)[8], float eps) {
  uint32_t m = max_u16x2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu);
#pragma unroll
  for (int i = 2; i < 8; ++i) m = max_u16x2(m, w[i] & 0x7FFF7FFFu);
  uint32_t mx = max(m & 0xFFFFu, m >> 16);
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
  const int E = min(max(int(mx >> 7) - 127, -40), 56);
  const float K2 = exp2i(2 * E + 9);
  const float K3 = 1.5f * exp2i(2 * E - 9);  // 48 u, u = 2^(2E - 14)
  f2 S = f2_make(K2, K2), R = f2_make(K3, K3), T = f2_make(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const f2 v = bf2_to_f2(w[i]);
    const f2 s = fma2(v, v, S);
    const f2 e = fma2(v, v, sub2(S, s));   // exact error of s
    S = s;
    const f2 r = add2(R, e);
    T = add2(T, sub2(e, sub2(r, R)));      // FastTwoSum error (|R| > |e|)
    R = r;
  }
  const float inv_u = exp2i(14 - 2 * E);
  int cs = __float2int_rn(__fmul_rn(__fsub_rn(f2_lo(S), K2), inv_u)) +
           __float2int_rn(__fmul_rn(__fsub_rn(f2_hi(S), K2), inv_u));
  const float inv_u2 = exp2i(32 - 2 * E);   // 1 / (u 2^-18)
  int cr = __float2int_rn(__fmul_rn(__fsub_rn(f2_lo(R), K3), inv_u2)) +
           __float2int_rn(__fmul_rn(__fsub_rn(f2_hi(R), K3), inv_u2));
  float t = __fadd_rn(f2_lo(T), f2_hi(T));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    cs += __shfl_xor_sync(0xFFFFFFFFu, cs, o);
    cr += __shfl_xor_sync(0xFFFFFFFFu, cr, o);
    t = __fadd_rn(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
  }
  dd sum = dd_add(int_to_dd(cs, exp2i(2 * E - 14)), int_to_dd(cr, exp2i(2 * E - 32)));
  sum = dd_add(sum, dd{t, 0.0f});
  const dd ms = dd{__fmul_rn(sum.hi, 1.0f / kHeadDim), __fmul_rn(sum.lo, 1.0f / kHeadDim)};
  return dd_rsqrt(dd_add(ms, dd{eps, 0.0f}));
}

// Exact path: RN_bf16(p * (r_hi + r_lo)) for an exact fp32 product p = x w.
__device__ __noinline__ uint32_t scaled_exact_bits(float p, float r_hi, float r_lo) {
  float ph, pe;
  two_prod(p, r_hi, ph, pe);
  pe = __fmaf_rn(p, r_lo, pe);
  float t_hi, t_lo;
  fast_two_sum(ph, pe, t_hi, t_lo);
  const uint32_t u = __float_as_uint(t_hi);
  if ((u & 0xFFFFu) == 0x8000u && t_lo != 0.0f) {
    const bool mag_up = (t_lo > 0.0f) == (t_hi > 0.0f);
    return (u >> 16) + (mag_up ? 1u : 0u);
  }
  return pack_bf16x2(t_hi, 0.0f) & 0xFFFFu;
}

// RMSNorm + RoPE of this lane's 16 values (8 pairs); x, wt: packed BF16 words; cw, sw: the
// lane's 8 cos and 8 sin values (fp32 bits). Returns the 8 output words.
__device__ __forceinline__ void qk_lane(const uint32_t (&x)[8], const uint32_t (&wt)[8],
                                        const uint32_t (&cw)[8], const uint32_t (&sw)[8], dd r,
                                        uint32_t (&o)[8]) {
  const f2 rh = f2_make(r.hi, r.hi), rl = f2_make(r.lo, r.lo);
  uint32_t n[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const f2 p = mul2(bf2_to_f2(x[i]), bf2_to_f2(wt[i]));   // exact
    const f2 t = fma2(p, rh, mul2(p, rl));
    n[i] = pack_bf16x2(f2_lo(t), f2_hi(t));
    if (near_bf16_midpoint(f2_lo(t)))   // rare (~2^-11): out-of-line exact rounding
      n[i] = (n[i] & 0xFFFF0000u) | scaled_exact_bits(f2_lo(p), r.hi, r.lo);
    if (near_bf16_midpoint(f2_hi(t)))
      n[i] = (n[i] & 0xFFFFu) | (scaled_exact_bits(f2_hi(p), r.hi, r.lo) << 16);
  }
  // Scalar _rn intrinsics: the products must be rounded before the sum (a packed
  // mul.rn.f32x2 feeding add.rn.f32x2 was fused into one rounding on sm_103a).
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = bf_lo(n[i]), b = bf_hi(n[i]);        // (n[2i], n[2i+1])
    const float c = __uint_as_float(cw[i]), s = __uint_as_float(sw[i]);
    const float o0 = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
    const float o1 = __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, s));
    o[i] = pack_bf16x2(o0, o1);
  }
}

__global__ void __launch_bounds__(kQkvWarps * 32, kQkvMinCtas) qkv_epilogue_kernel(QkvParams P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kind = warp >> 1;       // 0: Q, 1: K, 2: V
  const int first_quad = warp & 1;  // the two warps of a kind take alternate heads-of-four
  const int g = lane >> 3;          // head within a heads-of-four
  const int u = lane & 7;           // 16-value slice of the head
  const int heads = P.heads;
  const int quads = (heads + 3) >> 2;
  const int64_t row_len = int64_t(heads) * kHeadDim;
  const int64_t total = P.txt.tokens + P.img.tokens;
  wait_for_producers();

  for (int64_t jt = blockIdx.x; jt < total; jt += gridDim.x) {
    const bool is_txt = jt < P.txt.tokens;
    // field-wise selects keep the parameters in registers (a reference to either stream
    // would force a local copy of both)
    auto sel = [is_txt](auto a, auto b) { return is_txt ? a : b; };
    const int64_t row = is_txt ? jt : jt - P.txt.tokens;
    const int64_t ld = sel(P.txt.ld, P.img.ld);
    const uint16_t* base = kind == 0 ? sel(P.txt.q, P.img.q)
                         : kind == 1 ? sel(P.txt.k, P.img.k) : sel(P.txt.v, P.img.v);
    const uint16_t* src = base + row * ld + u * 16;
    uint16_t* dst = (kind == 0 ? P.jq : kind == 1 ? P.jk : P.jv) + jt * row_len + u * 16;
    if (kind == 2) {
      for (int qd0 = first_quad; qd0 < quads; qd0 += 2 * kQkvBatch) {
        uint32_t w[kQkvBatch][8];
#pragma unroll
        for (int b = 0; b < kQkvBatch; ++b) {
          const int h = (qd0 + 2 * b) * 4 + g;
          if (qd0 + 2 * b < quads && h < heads) ld_stream32(src + h * kHeadDim, w[b]);
        }
#pragma unroll
        for (int b = 0; b < kQkvBatch; ++b) {
          const int h = (qd0 + 2 * b) * 4 + g;
          if (qd0 + 2 * b < quads && h < heads) st_stream32(dst + h * kHeadDim, w[b]);
        }
      }
      continue;
    }
    const float eps = sel(P.txt.eps, P.img.eps);
    const uint16_t* wsrc = (kind == 0 ? sel(P.txt.wq, P.img.wq) : sel(P.txt.wk, P.img.wk)) + u * 16;
    const float* cs = sel(P.txt.cos_sin, P.img.cos_sin) + row * kHeadDim + u * 8;
    for (int qd0 = first_quad; qd0 < quads; qd0 += 2 * kQkvBatch) {
      uint32_t x[kQkvBatch][8];
#pragma unroll
      for (int b = 0; b < kQkvBatch; ++b) {
        const int h = (qd0 + 2 * b) * 4 + g;
        if (qd0 + 2 * b < quads && h < heads) {
          ld_stream32(src + h * kHeadDim, x[b]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[b][i] = 0u;
        }
      }
#pragma unroll
      for (int b = 0; b < kQkvBatch; ++b) {
        if (qd0 + 2 * b >= quads) break;  // warp-uniform
        const dd r = head_rrms(x[b], eps);
        // weight and cos/sin are re-read per head (L1 hits) rather than held in registers
        uint32_t wt[8], cw[8], sw[8];
        ld_nc32(wsrc, wt);
        ld_nc32(cs, cw);
        ld_nc32(cs + 64, sw);
        uint32_t o[8];
        qk_lane(x[b], wt, cw, sw, r, o);
        const int h = (qd0 + 2 * b) * 4 + g;
        if (h < heads) st_stream32(dst + h * kHeadDim, o);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// helpers of the warp-specialised kernel
// ------------------------------------------------------------------------------------------

constexpr int kQkvMaxWsHeads = 64;     // the warp-specialised kernel's head limit
// The four fp32 RMSNorm weight vectors (text q, k, image q, k), each 140 floats: the 8 weights
// of chunk c at 8c + 4 (c / 4), so that the lanes reading chunks c and c + 4 (the two head
// parities of a step) hit different banks.
constexpr int kQkvWeightStride = 140;
constexpr int kQkvWeightBytes = 4 * kQkvWeightStride * 4;

__device__ __forceinline__ void lds_words4(const uint8_t* p, uint32_t* w) {
  const float4 v = lds128(reinterpret_cast<const float4*>(p));
  w[0] = __float_as_uint(v.x);
  w[1] = __float_as_uint(v.y);
  w[2] = __float_as_uint(v.z);
  w[3] = __float_as_uint(v.w);
}

// ------------------------------------------------------------------------------------------
// Warp-specialised kernel (heads <= 64): one CTA per SM streams whole tokens through a ring
// ------------------------------------------------------------------------------------------
//
// A CTA owns a contiguous block of joint tokens (text first) and moves every token through a
// ring of S stages in shared memory. A stage holds the token's q, k and v rows (heads x 256 B
// each) and its cos/sin row (512 B), brought by four bulk copies (cp.async.bulk, TMA) that
// complete on the stage's `full` mbarrier.
//   producer warp  one lane issues the copies and refills a stage once its `empty` mbarrier
//                  completes;
//   V warp         one lane writes each token's v row back out with one bulk store from
//                  shared memory (no register traffic) and releases the stage once the store
//                  has read it;
//   Q/K warps      claim units (token, Q or K, block of eight heads) in order from a shared
//                  counter, normalise and rotate their heads, store the results directly and
//                  arrive on `empty`.
// Four lanes per head, 32 values per lane: lane q of a head holds the 16-byte chunks
// c = q + 4 (j ^ o), j = 0..3, o the parity of the head within the block, so that one
// 16-byte load of chunk index j by the warp reads 64 contiguous bytes per head and the eight
// heads split evenly over the two halves of the banks (no conflicts; the weight table is padded
// for the same reason, see kQkvWeightStride). Values 8c .. 8c + 7 of
// chunk c are RoPE pairs 4c .. 4c + 3.
// mbarrier phases: stage s = k % S holds tokens s, s + S, ...; token k waits for the phase of
// parity (k / S) & 1. The producer writes k into the stage's row word (release) before it
// issues the copies, and a Q/K warp that claims a later use of the stage first waits for that
// word, so it cannot take an older phase of the same parity for its own. The V warp and the
// producer take the stage's uses in order. Every wait is bounded; a wait that runs out records
// the device error and the warp stops.
// Q/K warps per CTA (NW), then the V warp and the producer warp. Measured on GB300 (graph
// replay of back-to-back launches, Qwen-Image 24 heads / FLUX.2 48 heads, microseconds):
// 13 warps 31.8 / 57.9, 14: 31.3 / 59.1, 15: 30.9 / 59.7, 16: 30.7 / 60.2; so 16 up to 32
// heads (18 warps: registers capped at 96, so that five warps fit a sub-partition's register
// file) and 13 above.
constexpr int kQwsMaxStages = 32;
__host__ __device__ constexpr int qws_qk_warps(int heads) { return heads <= 32 ? 16 : 13; }
__host__ __device__ constexpr int qws_threads(int nw) { return (nw + 2) * 32; }

// Dynamic shared memory of the warp-specialised kernel: weights, S stages, then per stage two
// mbarriers and the row word, and the unit counter.
__host__ __device__ constexpr size_t qws_stage_bytes(int heads) {
  return size_t(3) * heads * 256 + 512;
}
__host__ __device__ constexpr size_t qws_smem_bytes(int heads, int stages) {
  return kQkvWeightBytes + size_t(stages) * (qws_stage_bytes(heads) + 20) + 16;
}

// RMSNorm + interleaved RoPE of the 16 words this lane holds, written to `dst` (the head's
// output row). xs: the head's 256 bytes in the stage; wt: the padded fp32 weights; cs: the
// stage's cos (64 fp32) and sin (64 fp32) row; cidx: the lane's four chunk indices.
__device__ __forceinline__ void qws_head(const uint8_t* xs, const float* wt, const float* cs,
                                         float eps, const int (&cidx)[4], bool live,
                                         uint16_t* dst) {
  uint32_t x[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (live) {
      lds_words4(xs + cidx[j] * 16, x + 4 * j);
    } else {
      x[4 * j] = x[4 * j + 1] = x[4 * j + 2] = x[4 * j + 3] = 0u;
    }
  }
  // sum of squares (exact accumulation, as head_rrms) and p = x w (exact)
  uint32_t m = absmax_bf16x2(x[0], x[1]);
#pragma unroll
  for (int i = 2; i < 16; ++i) m = absmax_bf16x2(m, x[i]);
  uint32_t mx = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
  const int E = min(max(int(mx >> 7) - 127, -40), 56);
  const float K2 = exp2i(2 * E + 9);
  const float K3 = 1.5f * exp2i(2 * E - 9);  // 48 u, u = 2^(2E - 14)
  f2 S = f2_make(K2, K2), R = f2_make(K3, K3), T = f2_make(0.0f, 0.0f);
  f2 p[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float* wc = wt + 8 * cidx[j] + 4 * (cidx[j] >> 2);
    const float4 w0 = lds128(reinterpret_cast<const float4*>(wc));
    const float4 w1 = lds128(reinterpret_cast<const float4*>(wc + 4));
    const f2 wp[4] = {f2_make(w0.x, w0.y), f2_make(w0.z, w0.w), f2_make(w1.x, w1.y),
                      f2_make(w1.z, w1.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 v = bf2_to_f2(x[4 * j + i]);
      p[4 * j + i] = mul2(v, wp[i]);
      const f2 sn = fma2(v, v, S);
      const f2 e = fma2(v, v, sub2(S, sn));  // exact error of sn
      S = sn;
      const f2 r = add2(R, e);
      T = add2(T, sub2(e, sub2(r, R)));     // FastTwoSum error (|R| > |e|)
      R = r;
    }
  }
  const float inv_u = exp2i(14 - 2 * E);
  int cs_i = __float2int_rn(__fmul_rn(__fsub_rn(f2_lo(S), K2), inv_u)) +
             __float2int_rn(__fmul_rn(__fsub_rn(f2_hi(S), K2), inv_u));
  const float inv_u2 = exp2i(32 - 2 * E);
  int cr = __float2int_rn(__fmul_rn(__fsub_rn(f2_lo(R), K3), inv_u2)) +
           __float2int_rn(__fmul_rn(__fsub_rn(f2_hi(R), K3), inv_u2));
  float t = __fadd_rn(f2_lo(T), f2_hi(T));
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    cs_i += __shfl_xor_sync(0xFFFFFFFFu, cs_i, o);
    cr += __shfl_xor_sync(0xFFFFFFFFu, cr, o);
    t = __fadd_rn(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
  }
  dd sum = dd_add(int_to_dd(cs_i, exp2i(2 * E - 14)), int_to_dd(cr, exp2i(2 * E - 32)));
  sum = dd_add(sum, dd{t, 0.0f});
  const dd ms = dd{__fmul_rn(sum.hi, 1.0f / kHeadDim), __fmul_rn(sum.lo, 1.0f / kHeadDim)};
  const dd rr = dd_rsqrt(dd_add(ms, dd{eps, 0.0f}));
  const f2 rh = f2_make(rr.hi, rr.hi);
  // per chunk: n = RN_bf16(p r) (fast value within 1.5 ulps; the exact path where it may
  // round the other way), then RoPE on the pairs and one 16-byte store
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float n[8];
    bool unsure = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 tt = mul2(p[4 * j + i], rh);
      unsure |= near_bf16_midpoint(f2_lo(tt)) | near_bf16_midpoint(f2_hi(tt));
      n[2 * i] = round_bf16(f2_lo(tt));
      n[2 * i + 1] = round_bf16(f2_hi(tt));
    }
    if (unsure) {  // rare: redo the values whose fast value may round the other way
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float pv = (i & 1) ? f2_hi(p[4 * j + i / 2]) : f2_lo(p[4 * j + i / 2]);
        if (near_bf16_midpoint(__fmul_rn(pv, rr.hi)))
          n[i] = __uint_as_float(scaled_exact_bits(pv, rr.hi, rr.lo) << 16);
      }
    }
    const float4 c4 = lds128(reinterpret_cast<const float4*>(cs + 4 * cidx[j]));
    const float4 s4 = lds128(reinterpret_cast<const float4*>(cs + 64 + 4 * cidx[j]));
    const float cv[4] = {c4.x, c4.y, c4.z, c4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // products on both lanes at once, sums as separate roundings (no fused operation)
      const f2 ab = f2_make(n[2 * i], n[2 * i + 1]);
      const f2 pc = mul2(ab, f2_make(cv[i], cv[i])), ps = mul2(ab, f2_make(sv[i], sv[i]));
      o[i] = pack_bf16x2(__fsub_rn(f2_lo(pc), f2_hi(ps)), __fadd_rn(f2_hi(pc), f2_lo(ps)));
    }
    if (live) __stcs(reinterpret_cast<uint4*>(dst + cidx[j] * 8), make_uint4(o[0], o[1], o[2], o[3]));
  }
}

template <int NW>
__global__ void __maxnreg__(NW + 2 > 16 ? 96 : 128) qkv_ws_kernel(QkvParams P, int S) {
  constexpr int kVWarp = NW, kProducerWarp = NW + 1, kThreads = qws_threads(NW);
  extern __shared__ __align__(128) uint8_t qws_smem[];
  const int H = P.heads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int RB = H * 256;                          // bytes of one q, k or v row
  const int stage_bytes = int(qws_stage_bytes(H));
  float* wsm = reinterpret_cast<float*>(qws_smem);  // [4][kQkvWeightStride]: text q, k, image q, k
  uint8_t* ring = qws_smem + kQkvWeightBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + size_t(S) * stage_bytes);
  uint64_t* empty = full + S;
  int* rowid = reinterpret_cast<int*>(empty + S);
  int* next_unit = rowid + S;
  const int64_t total = P.txt.tokens + P.img.tokens;
  const int64_t t0 = total * blockIdx.x / gridDim.x;
  const int n = int(total * (blockIdx.x + 1) / gridDim.x - t0);
  if (n <= 0) return;  // uniform across the CTA
  const int nq = (H + 7) >> 3;  // blocks of eight heads per Q or K row
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 2 * nq + 1);
      rowid[s] = -1;
    }
    *next_unit = 0;
    fence_mbar_init();
  }
  wait_for_producers();
  allow_dependents();
  for (int t = threadIdx.x; t < 4 * 128; t += kThreads) {
    const int w = t >> 7, i = t & 127;
    const uint16_t* src = w == 0 ? P.txt.wq : w == 1 ? P.txt.wk : w == 2 ? P.img.wq : P.img.wk;
    const bool present = (w < 2 ? P.txt.tokens : P.img.tokens) > 0;
    wsm[w * kQkvWeightStride + i + 4 * (i >> 5)] =
        present ? __uint_as_float(uint32_t(__ldg(src + i)) << 16) : 0.0f;
  }
  __syncthreads();
  const int64_t row_len = int64_t(H) * kHeadDim;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int issued = 0;
      for (int k = 0, s = 0, u = 0; k < n; ++k) {
        if (u > 0 && !mbar_wait(empty + s, (u - 1) & 1)) {
          report_device_error(kDevErrWaitTimeout);
          break;
        }
        const int64_t tok = t0 + k;
        const bool txt = tok < P.txt.tokens;
        const QkvStream& st = txt ? P.txt : P.img;
        const int64_t row = txt ? tok : tok - P.txt.tokens;
        uint8_t* stg = ring + size_t(s) * stage_bytes;
        ws_set_row(rowid + s, k);
        mbar_arrive_expect_tx(full + s, uint32_t(3 * RB + 512));
        bulk_load(stg, st.q + row * st.ld, RB, full + s);
        bulk_load(stg + RB, st.k + row * st.ld, RB, full + s);
        bulk_load(stg + 2 * RB, st.v + row * st.ld, RB, full + s);
        bulk_load(stg + 3 * RB, st.cos_sin + row * kHeadDim, 512, full + s);
        issued = k + 1;
        if (++s == S) {
          s = 0;
          ++u;
        }
      }
      // the last copy into each stage has landed before this warp returns (always true on
      // the normal path, where every token is consumed; it matters only after a wait ran out)
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / S) * S;
        if (!mbar_wait(full + s, (last / S) & 1)) report_device_error(kDevErrWaitTimeout);
      }
    }
    return;
  }

  if (warp == kVWarp) {
    if (lane == 0) {
      int pend = -1;  // stage whose v store was issued last and is not yet released
      for (int k = 0, s = 0, u = 0; k < n; ++k) {
        if (!mbar_wait(full + s, u & 1)) {
          report_device_error(kDevErrWaitTimeout);
          break;
        }
        bulk_store(P.jv + (t0 + k) * row_len, ring + size_t(s) * stage_bytes + 2 * RB, RB);
        bulk_commit();
        if (pend >= 0) {
          bulk_wait_read<1>();  // the previous token's v row has been read
          mbar_arrive(empty + pend);
        }
        pend = s;
        if (++s == S) {
          s = 0;
          ++u;
        }
      }
      bulk_wait<0>();  // every store complete before the CTA can release shared memory
      if (pend >= 0) mbar_arrive(empty + pend);
    }
    return;
  }

  // Q/K warps
  const int g8 = lane >> 2, qtr = lane & 3, odd = g8 & 1;
  const int cidx[4] = {qtr + 4 * odd, qtr + 4 * (1 ^ odd), qtr + 4 * (2 ^ odd),
                       qtr + 4 * (3 ^ odd)};
  const int upt = 2 * nq;
  const int units = n * upt;
  for (int v = ws_claim(next_unit); v < units; v = ws_claim(next_unit)) {
    const int k = v / upt, rem = v - k * upt;
    const int kind = rem >= nq ? 1 : 0, oc = rem - kind * nq;
    const int s = k % S, u = k / S;
    if (!ws_wait_row(full + s, rowid, s, k, u)) {
      report_device_error(kDevErrWaitTimeout);
      break;
    }
    const int64_t tok = t0 + k;
    const bool txt = tok < P.txt.tokens;
    const int h = oc * 8 + g8;
    const uint8_t* stg = ring + size_t(s) * stage_bytes;
    uint16_t* dst = (kind == 0 ? P.jq : P.jk) + tok * row_len + int64_t(h) * kHeadDim;
    qws_head(stg + kind * RB + h * 256, wsm + ((txt ? 0 : 2) + kind) * kQkvWeightStride,
             reinterpret_cast<const float*>(stg + 3 * RB), txt ? P.txt.eps : P.img.eps, cidx,
             h < H, dst);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
}
}  // namespace fp8q
