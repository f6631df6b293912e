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
// Two kernels: qkv_ring_kernel (up to 64 heads; per-warp cp.async pipelines, four lanes per
// head, described below) and qkv_epilogue_kernel (any head count: one CTA per joint token,
// 6 warps, two per kind; 8 lanes per head with one 32-byte load each, so a lane's 8 packed BF16
// words are exactly its 8 RoPE pairs; a Q/K warp loads all its heads before computing any).
//
// Exactness of n: sum(x^2) per head is formed without rounding error that matters. Squares
// of BF16 values are exact in fp32. They are accumulated from an offset K2 = 2^(2E+9) >= 128
// max x^2 (E the exponent of the head's max |x|), so every partial sum lies in [K2, 2 K2)
// with one fixed ulp u: s = fma(v, v, S) and e = fma(v, v, S - s) give the exact rounding
// error; the e are added to a second offset accumulator 48u (one binade, ulp u 2^-18) with
// the FastTwoSum error kept, and those second-level errors summed in fp32 (their rounding is
// ~2^-53 of the total). Accumulator offsets come off as exact integers of their ulps, which
// the lanes of a head add as integers. 1/sqrt(mean + eps) is a double-float (~2^-45). The
// fast path (per-token kernel t = fma(p, r_hi, p r_lo), ring kernel t = RN(p r_hi); p = x w
// exact) is within 1.5 fp32 ulps of the exact value; only values whose low 16 bits lie within 3
// of the BF16 midpoint pattern take the exact path (TwoProduct + the tie broken by the low part).
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
// Ring kernel (heads <= 64): persistent CTAs stream whole tokens through a cp.async ring
// ------------------------------------------------------------------------------------------
//
// Four lanes per head, 32 values (16 packed words, 16 RoPE pairs) per lane, eight heads per
// warp: the per-head work (reductions, double-float constants) is shared by 32 values.
// Shared memory: the four RMSNorm weights (text q, k, image q, k; planar), then per warp
// `kQkvDepth` slots. q, k, the weights and cos/sin are stored in four planes: 16-byte chunk j
// of every 64-byte lane segment goes to plane j, so a warp's 16-byte loads of one plane are
// contiguous (no bank conflicts); v is stored as is.
constexpr int kQkvRingWarps = 8;
constexpr int kQkvRingMaxHeads = 64;

__device__ __forceinline__ void st_global16(void* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}

__device__ __forceinline__ void lds_words4(const uint8_t* p, uint32_t* w) {
  const float4 v = lds128(reinterpret_cast<const float4*>(p));
  w[0] = __float_as_uint(v.x);
  w[1] = __float_as_uint(v.y);
  w[2] = __float_as_uint(v.z);
  w[3] = __float_as_uint(v.w);
}

// 1 / sqrt(sum(x^2) / 128 + eps) for the head held by this lane's group of 4 lanes (32 values
// each), with the same exact accumulation as head_rrms; also returns p = x * weight (exact),
// the weight pairs read as fp32 from shared memory, so each value is unpacked once.
__device__ __forceinline__ dd head_rrms4(const uint32_t (&w)[16], const uint8_t* wv, float eps,
                                         f2 (&p)[16]) {
  uint32_t m = absmax_bf16x2(w[0], w[1]);
#pragma unroll
  for (int i = 2; i < 16; ++i) m = absmax_bf16x2(m, w[i]);
  uint32_t mx = max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
  const int E = min(max(int(mx >> 7) - 127, -40), 56);
  const float K2 = exp2i(2 * E + 9);
  const float K3 = 1.5f * exp2i(2 * E - 9);  // 48 u, u = 2^(2E - 14)
  f2 S = f2_make(K2, K2), R = f2_make(K3, K3), T = f2_make(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const f2 v = bf2_to_f2(w[i]);
    if ((i & 1) == 0) {
      const float4 w4 = lds128(reinterpret_cast<const float4*>(wv + (i >> 1) * 64));
      p[i] = mul2(v, f2_make(w4.x, w4.y));
      p[i + 1] = mul2(bf2_to_f2(w[i + 1]), f2_make(w4.z, w4.w));
    }
    const f2 sn = fma2(v, v, S);
    const f2 e = fma2(v, v, sub2(S, sn));  // exact error of sn
    S = sn;
    const f2 r = add2(R, e);
    T = add2(T, sub2(e, sub2(r, R)));     // FastTwoSum error (|R| > |e|)
    R = r;
  }
  const float inv_u = exp2i(14 - 2 * E);
  int cs = __float2int_rn(__fmul_rn(__fsub_rn(f2_lo(S), K2), inv_u)) +
           __float2int_rn(__fmul_rn(__fsub_rn(f2_hi(S), K2), inv_u));
  const float inv_u2 = exp2i(32 - 2 * E);
  int cr = __float2int_rn(__fmul_rn(__fsub_rn(f2_lo(R), K3), inv_u2)) +
           __float2int_rn(__fmul_rn(__fsub_rn(f2_hi(R), K3), inv_u2));
  float t = __fadd_rn(f2_lo(T), f2_hi(T));
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    cs += __shfl_xor_sync(0xFFFFFFFFu, cs, o);
    cr += __shfl_xor_sync(0xFFFFFFFFu, cr, o);
    t = __fadd_rn(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
  }
  dd sum = dd_add(int_to_dd(cs, exp2i(2 * E - 14)), int_to_dd(cr, exp2i(2 * E - 32)));
  sum = dd_add(sum, dd{t, 0.0f});
  const dd ms = dd{__fmul_rn(sum.hi, 1.0f / kHeadDim), __fmul_rn(sum.lo, 1.0f / kHeadDim)};
  return dd_rsqrt(dd_add(ms, dd{eps, 0.0f}));
}

// Normalised words n = RN_bf16(x w r) for one packed word; sets `unsure` when the fast value
// could round the other way (its low 16 bits lie within 3 of the BF16 midpoint pattern). The
// fast value RN(p r_hi) (p = x w exact) is within 1.5 fp32 ulps of the exact p (r_hi + r_lo):
// half an ulp from its rounding, under one from the neglected r_lo (|r_lo| <= 2^-24 r_hi).
__device__ __forceinline__ uint32_t norm_word(f2 p, f2 rh, f2 rl, bool& unsure) {
  (void)rl;
  const f2 t = mul2(p, rh);
  unsure |= near_bf16_midpoint(f2_lo(t)) | near_bf16_midpoint(f2_hi(t));
  return pack_bf16x2(f2_lo(t), f2_hi(t));
}

__device__ __noinline__ uint32_t norm_word_exact(float p0, float p1, float r_hi, float r_lo) {
  return scaled_exact_bits(p0, r_hi, r_lo) | (scaled_exact_bits(p1, r_hi, r_lo) << 16);
}

__device__ __forceinline__ uint32_t rope_word(uint32_t nw, float c, float s) {
  const float a = bf_lo(nw), b = bf_hi(nw);
  return pack_bf16x2(__fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)),
                     __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, s)));
}

// Each warp runs its own pipeline over a flat list of work items, `kQkvDepth - 1` items
// ahead, with no CTA-wide barrier after the start: item = (token, type), type one of the
// eight-head blocks of Q, of K or of V. A Q/K item brings 2 KB of values (planar) and the
// token's cos/sin row into the warp's slot; a V item brings 2 KB that go straight back out.
// Type of the item with remainder r < 3 * octs (r / octs, by comparison: no division).
__device__ __forceinline__ int item_type(int r, int octs) {
  return int(r >= octs) + int(r >= 2 * octs);
}

constexpr int kQkvDepth = 4;           // slots per warp
constexpr int kQkvWeightBytes = 2048;  // four fp32 RMSNorm weight vectors
constexpr int kQkvSlotBytes = 2560;    // 8 heads x 256 B + cos/sin 512 B

__global__ void __launch_bounds__(kQkvRingWarps * 32) qkv_ring_kernel(QkvParams P) {
  extern __shared__ __align__(16) uint8_t qkv_smem[];
  const int H = P.heads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, qtr = lane & 3;
  const int octs = (H + 7) >> 3;
  const int per_token = 3 * octs;
  const int64_t row_len = int64_t(H) * kHeadDim;
  uint8_t* wsm = qkv_smem;
  uint8_t* ring = qkv_smem + kQkvWeightBytes + warp * (kQkvDepth * kQkvSlotBytes);
  wait_for_producers();
  allow_dependents();

  // The four weight vectors as fp32, planar: 16-byte chunk c (values 4c .. 4c+3) of the
  // 32-value quarter q at c * 64 + q * 16 (a stream without tokens has none).
  for (int t = tid; t < 4 * 64; t += kQkvRingWarps * 32) {
    const int w = t >> 6, pi = t & 63;  // vector, value pair
    const uint16_t* src = w == 0 ? P.txt.wq : w == 1 ? P.txt.wk : w == 2 ? P.img.wq : P.img.wk;
    const bool present = (w < 2 ? P.txt.tokens : P.img.tokens) > 0;
    if (present) {
      const uint32_t pair = __ldg(reinterpret_cast<const uint32_t*>(src) + pi);
      const int q = pi >> 4, ii = pi & 15;
      *reinterpret_cast<float2*>(wsm + w * 512 + (ii >> 1) * 64 + q * 16 + (ii & 1) * 8) =
          make_float2(bf_lo(pair), bf_hi(pair));
    }
  }
  __syncthreads();

  // Items gw, gw + W, gw + 2W, ... as (token, remainder) pairs, advanced without division.
  struct Item {
    int64_t token;
    int r;     // 0 .. per_token - 1: type = r / octs, eight-head block = r % octs
  };
  const int64_t gw = int64_t(blockIdx.x) * kQkvRingWarps + warp;
  const int64_t W = int64_t(gridDim.x) * kQkvRingWarps;
  const int64_t w_tok = W / per_token;
  const int w_rem = int(W - w_tok * per_token);
  auto advance = [&](Item& it) {
    it.token += w_tok;
    it.r += w_rem;
    if (it.r >= per_token) {
      it.r -= per_token;
      ++it.token;
    }
  };
  const int64_t total_tokens = P.txt.tokens + P.img.tokens;
  auto issue = [&](const Item& it, int slot) {
    const bool is_txt = it.token < P.txt.tokens;
    auto sel = [is_txt](auto a, auto b) { return is_txt ? a : b; };
    const int64_t row = is_txt ? it.token : it.token - P.txt.tokens;
    const int type = item_type(it.r, octs), oc = it.r - type * octs;
    const uint16_t* base = type == 0 ? sel(P.txt.q, P.img.q)
                         : type == 1 ? sel(P.txt.k, P.img.k) : sel(P.txt.v, P.img.v);
    const uint16_t* src = base + row * sel(P.txt.ld, P.img.ld) + oc * 8 * kHeadDim;
    uint8_t* dst = ring + slot * kQkvSlotBytes;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = lane + 32 * k;          // 16-byte chunk of the 2 KB block
      const int hh = c >> 4, c16 = c & 15;  // head in the block, chunk in the head
      if (oc * 8 + hh < H) {
        const int off = type == 2 ? c * 16 : (c16 & 3) * 512 + (hh * 4 + (c16 >> 2)) * 16;
        cp_async16(dst + off, src + c * 8);
      }
    }
    if (type != 2) {  // cos (lanes 0..15) and sin (16..31), planar within each 256 bytes
      const float* cs = sel(P.txt.cos_sin, P.img.cos_sin) + row * kHeadDim;
      const int half = lane >> 4, k = lane & 15;
      cp_async16(dst + 2048 + half * 256 + (k & 3) * 64 + (k >> 2) * 16, cs + lane * 4);
    }
  };

  // the item being processed and the one being issued (kQkvDepth - 1 items ahead)
  Item cur{gw / per_token, int(gw % per_token)};
  Item ahead = cur;
#pragma unroll
  for (int k = 0; k < kQkvDepth - 1; ++k) {
    if (ahead.token < total_tokens) issue(ahead, k);
    cp_async_commit();
    advance(ahead);
  }
  for (int64_t k = 0; cur.token < total_tokens; ++k, advance(cur)) {
    if (ahead.token < total_tokens) issue(ahead, int((k + kQkvDepth - 1) % kQkvDepth));
    cp_async_commit();
    advance(ahead);
    cp_async_wait<kQkvDepth - 1>();
    __syncwarp();
    const uint8_t* sl = ring + int(k % kQkvDepth) * kQkvSlotBytes;
    const Item it = cur;
    const int type = item_type(it.r, octs), oc = it.r - type * octs;
    const bool is_txt = it.token < P.txt.tokens;
    if (type == 2) {
      uint16_t* dst = P.jv + it.token * row_len + oc * 8 * kHeadDim;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int c = lane + 32 * kk;
        if (oc * 8 + (c >> 4) < H)
          st_global16(dst + c * 8, lds128(reinterpret_cast<const float4*>(sl + c * 16)));
      }
    } else {
      const int h = oc * 8 + g8;
      uint32_t x[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (h < H) {
          lds_words4(sl + j * 512 + (g8 * 4 + qtr) * 16, x + 4 * j);
        } else {
          x[4 * j] = x[4 * j + 1] = x[4 * j + 2] = x[4 * j + 3] = 0u;
        }
      }
      const uint8_t* wv = wsm + ((is_txt ? 0 : 2) + type) * 512 + qtr * 16;
      f2 p[16];
      const dd r = head_rrms4(x, wv, is_txt ? P.txt.eps : P.img.eps, p);
      const f2 rh = f2_make(r.hi, r.hi), rl = f2_make(r.lo, r.lo);
      uint32_t n[16];
      bool unsure = false;
#pragma unroll
      for (int i = 0; i < 16; ++i) n[i] = norm_word(p[i], rh, rl, unsure);
      if (unsure) {  // rare: redo the words whose fast value may round the other way
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          bool u = false;
          norm_word(p[i], rh, rl, u);
          if (u) n[i] = norm_word_exact(f2_lo(p[i]), f2_hi(p[i]), r.hi, r.lo);
        }
      }
      const uint8_t* csv = sl + 2048 + qtr * 16;
      uint32_t o[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 c4 = lds128(reinterpret_cast<const float4*>(csv + j * 64));
        const float4 s4 = lds128(reinterpret_cast<const float4*>(csv + 256 + j * 64));
        o[4 * j + 0] = rope_word(n[4 * j + 0], c4.x, s4.x);
        o[4 * j + 1] = rope_word(n[4 * j + 1], c4.y, s4.y);
        o[4 * j + 2] = rope_word(n[4 * j + 2], c4.z, s4.z);
        o[4 * j + 3] = rope_word(n[4 * j + 3], c4.w, s4.w);
      }
      if (h < H) {
        uint16_t* dst = (type == 0 ? P.jq : P.jk) + it.token * row_len + h * kHeadDim + qtr * 32;
        st_stream32(dst, *reinterpret_cast<const uint32_t(*)[8]>(o));
        st_stream32(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(o + 8));
      }
    }
    __syncwarp();  // every lane is done with the slot before it is refilled
  }
  cp_async_wait<0>();
}

}  // namespace fp8q
