// nss_kernels.cuh -- LayerNorm (no affine) -> AdaLN modulate -> dual BF16 + E4M3 output, and
// the gated scale-residual variant, for sm_103a.
//
// Computation per row (sources: "sglang #37156 - Qwen-Image FP8 norm + activation-quant
// fusion", key source snippets; "sglang #37116 - Qwen-Image output-bias deferral",
// implementation breakdown item 3):
//   [residual variant] xb = bias ? RN_bf16(x + bias) : x ; x := RN_bf16(xb*gate + residual)
//   mu, var (population) ; n = RN_bf16((x - mu)/sqrt(var + eps))
//   y = RN_bf16(fma(n, RN(1 + scale), shift)) ; q = E4M3(RN(y * RN(1/input_scale)))
//
// Tuned path (cols = 256 * V * WPR, i.e. 3072 and 6144): WPR warps own one row, each lane
// holds V 16-byte chunks of it in registers (chunk j of lane l covers columns
// [(j*32 + l)*8, +8) of the warp's part), so every global load and store of a warp is one
// contiguous 512-byte (bf16) or 256-byte (e4m3) segment. The row sums sum(x) and sum(x^2)
// are accumulated per lane with FastTwoSum on packed fp32 pairs started at power-of-two
// offsets (every rounding error exact, the errors summed apart in fp32), and the lanes'
// totals are added as integers (redux.sync), so every lane ends with bit-identical row
// constants. Each warp streams its rows through a two-stage cp.async ring
// in shared memory, so the next row is in flight while the current one is processed.
// RN(1 + scale) and shift are expanded once per CTA into shared memory as fp32 in lane-major
// order (each warp-wide 16-byte shared load is conflict-free). CTAs are persistent, own a
// contiguous block of rows, and with per-sample modulation are assigned to one modulation
// group each, so the table holds a single modulation row.
//
// Generic path (any cols % 8 == 0 up to 32768): one CTA per row, the row staged in shared
// memory, same per-element arithmetic.
#pragma once

#include "fp8q_device.cuh"

namespace fp8q {

struct NssParams {
  const uint16_t* x;         // [rows, cols]
  const uint16_t* residual;  // [rows, cols]       (residual variant)
  const uint16_t* bias;      // [cols] or nullptr   (residual variant)
  const uint16_t* gate;      // [n_mod, cols]       (residual variant)
  const uint16_t* scale;     // [n_mod, cols]
  const uint16_t* shift;     // [n_mod, cols]
  uint16_t* residual_out;    // [rows, cols]        (residual variant)
  uint16_t* y;               // [rows, cols]
  uint8_t* q;                // [rows, cols]
  const float* input_scale;  // one fp32
  int64_t rows;
  int64_t mod_rows;          // 0: one modulation row for all rows
  int cols;
  float eps;
};

constexpr int kNssThreads = 256;
constexpr int kNssWarps = kNssThreads / 32;

// Double-float butterfly over the 32 lanes of a warp (all lanes get identical results).
__device__ __forceinline__ void warp_reduce_dd(dd& a, dd& b) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    dd pa{__shfl_xor_sync(0xffffffffu, a.hi, off), __shfl_xor_sync(0xffffffffu, a.lo, off)};
    dd pb{__shfl_xor_sync(0xffffffffu, b.hi, off), __shfl_xor_sync(0xffffffffu, b.lo, off)};
    a = dd_add(a, pa);
    b = dd_add(b, pb);
  }
}

// Error-free accumulation of one element into (sum, sum of squares). v*v is exact in fp32
// because v has an 8-bit significand.
__device__ __forceinline__ void acc_stats(float v, dd& s, dd& q) {
  float t, e;
  two_sum(s.hi, v, t, e);
  s.hi = t;
  s.lo = __fadd_rn(s.lo, e);
  two_sum(q.hi, __fmul_rn(v, v), t, e);
  q.hi = t;
  q.lo = __fadd_rn(q.lo, e);
}

__device__ __forceinline__ void acc_stats8(const uint4& v, dd& s, dd& q) {
  acc_stats(bf_lo(v.x), s, q);
  acc_stats(bf_hi(v.x), s, q);
  acc_stats(bf_lo(v.y), s, q);
  acc_stats(bf_hi(v.y), s, q);
  acc_stats(bf_lo(v.z), s, q);
  acc_stats(bf_hi(v.z), s, q);
  acc_stats(bf_lo(v.w), s, q);
  acc_stats(bf_hi(v.w), s, q);
}

// residual_out pair = fma_bf16(RN_bf16(x + bias), gate, residual) (bias optional).
template <bool kHasBias>
__device__ __forceinline__ uint32_t resid2(uint32_t x, uint32_t b, uint32_t g, uint32_t r) {
  uint32_t xb = x;
  if (kHasBias) xb = pack_bf16x2(__fadd_rn(bf_lo(x), bf_lo(b)), __fadd_rn(bf_hi(x), bf_hi(b)));
  return fma_bf16x2(xb, g, r);
}

// n for the 8 elements of a chunk, as 4 packed bf16 pairs; exact path where uncertain.
__device__ __forceinline__ uint4 normalise8(const uint4& v, const RowConst& k) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4];
  float t[8];
  bool any = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t[2 * i] = norm_fast(bf_lo(in[i]), k);
    t[2 * i + 1] = norm_fast(bf_hi(in[i]), k);
    any |= norm_uncertain(t[2 * i], k) | norm_uncertain(t[2 * i + 1], k);
    out[i] = pack_bf16x2(t[2 * i], t[2 * i + 1]);
  }
  if (any) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo = out[i] & 0xFFFFu, hi = out[i] >> 16;
      if (norm_uncertain(t[2 * i], k)) lo = norm_exact_bits(bf_lo(in[i]), k);
      if (norm_uncertain(t[2 * i + 1], k)) hi = norm_exact_bits(bf_hi(in[i]), k);
      out[i] = lo | (hi << 16);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// y and q for a chunk of 8: n pairs, RN(1+scale) and shift as fp32 (8 each).
__device__ __forceinline__ void modulate_quant8(const uint4& n, const float* ops, const float* sh,
                                                float inv, uint4& y, uint2& q) {
  const uint32_t np[4] = {n.x, n.y, n.z, n.w};
  uint32_t yp[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    yp[i] = modulate2(bf_lo(np[i]), bf_hi(np[i]), ops[2 * i], ops[2 * i + 1], sh[2 * i],
                      sh[2 * i + 1]);
  y = make_uint4(yp[0], yp[1], yp[2], yp[3]);
  q.x = quant2(yp[0], inv) | (quant2(yp[1], inv) << 16);
  q.y = quant2(yp[2], inv) | (quant2(yp[3], inv) << 16);
}

// ------------------------------------------------------------------------------------------
// tuned path
// ------------------------------------------------------------------------------------------

constexpr int kTunedMaxThreads = 512;
// The plain LayerNorm with two warps per row at width 3072 (3 KB stages) fits 24 warps in
// shared memory and within 85 registers; the other instantiations stay at 16 warps (the
// residual kernels need more registers, the wider stages more shared memory).
template <int V, int WPR, bool RESID>
__host__ __device__ constexpr int tuned_threads() {
  return (!RESID && V == 6 && WPR == 2) ? 768 : kTunedMaxThreads;
}
constexpr int kMaxTableUnitsPerThread = 4;  // the host guarantees 4 * threads >= table units
constexpr int kStages = 2;

// Shared memory of the tuned kernel: [table | ring | exchange].
//   table    float4 index (((w*V + j)*P + k)*32 + l) for row part w, chunk j, piece k, lane l.
//            Pieces: 0,1 = RN(1+scale) of the chunk's 8 columns, 2,3 = shift; the residual
//            variant adds 4 = gate (8 bf16) and 5 = bias (8 bf16).
//   ring     per warp, kStages row buffers (x, and residual for the residual variant), filled
//            by cp.async one row ahead of the row being processed.
//   exchange (two warps per row) double-buffered partial sums, one float4 per warp.
template <int V, int WPR, bool RESID>
struct TunedLayout {
  static constexpr int kCols = 256 * V * WPR;
  static constexpr int kPartCols = kCols / WPR;
  static constexpr int kPieces = RESID ? 6 : 4;
  static constexpr int kTableF4 = WPR * V * kPieces * 32;
  static constexpr int kStageBytes = kPartCols * 2 * (RESID ? 2 : 1);
  // + one float4 of row-claim state: the CTA's next-row counter and, with two or more warps
  // per row, the row each warp group claimed last
  static constexpr size_t smem_bytes(int nw) {
    return size_t(kTableF4) * 16 + size_t(nw) * kStages * kStageBytes +
           (WPR > 1 ? size_t(2 * nw) * 16 : 0) + 16 + size_t(nw / WPR) * 4;
  }
};

// Rows of CTA b out of G. Without per-sample modulation the rows are split evenly. With
// n_mod modulation groups (n_mod <= G) the CTAs are first divided among the groups, so every
// CTA works inside one group and needs a single modulation row.
struct RowBlock {
  int64_t begin, end, mod;
};

__device__ __forceinline__ RowBlock cta_rows(int64_t rows, int64_t mod_rows, int64_t n_mod,
                                             int64_t b, int64_t G) {
  if (n_mod <= 1) return RowBlock{rows * b / G, rows * (b + 1) / G, 0};
  const int64_t g = b * n_mod / G;
  const int64_t c0 = (g * G + n_mod - 1) / n_mod;        // first CTA of group g
  const int64_t c1 = ((g + 1) * G + n_mod - 1) / n_mod;  // first CTA of group g + 1
  const int64_t k = c1 - c0, i = b - c0;
  const int64_t g0 = g * mod_rows;
  const int64_t rg = rows - g0 < mod_rows ? rows - g0 : mod_rows;
  return RowBlock{g0 + rg * i / k, g0 + rg * (i + 1) / k, g};
}

__device__ __forceinline__ dd dd_norm(float hi, float lo) {
  dd r;
  two_sum(hi, lo, r.hi, r.lo);
  return r;
}

// Offsets of the row-sum accumulators from the warp's largest bf16 exponent field mexp
// (max|x| < 2^(mexp - 126)): K = 2^(mexp - 118) >= 256 max|x|, K2 = 2^(2 mexp - 245) >=
// 128 max x^2, kept inside the normal fp32 range (K2 = 2^-126 covers every row whose squares
// are below 2^-133; rows with |x| >= 2^60 are outside the supported range).
struct RowOffsets {
  float K, K2;
  int ek, ek2;  // unbiased exponents of K and K2
};

__device__ __forceinline__ RowOffsets row_offsets(uint32_t mexp) {
  const int fk = min(int(mexp) + 9, 254);
  const int fk2 = min(max(2 * int(mexp) - 118, 1), 254);
  return RowOffsets{__uint_as_float(uint32_t(fk) << 23), __uint_as_float(uint32_t(fk2) << 23),
                    fk - 127, fk2 - 127};
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(uint32_t(e + 127) << 23); }

// x * 2^e in two exact power-of-two steps (no intermediate overflow for |e| <= 250).
__device__ __forceinline__ float scale2(float x, int e) {
  const int e1 = e / 2;
  return __fmul_rn(__fmul_rn(x, pow2f(e1)), pow2f(e - e1));
}

// Exact warp sum of offset accumulators. Each lane holds two FastTwoSum accumulators
// s = K + (partial sum), all within [K/2, 2K) (unsigned: [K, 2K)), and the sum of their exact
// rounding errors e. s - K is an integer number of units u = 2^(ek - 24) (ulp below K; the
// ulp above K is 2u), read off the bit patterns; the errors are rounded to units of 2^(ek-43)
// (well below the errors' own fp32 rounding). Both integer totals are reduced with
// redux.sync (exact, within int32 by the bounds on K) and combined into a double-float.
__device__ __forceinline__ dd warp_sum_offset(f2 s, f2 e, float K, int ek, bool signed_terms) {
  const int kb = int(__float_as_uint(K));
  auto units = [&](float v) -> int {
    const int d = int(__float_as_uint(v)) - kb;
    return signed_terms ? (d >= 0 ? 2 * d : d) : d;
  };
  // unsigned terms (squares): s in [K, 2K) and the unit is the ulp of K itself
  const int shift = signed_terms ? 24 : 23;
  const int u = units(f2_lo(s)) + units(f2_hi(s));
  const float el = __fadd_rn(f2_lo(e), f2_hi(e));
  const int ue = __float2int_rn(scale2(el, 43 - ek));
  const int U = int(__reduce_add_sync(0xffffffffu, uint32_t(u)));
  const int UE = int(__reduce_add_sync(0xffffffffu, uint32_t(ue)));
  // total = U * 2^(ek - shift) + UE * 2^(ek - 43) = T * 2^(ek - 43) with the integer
  // T = V * 2^k + W, k = 43 - shift, V = U + floor(UE / 2^k), W = UE mod 2^k (|U| < 2^29,
  // |UE| < 2^31 by the bounds on K). T is formed in 32-bit pieces that are exact in fp32
  // (64-bit integer <-> float conversions run on the slow fp64 pipe): a = (V with its low 8
  // bits cleared) * 2^k, and the two parts of m = (V mod 2^8) * 2^k + W < 2^28.
  const int k = 43 - shift;
  const int V = U + (UE >> k);
  const int m = ((V & 0xFF) << k) | (UE & ((1 << k) - 1));
  const float a = __fmul_rn(__int2float_rn(V & ~0xFF), pow2f(k));
  float sa, ea;
  two_sum(a, __int2float_rn(m & ~0xF), sa, ea);
  // hi + lo == T exactly while |a + (m & ~0xF)| < 2^28 (then ea == 0), else within 2^-47 |T|
  float hi, lo;
  fast_two_sum(sa, __fadd_rn(ea, __int2float_rn(m & 0xF)), hi, lo);
  dd r;
  two_sum(scale2(hi, ek - 43), scale2(lo, ek - 43), r.hi, r.lo);
  return r;
}

// Exact-path fix-up of one 8-element chunk (rare: called only when some element of the chunk
// is uncertain). Out of line so that the hot loop stays small.
__device__ __noinline__ uint4 fix_uncertain8(const uint4 x, const uint4 n, const RowConst kc) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
  uint32_t nw[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo = nw[i] & 0xFFFFu, hi = nw[i] >> 16;
    if (norm_uncertain(norm_fast(bf_lo(xw[i]), kc), kc)) lo = norm_exact_bits(bf_lo(xw[i]), kc);
    if (norm_uncertain(norm_fast(bf_hi(xw[i]), kc), kc)) hi = norm_exact_bits(bf_hi(xw[i]), kc);
    nw[i] = lo | (hi << 16);
  }
  return make_uint4(nw[0], nw[1], nw[2], nw[3]);
}

// n, y and q for the warp's part of one row: chunk j of this lane is stage[j*32], its
// modulation constants tab[(j*P + 0..3)*32]. kSmallTest adds the per-element |t| < t_small
// test (rows whose mean lies close to a bf16 value).
template <int V, int P, bool kSmallTest>
__device__ __forceinline__ void row_outputs(const uint4* stage, const float4* tab,
                                            const RowConst& kc, f2 mu2, f2 r2, f2 c2, f2 inv2,
                                            uint4* yr, uint2* qr) {
  // unrolled 6 deep (measured: 2 -> 6 gains 3-4 %; the full 12 overflows the i-cache)
#pragma unroll 6
  for (int j = 0; j < V; ++j) {
    const uint4 xv = stage[j * 32];
    const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
    uint32_t n[4];
    bool any = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 tt = fma2(sub2(bf2_to_f2(w4[i]), mu2), r2, c2);
      const float t0 = f2_lo(tt), t1 = f2_hi(tt);
      any |= near_bf16_midpoint(t0) | near_bf16_midpoint(t1);
      if (kSmallTest) any |= (fabsf(t0) < kc.t_small) | (fabsf(t1) < kc.t_small);
      n[i] = pack_bf16x2(t0, t1);
    }
    uint4 nv = make_uint4(n[0], n[1], n[2], n[3]);
    if (any) nv = fix_uncertain8(xv, nv, kc);
    const float4 o0 = lds128(tab + (j * P + 0) * 32), o1 = lds128(tab + (j * P + 1) * 32);
    const float4 h0 = lds128(tab + (j * P + 2) * 32), h1 = lds128(tab + (j * P + 3) * 32);
    const uint32_t nn[4] = {nv.x, nv.y, nv.z, nv.w};
    const f2 ops[4] = {f2_make(o0.x, o0.y), f2_make(o0.z, o0.w), f2_make(o1.x, o1.y),
                       f2_make(o1.z, o1.w)};
    const f2 shs[4] = {f2_make(h0.x, h0.y), f2_make(h0.z, h0.w), f2_make(h1.x, h1.y),
                       f2_make(h1.z, h1.w)};
    uint32_t yw[4], qw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 yf = fma2(bf2_to_f2(nn[i]), ops[i], shs[i]);
      yw[i] = pack_bf16x2(f2_lo(yf), f2_hi(yf));
      const f2 qf = mul2(bf2_to_f2(yw[i]), inv2);
      qw[i] = pack_e4m3x2(f2_lo(qf), f2_hi(qf));
    }
    st_stream(yr + j * 32, make_uint4(yw[0], yw[1], yw[2], yw[3]));
    st_stream(qr + j * 32, make_uint2(qw[0] | (qw[1] << 16), qw[2] | (qw[3] << 16)));
  }
}

template <int V, int WPR, bool RESID, bool HAS_BIAS>
__global__ void __launch_bounds__(tuned_threads<V, WPR, RESID>(), 1)
    nss_tuned_kernel(const NssParams p, const int64_t n_mod) {
  using L = TunedLayout<V, WPR, RESID>;
  constexpr int C = L::kCols;
  constexpr int PC = L::kPartCols;
  constexpr int P = L::kPieces;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float4* table = reinterpret_cast<float4*>(smem_raw);
  const int nw = blockDim.x >> 5;
  const int rows_per_iter = nw / WPR;
  unsigned char* ring = smem_raw + size_t(L::kTableF4) * 16;
  float4* red = reinterpret_cast<float4*>(ring + size_t(nw) * kStages * L::kStageBytes);
  int* claim = reinterpret_cast<int*>(red + (WPR > 1 ? 2 * nw : 0));  // [0]: counter
  int* claimed = claim + 4;                                            // per warp group

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_slot = warp / WPR, part = warp % WPR;
  const RowBlock blk = cta_rows(p.rows, p.mod_rows, n_mod, blockIdx.x, gridDim.x);
  if (blk.begin >= blk.end) return;  // uniform across the CTA
  wait_for_producers();
  allow_dependents();
  unsigned char* my_ring = ring + size_t(warp) * kStages * L::kStageBytes;

  // Row r's part for this warp -> ring stage (each lane copies exactly the chunks it reads).
  auto issue = [&](int64_t r, int stage) {
    const size_t off = size_t(r) * C + size_t(part) * PC;
    uint4* dst = reinterpret_cast<uint4*>(my_ring + stage * L::kStageBytes) + lane;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + off) + lane;
#pragma unroll
    for (int j = 0; j < V; ++j) cp_async16(dst + j * 32, src + j * 32);
    if constexpr (RESID) {
      const uint4* src2 = reinterpret_cast<const uint4*>(p.residual + off) + lane;
#pragma unroll
      for (int j = 0; j < V; ++j) cp_async16(dst + (PC / 8) + j * 32, src2 + j * 32);
    }
  };

  if (threadIdx.x == 0) claim[0] = rows_per_iter;  // rows [begin, begin + rows_per_iter) are static

  // Modulation table of this CTA's group, built and published (barrier) before any row copy
  // is issued: a warp's row copies can stall under memory back-pressure while the first wave
  // drains, and the barrier must not wait for that.
  const size_t mrow = size_t(blk.mod) * C;
  constexpr int kUnits = WPR * V * 32;  // one unit = one (part, chunk, lane): 8 columns
  constexpr int kRaw = RESID ? 4 : 2;
  uint4 traw[kMaxTableUnitsPerThread][kRaw];
#pragma unroll
  for (int h = 0; h < kMaxTableUnitsPerThread; ++h) {
    const int u = h * blockDim.x + threadIdx.x;
    if (u < kUnits) {
      const int l = u & 31, jw = u >> 5;  // jw = w*V + j
      const size_t col = size_t(jw / V) * PC + size_t((jw % V) * 32 + l) * 8;
      traw[h][0] = __ldg(reinterpret_cast<const uint4*>(p.scale + mrow + col));
      traw[h][1] = __ldg(reinterpret_cast<const uint4*>(p.shift + mrow + col));
      if constexpr (RESID) {
        traw[h][2] = __ldg(reinterpret_cast<const uint4*>(p.gate + mrow + col));
        traw[h][3] = HAS_BIAS ? __ldg(reinterpret_cast<const uint4*>(p.bias + col))
                              : make_uint4(0, 0, 0, 0);
      }
    }
  }

#pragma unroll
  for (int h = 0; h < kMaxTableUnitsPerThread; ++h) {
    const int u = h * blockDim.x + threadIdx.x;
    if (u < kUnits) {
      const int l = u & 31, jw = u >> 5;
      float4* t = table + size_t(jw) * P * 32 + l;
      const uint4 sc = traw[h][0], sh = traw[h][1];
      t[0 * 32] = make_float4(__fadd_rn(1.0f, bf_lo(sc.x)), __fadd_rn(1.0f, bf_hi(sc.x)),
                              __fadd_rn(1.0f, bf_lo(sc.y)), __fadd_rn(1.0f, bf_hi(sc.y)));
      t[1 * 32] = make_float4(__fadd_rn(1.0f, bf_lo(sc.z)), __fadd_rn(1.0f, bf_hi(sc.z)),
                              __fadd_rn(1.0f, bf_lo(sc.w)), __fadd_rn(1.0f, bf_hi(sc.w)));
      t[2 * 32] = make_float4(bf_lo(sh.x), bf_hi(sh.x), bf_lo(sh.y), bf_hi(sh.y));
      t[3 * 32] = make_float4(bf_lo(sh.z), bf_hi(sh.z), bf_lo(sh.w), bf_hi(sh.w));
      if constexpr (RESID) {
        const uint4 g = traw[h][2], b = traw[h][3];
        t[4 * 32] = make_float4(__uint_as_float(g.x), __uint_as_float(g.y), __uint_as_float(g.z),
                                __uint_as_float(g.w));
        t[5 * 32] = make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z),
                                __uint_as_float(b.w));
      }
    }
  }
  __syncthreads();

  int64_t r = blk.begin + row_slot;
  if (r < blk.end) issue(r, 0);
  cp_async_commit();

  const float inv = __frcp_rn(__ldg(p.input_scale));
  const f2 inv2 = f2_make(inv, inv);
  const float colsf = float(C);
  const float rcols = __frcp_rn(colsf);
  const float4* tab = table + size_t(part) * V * P * 32 + lane;
  int parity = 0;

#pragma unroll 1
  for (int k = 0; r < blk.end; ++k) {
    // Wait for row r, then claim the CTA's next unprocessed row and prefetch it into the other
    // stage. Claiming when the current row has landed balances the rows among the warps:
    // a warp whose first row arrived late takes fewer of the remaining rows. The first wave
    // of copies carries only first rows, which therefore arrive sooner.
    cp_async_wait<0>();  // this lane's copies of row r have landed
    int64_t rn;
    if constexpr (WPR == 1) {
      int c = 0;
      if (lane == 0) c = atomicAdd(claim, 1);
      rn = blk.begin + __shfl_sync(0xffffffffu, c, 0);
    } else {
      if (part == 0 && lane == 0) claimed[row_slot] = atomicAdd(claim, 1);
      asm volatile("bar.sync %0, %1;" ::"r"(1 + row_slot), "r"(32 * WPR) : "memory");
      rn = blk.begin + claimed[row_slot];
    }
    if (rn < blk.end) issue(rn, (k + 1) & 1);
    cp_async_commit();
    const size_t row_off = size_t(r) * C + size_t(part) * PC;
    uint4* stage = reinterpret_cast<uint4*>(my_ring + (k & 1) * L::kStageBytes) + lane;

    if constexpr (RESID) {
      // residual_out replaces x in the stage; each lane rewrites only its own chunks.
      uint4* ro = reinterpret_cast<uint4*>(p.residual_out + row_off) + lane;
#pragma unroll 6
      for (int j = 0; j < V; ++j) {
        const uint4 xv = stage[j * 32], rv = stage[(PC / 8) + j * 32];
        const float4 gf = lds128(tab + (j * P + 4) * 32);
        const float4 bf = lds128(tab + (j * P + 5) * 32);
        uint4 o;
        o.x = resid2<HAS_BIAS>(xv.x, __float_as_uint(bf.x), __float_as_uint(gf.x), rv.x);
        o.y = resid2<HAS_BIAS>(xv.y, __float_as_uint(bf.y), __float_as_uint(gf.y), rv.y);
        o.z = resid2<HAS_BIAS>(xv.z, __float_as_uint(bf.z), __float_as_uint(gf.z), rv.z);
        o.w = resid2<HAS_BIAS>(xv.w, __float_as_uint(bf.w), __float_as_uint(gf.w), rv.w);
        stage[j * 32] = o;
        st_stream(ro + j * 32, o);
      }
    }

    // Row sums sum(x) and sum(x^2), error-free per element. The accumulators start at powers
    // of two K (sum) and K2 (squares) above anything a lane's partial sums can reach
    // (K >= 256 max|x|, K2 >= 128 max x^2 over the warp's part of the row), so every addition
    // satisfies FastTwoSum's exponent condition and its rounding error is exact; the errors
    // are accumulated separately. v*v is exact (8-bit significands). max|x| comes from a
    // packed bf16 abs-max (max.xorsign.abs.bf16x2) over the row part, reduced over the warp.
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint4 xv = stage[j * 32];
      m2 = absmax_bf16x2(m2, absmax_bf16x2(absmax_bf16x2(xv.x, xv.y), absmax_bf16x2(xv.z, xv.w)));
    }
    const uint32_t mexp =
        __reduce_max_sync(0xffffffffu, (max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu) >> 7) & 0xFFu);
    const RowOffsets off = row_offsets(mexp);
    f2 sx = f2_make(off.K, off.K), sq = f2_make(off.K2, off.K2), ex = f2_make(0.0f, 0.0f),
       eq = ex;
    // 4 deep for one warp per row, 6 with two (measured best for each)
#pragma unroll(WPR == 1 ? 4 : 6)
    for (int j = 0; j < V; ++j) {
      const uint4 xv = stage[j * 32];
      const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f2 v = bf2_to_f2(w4[i]);
        f2 s, e;
        fast_two_sum2(sx, v, s, e);
        sx = s;
        ex = add2(ex, e);
        // s = RN(sq + v*v) with v*v exact; its rounding error is v*v + (sq - s), exact
        // under the same exponent condition, obtained with one more FMA
        s = fma2(v, v, sq);
        e = fma2(v, v, sub2(sq, s));
        sq = s;
        eq = add2(eq, e);
      }
    }
    dd s1 = warp_sum_offset(sx, ex, off.K, off.ek, true);
    dd s2 = warp_sum_offset(sq, eq, off.K2, off.ek2, false);
    if constexpr (WPR > 1) {
      float4* buf = red + parity * nw + row_slot * WPR;
      if (lane == 0) buf[part] = make_float4(s1.hi, s1.lo, s2.hi, s2.lo);
      asm volatile("bar.sync %0, %1;" ::"r"(1 + row_slot), "r"(32 * WPR) : "memory");
      const float4 a0 = buf[0];
      s1 = dd{a0.x, a0.y};
      s2 = dd{a0.z, a0.w};
#pragma unroll
      for (int w = 1; w < WPR; ++w) {
        const float4 aw = buf[w];
        s1 = dd_add(s1, dd{aw.x, aw.y});
        s2 = dd_add(s2, dd{aw.z, aw.w});
      }
      parity ^= 1;
    }
    const RowConst kc = row_constants(s1, s2, colsf, rcols, p.eps);
    const f2 mu2 = f2_make(kc.mu_hi, kc.mu_hi), r2 = f2_make(kc.r_hi, kc.r_hi),
             c2 = f2_make(kc.c, kc.c);

    uint4* yr = reinterpret_cast<uint4*>(p.y + row_off) + lane;
    uint2* qr = reinterpret_cast<uint2*>(p.q + row_off) + lane;
    if (mean_far_from_bf16_grid(kc.mu_hi))
      row_outputs<V, P, false>(stage, tab, kc, mu2, r2, c2, inv2, yr, qr);
    else
      row_outputs<V, P, true>(stage, tab, kc, mu2, r2, c2, inv2, yr, qr);
    r = rn;
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------------------------------------
// generic path: one CTA per row, row staged in shared memory
// ------------------------------------------------------------------------------------------

template <bool RESID, bool HAS_BIAS>
__global__ void __launch_bounds__(kNssThreads) nss_generic_kernel(const NssParams p) {
  extern __shared__ uint4 srow[];  // cols / 8 chunks
  __shared__ float4 red[kNssWarps];
  const int chunks = p.cols / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  wait_for_producers();
  const float inv = __frcp_rn(__ldg(p.input_scale));
  const float colsf = float(p.cols);
  const float rcols = __frcp_rn(colsf);

  for (int64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
    const int64_t m = p.mod_rows > 0 ? r / p.mod_rows : 0;
    const size_t row_off = size_t(r) * p.cols;
    const size_t mod_off = size_t(m) * p.cols;
    dd s1{0.0f, 0.0f}, s2{0.0f, 0.0f};
    for (int c = threadIdx.x; c < chunks; c += kNssThreads) {
      uint4 v = ld_stream(reinterpret_cast<const uint4*>(p.x + row_off) + c);
      if constexpr (RESID) {
        const uint4 rv = ld_stream(reinterpret_cast<const uint4*>(p.residual + row_off) + c);
        const uint4 g = *(reinterpret_cast<const uint4*>(p.gate + mod_off) + c);
        uint4 b = make_uint4(0, 0, 0, 0);
        if (HAS_BIAS) b = *(reinterpret_cast<const uint4*>(p.bias) + c);
        uint4 o;
        o.x = resid2<HAS_BIAS>(v.x, b.x, g.x, rv.x);
        o.y = resid2<HAS_BIAS>(v.y, b.y, g.y, rv.y);
        o.z = resid2<HAS_BIAS>(v.z, b.z, g.z, rv.z);
        o.w = resid2<HAS_BIAS>(v.w, b.w, g.w, rv.w);
        st_stream(reinterpret_cast<uint4*>(p.residual_out + row_off) + c, o);
        v = o;
      }
      srow[c] = v;
      acc_stats8(v, s1, s2);
    }
    warp_reduce_dd(s1, s2);
    if (lane == 0) red[warp] = make_float4(s1.hi, s1.lo, s2.hi, s2.lo);
    __syncthreads();
    {
      const float4 a0 = red[0];
      s1 = dd{a0.x, a0.y};
      s2 = dd{a0.z, a0.w};
#pragma unroll
      for (int w = 1; w < kNssWarps; ++w) {
        const float4 aw = red[w];
        s1 = dd_add(s1, dd{aw.x, aw.y});
        s2 = dd_add(s2, dd{aw.z, aw.w});
      }
    }
    const RowConst k = row_constants(s1, s2, colsf, rcols, p.eps);
    for (int c = threadIdx.x; c < chunks; c += kNssThreads) {
      const uint4 n = normalise8(srow[c], k);
      const uint4 sc = *(reinterpret_cast<const uint4*>(p.scale + mod_off) + c);
      const uint4 sh = *(reinterpret_cast<const uint4*>(p.shift + mod_off) + c);
      const float ops[8] = {__fadd_rn(1.0f, bf_lo(sc.x)), __fadd_rn(1.0f, bf_hi(sc.x)),
                            __fadd_rn(1.0f, bf_lo(sc.y)), __fadd_rn(1.0f, bf_hi(sc.y)),
                            __fadd_rn(1.0f, bf_lo(sc.z)), __fadd_rn(1.0f, bf_hi(sc.z)),
                            __fadd_rn(1.0f, bf_lo(sc.w)), __fadd_rn(1.0f, bf_hi(sc.w))};
      const float shf[8] = {bf_lo(sh.x), bf_hi(sh.x), bf_lo(sh.y), bf_hi(sh.y),
                            bf_lo(sh.z), bf_hi(sh.z), bf_lo(sh.w), bf_hi(sh.w)};
      uint4 y;
      uint2 q;
      modulate_quant8(n, ops, shf, inv, y, q);
      st_stream(reinterpret_cast<uint4*>(p.y + row_off) + c, y);
      st_stream(reinterpret_cast<uint2*>(p.q + row_off) + c, q);
    }
    __syncthreads();  // srow and red are reused by the next row
  }
}

}  // namespace fp8q
