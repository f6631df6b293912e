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
// are accumulated error-free (TwoSum) per lane and reduced across the warp by an xor
// butterfly of double-float additions (commutative, so every lane ends with bit-identical
// row constants). RN(1 + scale) and shift are pre-expanded once per CTA into shared memory
// as fp32 in lane-major order, so each warp-wide 16-byte shared load is conflict-free. CTAs
// are persistent and own a contiguous block of rows; a block touches at most two modulation
// rows, which is why the table has at most two slots.
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

// Shared-memory table layout (float4 units), per modulation slot s, row part w, chunk j,
// piece k, lane l: index (((s*WPR + w)*V + j)*P + k)*32 + l. Pieces: 0,1 = RN(1+scale) for
// the chunk's 8 columns, 2,3 = shift; residual variant adds 4 = gate (8 bf16), 5 = bias.
template <int V, int WPR, bool RESID>
struct TunedLayout {
  static constexpr int kCols = 256 * V * WPR;
  static constexpr int kPieces = RESID ? 6 : 4;
  static constexpr int kSlotF4 = WPR * V * kPieces * 32;       // float4 per slot
  static constexpr int kRowsPerIter = kNssWarps / WPR;
  static constexpr int kRedF4 = 2 * kRowsPerIter * WPR;         // WPR>1 exchange buffers
  static constexpr size_t smem_bytes(int slots) {
    return (size_t(slots) * kSlotF4 + (WPR > 1 ? kRedF4 : 0)) * sizeof(float4);
  }
};

template <int V, int WPR, bool RESID, bool HAS_BIAS>
__global__ void __launch_bounds__(kNssThreads, 1) nss_tuned_kernel(const NssParams p) {
  using L = TunedLayout<V, WPR, RESID>;
  constexpr int C = L::kCols;
  constexpr int P = L::kPieces;
  extern __shared__ float4 smem[];
  float4* table = smem;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_slot = warp / WPR, part = warp % WPR;
  const int64_t rb = (p.rows * blockIdx.x) / gridDim.x;
  const int64_t re = (p.rows * (blockIdx.x + 1)) / gridDim.x;
  if (rb >= re) return;  // uniform across the CTA
  const int64_t m_lo = p.mod_rows > 0 ? rb / p.mod_rows : 0;
  const int64_t m_hi = p.mod_rows > 0 ? (re - 1) / p.mod_rows : 0;
  const int slots = int(m_hi - m_lo + 1);  // host guarantees <= 2

  // Build the modulation table: one float4 per (slot, part, chunk, piece, lane).
  for (int idx = threadIdx.x; idx < slots * L::kSlotF4; idx += kNssThreads) {
    const int l = idx & 31;
    int rest = idx >> 5;
    const int k = rest % P;
    rest /= P;
    const int j = rest % V;
    rest /= V;
    const int w = rest % WPR;
    const int s = rest / WPR;
    const int col = w * (C / WPR) + (j * 32 + l) * 8;
    const int64_t mrow = (m_lo + s) * C;
    float4 out;
    if (k < 4) {
      const uint16_t* src = (k < 2 ? p.scale : p.shift) + mrow + col + (k & 1) * 4;
      const uint2 raw = *reinterpret_cast<const uint2*>(src);
      float a = bf_lo(raw.x), b = bf_hi(raw.x), c = bf_lo(raw.y), d = bf_hi(raw.y);
      if (k < 2) {
        a = __fadd_rn(1.0f, a);
        b = __fadd_rn(1.0f, b);
        c = __fadd_rn(1.0f, c);
        d = __fadd_rn(1.0f, d);
      }
      out = make_float4(a, b, c, d);
    } else {
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (k == 4) raw = *reinterpret_cast<const uint4*>(p.gate + mrow + col);
      else if (HAS_BIAS) raw = *reinterpret_cast<const uint4*>(p.bias + col);
      out = make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z),
                        __uint_as_float(raw.w));
    }
    table[idx] = out;
  }
  __syncthreads();

  const float inv = __frcp_rn(__ldg(p.input_scale));
  const float colsf = float(C);
  float4* red = smem + size_t(slots) * L::kSlotF4;  // WPR > 1 exchange, double-buffered
  int parity = 0;

  for (int64_t r = rb + row_slot; r < re; r += L::kRowsPerIter) {
    const int s = p.mod_rows > 0 ? int(r / p.mod_rows - m_lo) : 0;
    const float4* tab = table + size_t(s * WPR + part) * V * P * 32 + lane;
    const size_t row_off = size_t(r) * C + size_t(part) * (C / WPR);

    uint4 xv[V];
    {
      const uint4* xr = reinterpret_cast<const uint4*>(p.x + row_off) + lane;
#pragma unroll
      for (int j = 0; j < V; ++j) xv[j] = ld_stream(xr + j * 32);
    }
    if constexpr (RESID) {
      const uint4* rr = reinterpret_cast<const uint4*>(p.residual + row_off) + lane;
      uint4* ro = reinterpret_cast<uint4*>(p.residual_out + row_off) + lane;
      uint4 rv[V];
#pragma unroll
      for (int j = 0; j < V; ++j) rv[j] = ld_stream(rr + j * 32);
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const float4 gf = tab[(j * P + 4) * 32];
        const float4 bf = tab[(j * P + 5) * 32];
        const uint32_t g[4] = {__float_as_uint(gf.x), __float_as_uint(gf.y),
                               __float_as_uint(gf.z), __float_as_uint(gf.w)};
        const uint32_t b[4] = {__float_as_uint(bf.x), __float_as_uint(bf.y),
                               __float_as_uint(bf.z), __float_as_uint(bf.w)};
        uint4 o;
        o.x = resid2<HAS_BIAS>(xv[j].x, b[0], g[0], rv[j].x);
        o.y = resid2<HAS_BIAS>(xv[j].y, b[1], g[1], rv[j].y);
        o.z = resid2<HAS_BIAS>(xv[j].z, b[2], g[2], rv[j].z);
        o.w = resid2<HAS_BIAS>(xv[j].w, b[3], g[3], rv[j].w);
        xv[j] = o;
        st_stream(ro + j * 32, o);
      }
    }

    dd s1{0.0f, 0.0f}, s2{0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < V; ++j) acc_stats8(xv[j], s1, s2);
    warp_reduce_dd(s1, s2);
    if constexpr (WPR > 1) {
      float4* buf = red + parity * (L::kRowsPerIter * WPR) + row_slot * WPR;
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
    const RowConst k = row_constants(s1, s2, colsf, p.eps);

    uint4* yr = reinterpret_cast<uint4*>(p.y + row_off) + lane;
    uint2* qr = reinterpret_cast<uint2*>(p.q + row_off) + lane;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint4 n = normalise8(xv[j], k);
      const float4 o0 = tab[(j * P + 0) * 32];
      const float4 o1 = tab[(j * P + 1) * 32];
      const float4 h0 = tab[(j * P + 2) * 32];
      const float4 h1 = tab[(j * P + 3) * 32];
      const float ops[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
      const float sh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      uint4 y;
      uint2 q;
      modulate_quant8(n, ops, sh, inv, y, q);
      st_stream(yr + j * 32, y);
      st_stream(qr + j * 32, q);
    }
  }
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
  const float inv = __frcp_rn(__ldg(p.input_scale));
  const float colsf = float(p.cols);

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
    const RowConst k = row_constants(s1, s2, colsf, p.eps);
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
