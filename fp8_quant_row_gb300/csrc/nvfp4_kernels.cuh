// nvfp4_kernels.cuh -- token-concat -> NVFP4 for sm_103a.
//
// "sglang #37141 - FLUX.2 token-cat + NVFP4 fusion" (features and motivation; implementation
// breakdown items 1-3) and the public NVFP4 format (E2M1 elements, one E4M3 scale per 16
// consecutive elements of a row, an fp32 per-tensor global scale g, scales stored in the
// 128x4-tiled layout the FP4 GEMMs read). Per 16-element group of the row cat(a[r], m[r]):
//   amax = max |x_i|
//   code = E4M3_satfinite(RN(g * RN(amax * RN(1/6))))             stored block scale
//   out  = code == +-0 ? 0 : RN(1 / RN(E4M3(code) * RN(1/g)))
//   e_i  = E2M1_satfinite(RN(x_i * out)),  element 2j -> low nibble of byte j
// All roundings are IEEE fp32 round-to-nearest-even; the BF16 concat is never formed.
//
// Work unit: four consecutive groups (64 elements = 128 source bytes) of one part of one row.
// They are one column of one 128x4 scale tile, so their four scale codes form one aligned
// 32-bit word of the scale buffer, and their 32 bytes of packed codes one aligned 32-byte
// store. A thread moves its unit with four 32-byte loads and one 32-byte store; the scale
// words of a warp are regrouped by one shuffle into whole 32-byte sectors (see the kernel).
// Rows past `rows` (the padding of the last 128-row tile) take part with zero scale words.
// The output scale needs one correctly rounded reciprocal per group.
#pragma once

#include "fp8q_device.cuh"

namespace fp8q {

constexpr int kFp4Threads = 256;

// 32-byte streaming load / store (sm_100+ 256-bit global accesses).
__device__ __forceinline__ void ld_stream32(const void* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}
__device__ __forceinline__ void st_stream32(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                  "r"(w[6]), "r"(w[7])
               : "memory");
}

// Value of an E4M3 code (exact: E4M3 -> f16 -> f32 are both widening).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint16_t c = uint16_t(code & 0xFF);
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(uint16_t(h2 & 0xFFFF)));
  return f;
}

// Four packed fp32 pairs (elements 0..7 in order) -> eight E2M1 codes, element 0 in bits 0..3.
// cvt.rn.satfinite.e2m1x2 puts its first source in the high nibble.
__device__ __forceinline__ uint32_t pack_e2m1x8(f2 p0, f2 p1, f2 p2, f2 p3) {
  uint32_t r;
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n"
      "}"
      : "=r"(r)
      : "f"(f2_lo(p0)), "f"(f2_hi(p0)), "f"(f2_lo(p1)), "f"(f2_hi(p1)), "f"(f2_lo(p2)),
        "f"(f2_hi(p2)), "f"(f2_lo(p3)), "f"(f2_hi(p3)));
  return r;
}

// max |x| of a 16-element group held as eight bf16x2 words, as an fp32 value (packed BF16
// abs-max, then the larger magnitude of the two lanes).
__device__ __forceinline__ float group_amax(const uint32_t (&w)[8]) {
  uint32_t m = absmax_bf16x2(w[0], w[1]);
#pragma unroll
  for (int i = 2; i < 8; ++i) m = absmax_bf16x2(m, w[i]);
  const uint32_t lo = m & 0x7FFFu, hi = (m >> 16) & 0x7FFFu;
  return __uint_as_float((lo > hi ? lo : hi) << 16);
}

// The 8 bytes of packed codes of one group, given its output scale.
__device__ __forceinline__ void quant_group(const uint32_t (&w)[8], float out, uint32_t& lo,
                                            uint32_t& hi) {
  const f2 o = f2_make(out, out);
  lo = pack_e2m1x8(mul2(bf2_to_f2(w[0]), o), mul2(bf2_to_f2(w[1]), o), mul2(bf2_to_f2(w[2]), o),
                   mul2(bf2_to_f2(w[3]), o));
  hi = pack_e2m1x8(mul2(bf2_to_f2(w[4]), o), mul2(bf2_to_f2(w[5]), o), mul2(bf2_to_f2(w[6]), o),
                   mul2(bf2_to_f2(w[7]), o));
}

// One warp covers 8 rows x 4 units: the rows {t, t+1} + {0, 32, 64, 96} of one 128-row band
// (t even), whose scale words for one unit fill one aligned 32-byte sector of the scale
// tile. Lane l takes row j = l / 4 of the group and unit k = l % 4 of the warp's four, so
// after one shuffle the warp writes four whole sectors with one store instruction, and the
// L2 never sees a partial-sector scale write. A CTA (8 warps) covers 32 consecutive units
// of its 8 rows. Grid: x = unit blocks of a row, y = row groups (grid-stride).
// Work items are warp-sized: (8-row group, 4 consecutive units), taken in order by the warps of
// a persistent grid (item it of warp w of CTA b: it = b * 8 + w, then + 8 * gridDim.x). A warp
// item covers four scale words of each of its 8 rows, which share 32-byte sectors of the
// 128x4 tile (see the shuffle below). Items rather than CTAs are the unit of balance, so a
// launch of a little more than one wave of CTAs (512 tokens: 768 CTA-sized blocks on 608
// slots) spreads evenly over every warp instead of running a second, mostly empty wave.
__global__ void __launch_bounds__(kFp4Threads) token_cat_nvfp4_kernel(
    uint8_t* __restrict__ q, uint8_t* __restrict__ sf, const uint16_t* __restrict__ a,
    int a_units, const uint16_t* __restrict__ m, int m_units,
    const float* __restrict__ global_scale, int64_t rows, int64_t rows_pad) {
  const int units = a_units + m_units;  // also the number of 4-group scale tiles per row
  const int quads = (units + 3) / 4;    // warp items per 8-row group
  const int64_t items = (rows_pad / 8) * quads;
  const int a_cols = a_units * 64, m_cols = m_units * 64;
  const int lane = threadIdx.x & 31;
  const int j = lane >> 2;                        // row of the group: line parity j & 1, band j >> 1
  // shuffle source for the sector layout: lane L stores word L & 7 of sector L >> 3, which
  // holds line parity (L & 7) >> 2 and band (L & 3)
  const int src_j = ((lane & 3) << 1) | ((lane >> 2) & 1);
  const int src = src_j * 4 + (lane >> 3);
  wait_for_producers();
  const float g = __ldg(global_scale);
  const float inv6 = __frcp_rn(6.0f);
  const float inv_g = __frcp_rn(g);
  constexpr int kWarps = kFp4Threads / 32;

  for (int64_t it = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); it < items;
       it += int64_t(gridDim.x) * kWarps) {
    const int64_t grp = it / quads;
    const int uq = int(it - grp * quads);
    const int ku = uq * 4 + (lane & 3);
    const int st_ku = uq * 4 + (lane >> 3);
    const int64_t band = grp >> 4;
    const int t0 = int(grp & 15) * 2;  // even line of the band
    const int64_t r = band * 128 + (j >> 1) * 32 + t0 + (j & 1);
    uint32_t codes = 0;
    if (r < rows && ku < units) {
      const uint16_t* src_p = ku < a_units ? a + size_t(r) * a_cols + size_t(ku) * 64
                                           : m + size_t(r) * m_cols + size_t(ku - a_units) * 64;
      uint32_t w[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i) ld_stream32(src_p + 16 * i, w[i]);
      float s[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) s[i] = __fmul_rn(g, __fmul_rn(group_amax(w[i]), inv6));
      codes = pack_e4m3x2(s[0], s[1]) | (pack_e4m3x2(s[2], s[3]) << 16);
      uint32_t packed[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c = (codes >> (8 * i)) & 0xFF;
        const float out = (c & 0x7F) ? __frcp_rn(__fmul_rn(e4m3_value(c), inv_g)) : 0.0f;
        quant_group(w[i], out, packed[2 * i], packed[2 * i + 1]);
      }
      st_stream32(q + size_t(r) * (size_t(units) * 32) + size_t(ku) * 32, packed);
    }
    const uint32_t word = __shfl_sync(0xFFFFFFFFu, codes, src);
    if (st_ku < units)
      *reinterpret_cast<uint32_t*>(sf + (size_t(band) * units + st_ku) * 512 + t0 * 16 +
                                   (lane & 7) * 4) = word;
  }
}

}  // namespace fp8q
