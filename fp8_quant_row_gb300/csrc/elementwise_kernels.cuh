// elementwise_kernels.cuh -- the two reduction-free kernels of the path, for sm_103a.
//
// bias_mul_add ("sglang #37116 - Qwen-Image output-bias deferral", key source snippets):
//   y = fma_bf16(RN_bf16(x + bias), gate, residual), the FMA rounded once (native BF16 FMA).
// token_cat_fp8 ("sglang #37162 - FLUX.2 FP8 LayerNorm/quant/QKV fusions", implementation
// breakdown item 4 and key source snippets):
//   q[r, c] = E4M3(RN(v * RN(1/input_scale))), v = a[r, c] for c < a_cols else m[r, c-a_cols],
//   read straight from the two sources: the BF16 concat is never formed.
//
// Both are pure HBM streams. Grid: x = rows (grid-stride beyond 2^31-1), y = column blocks;
// each thread moves several 16-byte source chunks, all loads issued before any use, so
// every warp-wide access is one contiguous 512-byte load or 256-byte store.
#pragma once

#include "fp8q_device.cuh"

namespace fp8q {

constexpr int kEwThreads = 128;
constexpr int kBmaUnroll = 3;  // 128 threads x 3 chunks x 8 = 3072 columns per CTA
constexpr int kCatUnroll = 8;  // 128 threads x 8 chunks x 8 = 8192 columns per CTA

// RPC rows per CTA step, all of their loads issued before any use.
template <int RPC>
__global__ void __launch_bounds__(kEwThreads) bias_mul_add_kernel(
    uint16_t* __restrict__ y, const uint16_t* __restrict__ x, const uint16_t* __restrict__ bias,
    const uint16_t* __restrict__ gate, const uint16_t* __restrict__ residual, int64_t rows,
    int cols) {
  const int chunks = cols / 8;
  const int c0 = (blockIdx.y * kEwThreads) * kBmaUnroll + threadIdx.x;
  const uint4* b4 = reinterpret_cast<const uint4*>(bias);
  const uint4* g4 = reinterpret_cast<const uint4*>(gate);
  wait_for_producers();
  for (int64_t r0 = int64_t(blockIdx.x) * RPC; r0 < rows; r0 += int64_t(gridDim.x) * RPC) {
    uint4 xv[RPC][kBmaUnroll], rv[RPC][kBmaUnroll];
#pragma unroll
    for (int h = 0; h < RPC; ++h) {
      const int64_t r = r0 + h;
      const uint4* x4 = reinterpret_cast<const uint4*>(x + size_t(r) * cols);
      const uint4* r4 = reinterpret_cast<const uint4*>(residual + size_t(r) * cols);
#pragma unroll
      for (int u = 0; u < kBmaUnroll; ++u) {
        const int c = c0 + u * kEwThreads;
        if (r < rows && c < chunks) {
          xv[h][u] = ld_stream(x4 + c);
          rv[h][u] = ld_stream(r4 + c);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBmaUnroll; ++u) {
      const int c = c0 + u * kEwThreads;
      if (c >= chunks) continue;
      const uint4 b = __ldg(b4 + c);
      const uint4 g = __ldg(g4 + c);
      const uint32_t bs[4] = {b.x, b.y, b.z, b.w};
      const uint32_t gs[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int h = 0; h < RPC; ++h) {
        const int64_t r = r0 + h;
        if (r >= rows) continue;
        const uint32_t xs[4] = {xv[h][u].x, xv[h][u].y, xv[h][u].z, xv[h][u].w};
        const uint32_t rs[4] = {rv[h][u].x, rv[h][u].y, rv[h][u].z, rv[h][u].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t xb = pack_bf16x2(__fadd_rn(bf_lo(xs[i]), bf_lo(bs[i])),
                                          __fadd_rn(bf_hi(xs[i]), bf_hi(bs[i])));
          o[i] = fma_bf16x2(xb, gs[i], rs[i]);
        }
        st_stream(reinterpret_cast<uint4*>(y + size_t(r) * cols) + c,
                  make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
}

// 8 bf16 (one 16-byte chunk) -> 8 E4M3 codes (8 bytes).
__device__ __forceinline__ uint2 quant8(const uint4& v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = pack_e4m3x2(__fmul_rn(bf_lo(w[i]), inv), __fmul_rn(bf_hi(w[i]), inv));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__global__ void __launch_bounds__(kEwThreads) token_cat_fp8_kernel(
    uint8_t* __restrict__ q, const uint16_t* __restrict__ a, int a_cols,
    const uint16_t* __restrict__ m, int m_cols, const float* __restrict__ input_scale,
    int64_t rows) {
  wait_for_producers();
  const float inv = __frcp_rn(__ldg(input_scale));
  const int a_chunks = a_cols / 8;
  const int chunks = (a_cols + m_cols) / 8;
  const int c0 = (blockIdx.y * kEwThreads) * kCatUnroll + threadIdx.x;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* ar = reinterpret_cast<const uint4*>(a + size_t(r) * a_cols);
    const uint4* mr = reinterpret_cast<const uint4*>(m + size_t(r) * m_cols);
    uint2* qr = reinterpret_cast<uint2*>(q + size_t(r) * (a_cols + m_cols));
    uint4 v[kCatUnroll];
#pragma unroll
    for (int u = 0; u < kCatUnroll; ++u) {
      const int c = c0 + u * kEwThreads;
      if (c < chunks) v[u] = ld_stream(c < a_chunks ? ar + c : mr + (c - a_chunks));
    }
#pragma unroll
    for (int u = 0; u < kCatUnroll; ++u) {
      const int c = c0 + u * kEwThreads;
      if (c < chunks) st_stream(qr + c, quant8(v[u], inv));
    }
  }
}

}  // namespace fp8q
