// nss_ws_kernels.cuh -- warp-specialised LayerNorm (no affine) -> AdaLN modulate -> dual
// BF16 + E4M3 output for row widths that are multiples of 768 (Qwen-Image: 3072), sm_103a.
//
// Same arithmetic as nss_kernels.cuh ("sglang #37156 - Qwen-Image FP8 norm + activation-quant
// fusion", key source snippets): mu, var (population) from error-free row sums; n =
// RN_bf16((x - mu)/sqrt(var + eps)); y = RN_bf16(fma(n, RN(1 + scale), shift)); q =
// E4M3(RN(y * RN(1/input_scale))). What differs is how a CTA moves rows through the SM:
//
//   producer warp   one lane issues one bulk copy (cp.async.bulk, TMA) per row into a ring of
//                   kStages row stages in shared memory; stage s's `full` mbarrier completes
//                   when the row has landed. A stage is refilled once its `empty` mbarrier
//                   completes, and at most `depth` rows are in flight at a time.
//   statistics      NS warps; each claims the CTA's next row in order (a shared counter), waits
//   warps           for it, forms the error-free row sums and the row constants once per row,
//                   stores them in the stage's constant slot and arrives on its `done` mbarrier.
//   output warps    the row is cut into parts of 768 columns; NO warps per part claim the next
//                   row of their part in order (a counter per part). Each keeps RN(1 + scale)
//                   and shift of its 768 columns in registers for the whole launch, waits for
//                   `done`, writes y and q of its part and arrives on `empty`.
//
// The constants of a row are formed once (not once per warp that touches the row), the
// statistics (FMA-pipe heavy) and output (ALU heavy) phases of different rows run at the same
// time on different warps, no consumer warp loads row data from global memory, and a row
// goes to whichever warp of a role is free first (a static row-to-warp assignment made rows
// wait for one busy warp while others idled).
//
// mbarrier phases: stage s = k % kStages holds rows s, s + kStages, ...; row k is the
// (k / kStages)-th use of its stage and waits for the phase of that parity. Before a stage's
// second and later uses the waiter first checks the stage's row word, which the producer
// writes just before it issues the copy (bounded wait): once it holds k, the stage's previous
// use has been released, so every earlier phase of its barriers has completed and the parity
// cannot be mistaken for an older phase's.
//
// A statistics warp that finds no row left joins the output warps of one part (the same
// per-part claim counter), so the last rows' outputs, which end the CTA, are shared among more
// warps (the producer warp joining as well, once every row is issued, was slower).
//
// Every wait is bounded (kWaitLimitCycles); a wait that runs out records kDevErrWaitTimeout
// in the device error word and the warp stops taking rows. The producer finally waits
// (bounded) for its own copies still in flight before it returns.
#pragma once

#include "nss_kernels.cuh"

namespace fp8q {

constexpr int kWsPartCols = 768;                  // columns of one output part
constexpr int kWsPartChunks = kWsPartCols / 256;  // 16-byte chunks per lane per part (3)

template <int C, int NS, int NO>
struct WsLayout {
  static_assert(C % kWsPartCols == 0, "row width must be a multiple of 768");
  static constexpr int kParts = C / kWsPartCols;
  static constexpr int kRowBytes = C * 2;
  static constexpr int kStatsChunks = C / 256;  // 16-byte chunks per lane of a whole row
  static constexpr int kWarps = NS + kParts * NO + 1;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kProducerWarp = kWarps - 1;
  static constexpr int kLogStages = 5;
  static constexpr int kStages = 1 << kLogStages;  // deeper than NS and NO (see the header)
  static_assert(kStages > NS && kStages > NO, "ring too shallow for the claiming argument");
  // per stage: the row, two float4 of row constants, three mbarriers, the row word; then the
  // claim counters (statistics, one per output part)
  static constexpr size_t kStageBytes = size_t(kRowBytes) + 32 + 24 + 4;
  static constexpr size_t kSmemBytes = size_t(kStages) * kStageBytes + 16 * ((kParts + 4) / 4);
};

// Row constants of the row held in `stage` (this lane's chunks at stage[j * 32]), read from
// shared memory twice: once for max|x| (the accumulator offsets), once for the sums.
template <int VS>
__device__ __forceinline__ RowConst ws_row_stats(const uint4* stage, float cols, float rcols,
                                                 float eps) {
  uint32_t m2 = 0;
#pragma unroll
  for (int j = 0; j < VS; ++j) {
    const uint4 xv = stage[j * 32];
    m2 = absmax_bf16x2(m2, absmax_bf16x2(absmax_bf16x2(xv.x, xv.y), absmax_bf16x2(xv.z, xv.w)));
  }
  const uint32_t mexp =
      __reduce_max_sync(0xffffffffu, (max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu) >> 7) & 0xFFu);
  const RowOffsets off = row_offsets(mexp);
  f2 sx = f2_make(off.K, off.K), sq = f2_make(off.K2, off.K2), ex = f2_make(0.0f, 0.0f),
     eq = ex;
#pragma unroll 4
  for (int j = 0; j < VS; ++j) {
    const uint4 xv = stage[j * 32];
    const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 v = bf2_to_f2(w4[i]);
      f2 s, e;
      fast_two_sum2(sx, v, s, e);
      sx = s;
      ex = add2(ex, e);
      s = fma2(v, v, sq);
      e = fma2(v, v, sub2(sq, s));
      sq = s;
      eq = add2(eq, e);
    }
  }
  const dd s1 = warp_sum_offset(sx, ex, off.K, off.ek, true);
  const dd s2 = warp_sum_offset(sq, eq, off.K2, off.ek2, false);
  return row_constants(s1, s2, cols, rcols, eps);
}

// Exact-path fix-up of one 8-element chunk, for the few chunks that hold an uncertain element
// (same rule as fix_uncertain8, inlined here: the call was dearer than the code it runs).
__device__ __forceinline__ uint4 ws_fix_uncertain8(const uint4 x, const uint4 n,
                                                   const RowConst kc) {
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

// y and q of one 768-column part of a row: this lane's chunks are xs[j * 32] (shared memory),
// its RN(1 + scale) and shift pairs ops[j][i], sh[j][i] (registers). kSmall adds the
// per-element |t| < t_small test; t_small is zero unless the row's mean lies close to a bf16
// value (where the absolute error of t matters), so the body without the test serves almost
// every row (the choice is per row and uniform across the warp).
template <bool kSmall>
__device__ __forceinline__ void ws_part_outputs(const uint4* xs, const f2 (&ops)[kWsPartChunks][4],
                                                const f2 (&sh)[kWsPartChunks][4],
                                                const RowConst& kc, f2 inv2, uint4* yr,
                                                uint2* qr) {
  const f2 mu2 = f2_make(kc.mu_hi, kc.mu_hi), r2 = f2_make(kc.r_hi, kc.r_hi),
           c2 = f2_make(kc.c, kc.c);
#pragma unroll
  for (int j = 0; j < kWsPartChunks; ++j) {
    const uint4 xv = xs[j * 32];
    const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
    float n[8];
    bool any = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 tt = fma2(sub2(bf2_to_f2(w4[i]), mu2), r2, c2);
      const float t0 = f2_lo(tt), t1 = f2_hi(tt);
      any |= near_bf16_midpoint(t0) | near_bf16_midpoint(t1);
      if (kSmall) any |= (fabsf(t0) < kc.t_small) | (fabsf(t1) < kc.t_small);
      n[2 * i] = round_bf16(t0);
      n[2 * i + 1] = round_bf16(t1);
    }
    if (any) {
      uint4 nb = make_uint4(pack_bf16x2(n[0], n[1]), pack_bf16x2(n[2], n[3]),
                            pack_bf16x2(n[4], n[5]), pack_bf16x2(n[6], n[7]));
      nb = ws_fix_uncertain8(xv, nb, kc);
      const uint32_t nw[4] = {nb.x, nb.y, nb.z, nb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        n[2 * i] = bf_lo(nw[i]);
        n[2 * i + 1] = bf_hi(nw[i]);
      }
    }
    uint32_t yw[4];
    f2 yb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f2 yf = fma2(f2_make(n[2 * i], n[2 * i + 1]), ops[j][i], sh[j][i]);
      // y rounded to bf16 as fp32 values (for q), and the same values packed (for y)
      yb[i] = f2_make(round_bf16(f2_lo(yf)), round_bf16(f2_hi(yf)));
      yw[i] = __byte_perm(__float_as_uint(f2_lo(yb[i])), __float_as_uint(f2_hi(yb[i])), 0x7632);
    }
    st_stream(yr + j * 32, make_uint4(yw[0], yw[1], yw[2], yw[3]));
    st_stream(qr + j * 32, make_uint2(quant4f(yb[0], yb[1], inv2), quant4f(yb[2], yb[3], inv2)));
  }
}

template <int C, int NS, int NO>
__global__ void __launch_bounds__(WsLayout<C, NS, NO>::kThreads, 1)
    nss_ws_kernel(const NssParams p, const int64_t n_mod, const int depth) {
  using L = WsLayout<C, NS, NO>;
  constexpr int P = L::kParts;
  constexpr int S = L::kStages;
  extern __shared__ __align__(128) unsigned char ws_smem[];
  unsigned char* ring = ws_smem;
  float4* kslot = reinterpret_cast<float4*>(ws_smem + size_t(S) * L::kRowBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(kslot + 2 * S);
  uint64_t* done = full + S;
  uint64_t* empty = done + S;
  int* rowid = reinterpret_cast<int*>(empty + S);
  int* next_stats = rowid + S;  // then one counter per output part

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RowBlock blk = cta_rows(p.rows, p.mod_rows, n_mod, blockIdx.x, gridDim.x);
  const int n = int(blk.end - blk.begin);
  if (n <= 0) return;  // uniform across the CTA
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(done + s, 1);
      mbar_init(empty + s, P);
      rowid[s] = -1;
    }
    for (int c = 0; c <= P; ++c) next_stats[c] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  wait_for_producers();
  allow_dependents();

  if (warp == L::kProducerWarp) {
    if (lane == 0) {
      const unsigned char* src = reinterpret_cast<const unsigned char*>(p.x) +
                                 size_t(blk.begin) * L::kRowBytes;
      int issued = 0;
      for (int k = 0, s = 0, u = 0; k < n; ++k) {
        if (u > 0 && !mbar_wait(empty + s, (u - 1) & 1)) {
          report_device_error(kDevErrWaitTimeout);
          break;
        }
        // at most `depth` rows in flight: row k waits for row k - depth to land (that row is
        // still the last one issued into its stage, since depth < S)
        if (depth < S && k >= depth) {
          const int kd = k - depth;
          if (!mbar_wait(full + kd % S, (kd / S) & 1)) {
            report_device_error(kDevErrWaitTimeout);
            break;
          }
        }
        ws_set_row(rowid + s, k);
        mbar_arrive_expect_tx(full + s, L::kRowBytes);
        bulk_load(ring + size_t(s) * L::kRowBytes, src + size_t(k) * L::kRowBytes, L::kRowBytes,
                  full + s);
        issued = k + 1;
        if (++s == S) {
          s = 0;
          ++u;
        }
      }
      // The last copy into each stage has landed before this warp returns (always true on the
      // normal path, where every row is consumed; it matters only after a wait ran out).
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / S) * S;
        if (!mbar_wait(full + s, (last / S) & 1)) report_device_error(kDevErrWaitTimeout);
      }
    }
    return;
  }

  int part;
  if (warp < NS) {
    // statistics warp
    const float colsf = float(C);
    const float rcols = __frcp_rn(colsf);
    for (int k = ws_claim(next_stats); k < n; k = ws_claim(next_stats)) {
      const int s = k & (S - 1), u = k >> L::kLogStages;
      if (!ws_wait_row(full + s, rowid, s, k, u)) {
        report_device_error(kDevErrWaitTimeout);
        return;
      }
      const uint4* stage = reinterpret_cast<const uint4*>(ring + size_t(s) * L::kRowBytes) + lane;
      const RowConst kc = ws_row_stats<L::kStatsChunks>(stage, colsf, rcols, p.eps);
      if (lane == 0) {
        kslot[2 * s] = make_float4(kc.mu_hi, kc.mu_lo, kc.r_hi, kc.r_lo);
        kslot[2 * s + 1] =
            make_float4(kc.c, mean_far_from_bf16_grid(kc.mu_hi) ? 0.0f : kc.t_small, 0.0f, 0.0f);
        mbar_arrive(done + s);
      }
    }
    // No row is left for the statistics role (the end of the CTA's rows): the warp joins the
    // output warps of part warp % P, whose rows still wait there, and takes rows from the same
    // counter, so every part-row is still written once.
    part = warp % P;
  } else {
    part = (warp - NS) % P;
  }

  // output warp: part `part` of the rows it claims
  const size_t col0 = size_t(part) * kWsPartCols;
  f2 ops[kWsPartChunks][4], sh[kWsPartChunks][4];
  {
    const size_t mrow = size_t(blk.mod) * C + col0;
#pragma unroll
    for (int j = 0; j < kWsPartChunks; ++j) {
      const size_t col = mrow + size_t(j * 32 + lane) * 8;
      const uint4 sc = __ldg(reinterpret_cast<const uint4*>(p.scale + col));
      const uint4 sf = __ldg(reinterpret_cast<const uint4*>(p.shift + col));
      const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w}, sfw[4] = {sf.x, sf.y, sf.z, sf.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ops[j][i] = f2_make(__fadd_rn(1.0f, bf_lo(scw[i])), __fadd_rn(1.0f, bf_hi(scw[i])));
        sh[j][i] = bf2_to_f2(sfw[i]);
      }
    }
  }
  const float inv = __frcp_rn(__ldg(p.input_scale));
  const f2 inv2 = f2_make(inv, inv);
  int* const next_row = next_stats + 1 + part;
  for (int k = ws_claim(next_row); k < n; k = ws_claim(next_row)) {
    const int s = k & (S - 1), u = k >> L::kLogStages;
    // `full` first: the stage's row word and the row's landing, then its constants
    if (!ws_wait_row(full + s, rowid, s, k, u) || !mbar_wait(done + s, u & 1)) {
      report_device_error(kDevErrWaitTimeout);
      break;
    }
    const float4 k0 = kslot[2 * s], k1 = kslot[2 * s + 1];
    RowConst kc;
    kc.mu_hi = k0.x;
    kc.mu_lo = k0.y;
    kc.r_hi = k0.z;
    kc.r_lo = k0.w;
    kc.c = k1.x;
    kc.t_small = k1.y;
    const uint4* xs =
        reinterpret_cast<const uint4*>(ring + size_t(s) * L::kRowBytes + col0 * 2) + lane;
    const size_t off = size_t(blk.begin + k) * C + col0;
    uint4* yr = reinterpret_cast<uint4*>(p.y + off) + lane;
    uint2* qr = reinterpret_cast<uint2*>(p.q + off) + lane;
    if (kc.t_small != 0.0f)
      ws_part_outputs<true>(xs, ops, sh, kc, inv2, yr, qr);
    else
      ws_part_outputs<false>(xs, ops, sh, kc, inv2, yr, qr);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
}

}  // namespace fp8q
