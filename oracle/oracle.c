/*
 * oracle.c -- plain CPU oracle for the row-wise DiT-block prologue:
 *   LayerNorm (no affine) -> AdaLN modulate -> static per-tensor FP8 E4M3 quantisation,
 * and its variants (gated scale-residual with input bias, deferred output-bias epilogue,
 * token-concat -> FP8, token-concat -> NVFP4), and the attention-input epilogue after the
 * packed QKV GEMM (per-head Q/K RMSNorm, interleaved RoPE, V copy, joint [text, image] pack).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the correctness reference that the CUDA path is
 * compared against. Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it; the product path (the C-ABI library and its Python binding) never calls it, and
 * it shares no code, header, table or helper with that path.
 *
 * Style: single-threaded, one element at a time, in the order the pages state the steps.
 * Floating point is fp64 wherever the pages leave the precision open (LayerNorm statistics,
 * the normalised value before its BF16 rounding, the single-rounded BF16 FMA). Where the
 * pages fix fp32 (the modulate FMA, the reciprocal, the quantise multiply) the oracle uses
 * IEEE fp32 exactly as stated. Build with -ffp-contract=off so no a*b+c is fused silently.
 *
 * Sources (page title, section):
 *  [QWEN-NQ]  "sglang #37156 - Qwen-Image FP8 norm + activation-quant fusion",
 *             sections "implementation breakdown" and "key source snippets"
 *             (norm_scale_shift.cuh excerpt: norm, modulate, reciprocal, clamp + cast).
 *  [QWEN-BIAS] "sglang #37116 - Qwen-Image output-bias deferral",
 *             "key source snippets" (bias_mul_add_kernel excerpt) and
 *             "review highlights" (BF16 rounding of the bias add, native BF16 FMA,
 *             the x=-24576 worked example).
 *  [FLUX-FP8] "sglang #37162 - FLUX.2 FP8 LayerNorm/quant/QKV fusions",
 *             "implementation breakdown" item 4 and "key source snippets"
 *             (_token_cat_fp8_kernel excerpt: cat(attention, mlp) * (1/scale), clamp, cast).
 *  [FLUX-FP4] "sglang #37141 - FLUX.2 token-cat + NVFP4 fusion", "features and motivation"
 *             (attention 6144 + MLP 18432 BF16 -> NVFP4 without the concat) and
 *             "implementation breakdown" items 1-3 (per-group conversion primitive,
 *             128x4-swizzled block-scale offsets, input_scale_inv as the global scale).
 *  [QWEN-QKV] "sglang #37123 - Qwen-Image FP8 QKV fusion", "implementation breakdown" item 3
 *             (Q/K RMSNorm + RoPE, V copy, joint [text, image] output; head_dim 128) and
 *             "key source snippets" (per-stream norm weights and epsilons, per-stream cos/sin
 *             caches, is_neox=False: interleaved pairs).
 *  [FLUX-QKV] "sglang #37162 - FLUX.2 FP8 LayerNorm/quant/QKV fusions", "implementation
 *             breakdown" item 3 (QK RMSNorm, RoPE, QKV pack and text/image concat in one kernel).
 *  [NVFP4]    the public NVFP4 format: E2M1 elements (values 0, 0.5, 1, 1.5, 2, 3, 4, 6),
 *             one E4M3 scale per 16 consecutive elements of a row, an fp32 per-tensor scale;
 *             and the public 128x4 block-scale tile layout of the FP4 GEMMs that consume it.
 *
 * Parity pins: every function below is pinned by tests/test_oracle_pins.py against
 * something other than itself (exact rational arithmetic, torch's float8/bfloat16 casts,
 * closed forms, brute force). No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------------------ */
/* BF16 <-> fp64                                                                        */
/* ------------------------------------------------------------------------------------ */

/* Value of a bfloat16 bit pattern: bf16 is the upper half of an IEEE binary32. */
ORC_API double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint16_t bf16_bits_of_exact(double v)
{
    /* v is exactly representable in bf16 (or is +-0 / +-Inf): go through binary32. */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/*
 * Round s + tiny to bfloat16, ties to even, where "tiny" is an infinitesimal whose sign is
 * sticky_sign (-1, 0 or +1) and whose magnitude is below any bf16 quantum. With
 * sticky_sign = 0 this is plain round-to-nearest-even of s.
 *
 * Definition used: bf16 has an 8-bit significand (7 stored bits), minimum normal exponent
 * -126, subnormal quantum 2^-133, largest finite (2 - 2^-7) * 2^127. A value is rounded to
 * the nearest multiple of its binade's quantum q = 2^(e-7) (e = floor(log2|s|), clamped to
 * -126 below the normal range); halfway cases go to the even multiple. Magnitudes that round
 * to 2^128 or beyond overflow to infinity.
 */
static uint16_t bf16_round(double s, int sticky_sign)
{
    if (isnan(s))
        return 0x7FC0;
    if (isinf(s))
        return s > 0 ? 0x7F80 : 0xFF80;
    const int neg = signbit(s) != 0;
    double a = fabs(s);
    if (a == 0.0) {
        if (sticky_sign == 0)
            return neg ? 0x8000 : 0x0000;
        /* An exact zero with a nonzero remainder cannot occur for the callers here
         * (TwoSum returns s == 0 only with e == 0); treat it as the remainder's sign. */
        return sticky_sign < 0 ? 0x8000 : 0x0000;
    }
    int E;
    (void)frexp(a, &E);          /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;               /* a in [2^e, 2^(e+1)) */
    if (e < -126)
        e = -126;                /* subnormal range: fixed quantum 2^-133 */
    const double q = ldexp(1.0, e - 7);
    const double k = a / q;      /* exact: division by a power of two */
    const double fl = floor(k);
    const double frac = k - fl;  /* exact */
    /* Direction of the infinitesimal relative to |s|: +1 means "slightly larger magnitude". */
    const int away = (sticky_sign == 0) ? 0 : (((sticky_sign > 0) != neg) ? +1 : -1);
    double kr;
    if (frac > 0.5)
        kr = fl + 1.0;
    else if (frac < 0.5)
        kr = fl;
    else if (away > 0)
        kr = fl + 1.0;
    else if (away < 0)
        kr = fl;
    else
        kr = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0; /* tie: even multiple */
    /* frac == 0 with a nonzero remainder keeps the exact value: the remainder is far below
     * half a quantum, which the branches above already give (frac < 0.5 -> fl). */
    double r = kr * q;
    if (r >= ldexp(1.0, 128))
        return neg ? 0xFF80 : 0x7F80;
    uint16_t b = bf16_bits_of_exact(r);
    return neg ? (uint16_t)(b | 0x8000) : b;
}

/* Round-to-nearest-even of an fp64 value to bf16 (one rounding). */
ORC_API uint16_t orc_bf16_from_f64(double v) { return bf16_round(v, 0); }

/* Round-to-nearest-even of an fp32 value to bf16 (fp32 -> fp64 is exact). */
ORC_API uint16_t orc_bf16_from_f32(float v) { return bf16_round((double)v, 0); }

/* Knuth's TwoSum: s = fl(a+b) and e with s + e == a + b exactly (no FMA, no reordering). */
static void two_sum(double a, double b, double *s, double *e)
{
    double sum = a + b;
    double bv = sum - a;
    double av = sum - bv;
    double br = b - bv;
    double ar = a - av;
    *s = sum;
    *e = ar + br;
}

/*
 * Single-rounded BF16 fused multiply-add: RN_bf16(a*b + c) with one rounding of the exact
 * value, which is what a native BF16 FMA computes [QWEN-BIAS, key source snippets: the
 * kernel calls the native BF16 FMA after the BF16-rounded bias add; review highlights: an
 * fp32 round trip loses the product's tie information at large magnitudes].
 * The product of two 8-bit significands is exact in fp64; TwoSum gives the sum as s + e
 * exactly; bf16_round then rounds s with e as the sticky remainder (e is far below half a
 * bf16 quantum of s, and s itself can sit exactly on a bf16 midpoint only because of e).
 */
ORC_API uint16_t orc_bf16_fma(uint16_t a, uint16_t b, uint16_t c)
{
    const double da = orc_bf16_to_f64(a), db = orc_bf16_to_f64(b), dc = orc_bf16_to_f64(c);
    const double p = da * db; /* exact */
    if (!isfinite(p) || !isfinite(dc))
        return orc_bf16_from_f64(p + dc);
    double s, e;
    two_sum(p, dc, &s, &e);
    const int sticky = (e > 0) - (e < 0);
    return bf16_round(s, sticky);
}

/* RN_bf16(a + b) of two bf16 values: the exact sum is rounded once. */
ORC_API uint16_t orc_bf16_add(uint16_t a, uint16_t b)
{
    const double da = orc_bf16_to_f64(a), db = orc_bf16_to_f64(b);
    if (!isfinite(da) || !isfinite(db))
        return orc_bf16_from_f64(da + db);
    double s, e;
    two_sum(da, db, &s, &e);
    const int sticky = (e > 0) - (e < 0);
    return bf16_round(s, sticky);
}

/* ------------------------------------------------------------------------------------ */
/* FP8 E4M3 (the "fn" variant: no infinities, 0x7F/0xFF are NaN, max finite 448)         */
/* ------------------------------------------------------------------------------------ */

/* Decoded value of an E4M3 code: sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 is subnormal (m * 2^-9); code 0x7F / 0xFF is NaN. */
ORC_API double orc_e4m3_decode(uint8_t c)
{
    const int s = c >> 7, ef = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (ef == 0xF && m == 7)
        return NAN;
    if (ef == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, ef - 7);
    return s ? -v : v;
}

static double g_e4m3_pos[127]; /* decoded values of codes 0x00..0x7E, ascending */
static int g_e4m3_ready = 0;

static void e4m3_table_init(void)
{
    if (g_e4m3_ready)
        return;
    for (int c = 0; c < 127; ++c)
        g_e4m3_pos[c] = orc_e4m3_decode((uint8_t)c);
    g_e4m3_ready = 1;
}

/*
 * Saturating round-to-nearest-even encode to E4M3: clamp to [-448, 448] first (the pages
 * clamp to +-kFloatMax before the cast [QWEN-NQ key source snippets]; the Triton path
 * clamps to [FP8_MIN, FP8_MAX] [FLUX-FP8 key source snippets]), then pick the code whose
 * value is nearest, ties to the code with an even mantissa (code LSB 0). Negative inputs
 * that round to zero give 0x80 (-0). NaN gives 0x7F.
 */
ORC_API uint8_t orc_e4m3_encode(float v)
{
    e4m3_table_init();
    if (isnan(v))
        return 0x7F;
    const int neg = signbit(v) != 0;
    double a = fabs((double)v);
    uint8_t code;
    if (a >= 448.0) {
        code = 0x7E;
    } else {
        /* binary search: largest code lo with value <= a (codes ascend with value) */
        int lo = 0, hi = 126;
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (g_e4m3_pos[mid] <= a)
                lo = mid;
            else
                hi = mid - 1;
        }
        if (g_e4m3_pos[lo] == a) {
            code = (uint8_t)lo;
        } else {
            const int up = lo + 1; /* exists because a < 448 = value(0x7E) */
            const double dlo = a - g_e4m3_pos[lo];  /* exact: few significant bits */
            const double dup = g_e4m3_pos[up] - a;
            if (dlo < dup)
                code = (uint8_t)lo;
            else if (dup < dlo)
                code = (uint8_t)up;
            else
                code = (uint8_t)((lo & 1) == 0 ? lo : up);
        }
    }
    return neg ? (uint8_t)(code | 0x80) : code;
}

/* ------------------------------------------------------------------------------------ */
/* Reciprocal and quantise stage                                                        */
/* ------------------------------------------------------------------------------------ */

/* inv = RN_fp32(1 / s): IEEE fp32 division, correctly rounded. (The pages' kernel uses
 * the PTX div.full.f32 form to match Triton [QWEN-NQ key source snippets]; the correctly
 * rounded quotient is the reading this build takes.) */
ORC_API float orc_recip_f32(float s)
{
    volatile float one = 1.0f; /* keep the division at run time, in fp32 */
    return one / s;
}

/* q = E4M3(RN_fp32(v * inv)) [QWEN-NQ: scaled = float(rounded) * input_scale_inv]. */
ORC_API uint8_t orc_quantize(float v, float inv)
{
    volatile float prod = v * inv; /* one fp32 rounding, no contraction */
    return orc_e4m3_encode(prod);
}

/* ------------------------------------------------------------------------------------ */
/* LayerNorm (no affine) in fp64                                                         */
/* ------------------------------------------------------------------------------------ */

/*
 * Normalised values of one row, before the BF16 rounding: t_j = (x_j - mu) / sqrt(var + eps)
 * with mu = sum(x)/C and var = sum((x - mu)^2)/C (population variance), no affine weight or
 * bias [QWEN-NQ implementation breakdown item 2: layer norm without affine; key source
 * snippets: (v - mean) * factor]. Two passes, fp64, index order. eps is the fp32 value the
 * caller passes, widened exactly.
 */
ORC_API void orc_ln_row_t(const uint16_t *x, int64_t cols, float eps, double *t)
{
    double sum = 0.0;
    for (int64_t j = 0; j < cols; ++j)
        sum += orc_bf16_to_f64(x[j]);
    const double mu = sum / (double)cols;
    double ss = 0.0;
    for (int64_t j = 0; j < cols; ++j) {
        const double d = orc_bf16_to_f64(x[j]) - mu;
        ss += d * d;
    }
    const double var = ss / (double)cols;
    const double rstd = 1.0 / sqrt(var + (double)eps);
    for (int64_t j = 0; j < cols; ++j)
        t[j] = (orc_bf16_to_f64(x[j]) - mu) * rstd;
}

/* Modulate one element: y = RN_bf16(RN_fp32(n * RN_fp32(1 + scale) + shift)) with a single
 * fp32 FMA [QWEN-NQ key source snippets: bf16(norm * (1.0f + sc) + sh), which the CUDA
 * compiler contracts to one FMA]. */
ORC_API uint16_t orc_modulate(uint16_t n, uint16_t scale, uint16_t shift)
{
    const float nf = (float)orc_bf16_to_f64(n);
    volatile float one_plus = 1.0f + (float)orc_bf16_to_f64(scale); /* fp32 add */
    const float r = fmaf(nf, one_plus, (float)orc_bf16_to_f64(shift));
    return orc_bf16_from_f32(r);
}

/* ------------------------------------------------------------------------------------ */
/* Whole operations (row-major, contiguous; bf16 as uint16 bits, E4M3 as uint8 codes)     */
/* ------------------------------------------------------------------------------------ */

static int64_t mod_row(int64_t r, int64_t mod_rows) { return mod_rows > 0 ? r / mod_rows : 0; }

/* LayerNorm -> modulate -> dual output (bf16 y, E4M3 q) for rows of width cols.
 * scale/shift row for data row r is r / mod_rows (mod_rows == 0: one row for all). */
ORC_API int orc_nss_fp8(uint16_t *y, uint8_t *q, const uint16_t *x, const uint16_t *scale,
                        const uint16_t *shift, int64_t mod_rows, float input_scale, int64_t rows,
                        int64_t cols, float eps, double *t_scratch)
{
    const float inv = orc_recip_f32(input_scale);
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * cols;
        const int64_t m = mod_row(r, mod_rows);
        orc_ln_row_t(xr, cols, eps, t_scratch);
        for (int64_t j = 0; j < cols; ++j) {
            const uint16_t n = orc_bf16_from_f64(t_scratch[j]);
            const uint16_t yv = orc_modulate(n, scale[m * cols + j], shift[m * cols + j]);
            y[r * cols + j] = yv;
            q[r * cols + j] = orc_quantize((float)orc_bf16_to_f64(yv), inv);
        }
    }
    return 0;
}

/* Deferred output-bias epilogue: y = RN_bf16(RN_bf16(x + bias) * gate + residual), the
 * second rounding single (native BF16 FMA) [QWEN-BIAS key source snippets]. bias and gate
 * are one row of width cols, broadcast over rows. */
ORC_API int orc_bias_mul_add(uint16_t *y, const uint16_t *x, const uint16_t *bias,
                             const uint16_t *gate, const uint16_t *residual, int64_t rows,
                             int64_t cols)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < cols; ++j) {
            const uint16_t xb = orc_bf16_add(x[r * cols + j], bias[j]);
            y[r * cols + j] = orc_bf16_fma(xb, gate[j], residual[r * cols + j]);
        }
    return 0;
}

/*
 * Gated scale-residual form with optional input bias, then the LayerNorm path:
 *   xb = bias ? RN_bf16(x + bias) : x
 *   residual_out = RN_bf16(xb * gate + residual)          (single rounding)
 *   (y, q) = nss_fp8(residual_out)
 * [QWEN-NQ implementation breakdown item 1 (ScaleResidualNormScaleShiftFp8Kernel);
 *  QWEN-BIAS implementation breakdown item 3 (x + bias, gated residual, LayerNorm,
 *  scale/shift in one kernel)]. gate/scale/shift follow mod_rows; bias is one row.
 */
ORC_API int orc_scale_residual_nss_fp8(uint16_t *residual_out, uint16_t *y, uint8_t *q,
                                       const uint16_t *x, const uint16_t *residual,
                                       const uint16_t *bias, const uint16_t *gate,
                                       const uint16_t *scale, const uint16_t *shift,
                                       int64_t mod_rows, float input_scale, int64_t rows,
                                       int64_t cols, float eps, double *t_scratch)
{
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t m = mod_row(r, mod_rows);
        for (int64_t j = 0; j < cols; ++j) {
            const uint16_t xv = x[r * cols + j];
            const uint16_t xb = bias ? orc_bf16_add(xv, bias[j]) : xv;
            residual_out[r * cols + j] = orc_bf16_fma(xb, gate[m * cols + j], residual[r * cols + j]);
        }
    }
    /* The LayerNorm stage reads the updated residual exactly as nss_fp8 would; each data row
     * keeps its own modulation row, so run it row by row with the row's modulation slice. */
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t m = mod_row(r, mod_rows);
        orc_nss_fp8(y + r * cols, q + r * cols, residual_out + r * cols, scale + m * cols,
                    shift + m * cols, 0, input_scale, 1, cols, eps, t_scratch);
    }
    return 0;
}

/* Token-concat -> FP8: q[r, c] = E4M3(RN_fp32(v * inv)), v = a[r, c] for c < a_cols else
 * m[r, c - a_cols]; output row stride a_cols + m_cols [FLUX-FP8 key source snippets]. */
ORC_API int orc_token_cat_fp8(uint8_t *q, const uint16_t *a, int64_t a_cols, const uint16_t *m,
                              int64_t m_cols, float input_scale, int64_t rows)
{
    const float inv = orc_recip_f32(input_scale);
    const int64_t oc = a_cols + m_cols;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < oc; ++c) {
            const uint16_t v = c < a_cols ? a[r * a_cols + c] : m[r * m_cols + (c - a_cols)];
            q[r * oc + c] = orc_quantize((float)orc_bf16_to_f64(v), inv);
        }
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Token-concat -> NVFP4                                                                 */
/* ------------------------------------------------------------------------------------ */

/* Value of an E2M1 code [NVFP4]: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
 * exponent field 0 is subnormal (m * 0.5). Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
ORC_API double orc_e2m1_decode(uint8_t c)
{
    const int ef = (c >> 1) & 3, m = c & 1;
    const double v = ef == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, ef - 1);
    return (c & 8) ? -v : v;
}

/*
 * Saturating round-to-nearest-even encode to E2M1: magnitudes at or above 6 give 6; below,
 * the nearest of the eight magnitudes, a tie going to the code with mantissa bit 0. The
 * sign bit is the sign of v, also when the magnitude rounds to 0 (-0.1 -> 0x8). E2M1 has no
 * NaN: a NaN input gives 0 here and is outside the operation's contract.
 */
ORC_API uint8_t orc_e2m1_encode(float v)
{
    if (isnan(v))
        return 0;
    const uint8_t sign = signbit(v) ? 8 : 0;
    const double a = fabs((double)v);
    if (a >= 6.0)
        return sign | 7;
    uint8_t best = 0; /* below 6 every distance is exact in fp64 */
    for (uint8_t c = 1; c < 8; ++c) { /* magnitudes ascend with the code */
        const double d_best = fabs(a - orc_e2m1_decode(best));
        const double d_c = fabs(a - orc_e2m1_decode(c));
        if (d_c < d_best || (d_c == d_best && (c & 1) == 0))
            best = c;
    }
    return sign | best;
}

/*
 * One 16-element group [NVFP4; FLUX-FP4 implementation breakdown item 1]. Reading of the
 * conversion step, in IEEE fp32 with every operation correctly rounded:
 *   amax  = max |x_i|                                   (exact)
 *   s     = RN(g * RN(amax * RN(1/6)))                  block scale before encoding
 *   code  = E4M3_satfinite(s)                           stored block scale
 *   out   = code == +-0 ? 0 : RN(1 / RN(E4M3(code) * RN(1/g)))
 *   e_i   = E2M1_satfinite(RN(x_i * out))
 * g is the per-tensor global scale (the GEMM's input_scale_inv). Element 2j goes to the
 * low nibble of byte j, element 2j+1 to the high nibble. Returns the scale code.
 */
ORC_API uint8_t orc_nvfp4_group(const uint16_t *x, float g, uint8_t *packed)
{
    double amax = 0.0;
    for (int i = 0; i < 16; ++i) {
        const double a = fabs(orc_bf16_to_f64(x[i]));
        if (a > amax)
            amax = a;
    }
    const float inv6 = 1.0f / 6.0f;
    const float s = g * ((float)amax * inv6);
    const uint8_t code = orc_e4m3_encode(s);
    float out = 0.0f;
    if ((code & 0x7F) != 0) {
        const float inv_g = 1.0f / g;
        const float d = (float)orc_e4m3_decode(code) * inv_g;
        out = 1.0f / d;
    }
    for (int j = 0; j < 8; ++j) {
        const uint8_t lo = orc_e2m1_encode((float)orc_bf16_to_f64(x[2 * j]) * out);
        const uint8_t hi = orc_e2m1_encode((float)orc_bf16_to_f64(x[2 * j + 1]) * out);
        packed[j] = (uint8_t)(lo | (hi << 4));
    }
    return code;
}

/*
 * Byte offset of block scale (m, k) -- row m, 16-element group k of K groups per row -- in
 * the 128x4-tiled layout [FLUX-FP4 implementation breakdown item 1: 128x4 swizzled scale
 * offsets]: rows are padded to a multiple of 128 and groups to a multiple of 4; each
 * 128-row x 4-group tile is one 512-byte block, blocks ordered row-tile-major then
 * group-tile; inside a block, tile row t (0..127) and tile column c (0..3) sit at byte
 * (t mod 32) * 16 + (t div 32) * 4 + c.
 */
ORC_API int64_t orc_nvfp4_sf_offset(int64_t m, int64_t k, int64_t K)
{
    const int64_t k_tiles = (K + 3) / 4;
    const int64_t t = m % 128, c = k % 4;
    return ((m / 128) * k_tiles + k / 4) * 512 + (t % 32) * 16 + (t / 32) * 4 + c;
}

/*
 * Token-concat -> NVFP4 [FLUX-FP4 features and motivation; implementation breakdown items
 * 1-3]: the row r of cat(a, m) (a_cols + m_cols wide, a multiple of 16) is quantised group by
 * group with orc_nvfp4_group, without forming the concatenation. q is [rows, cols/2] packed
 * bytes; sf is the padded 128x4-tiled scale buffer of ceil(rows/128)*128 x ceil(K/4)*4 bytes,
 * K = cols/16, whose padding entries (rows >= rows, groups >= K) are 0.
 */
ORC_API int orc_token_cat_nvfp4(uint8_t *q, uint8_t *sf, const uint16_t *a, int64_t a_cols,
                                const uint16_t *m, int64_t m_cols, float g, int64_t rows)
{
    const int64_t cols = a_cols + m_cols;
    if (cols % 16 != 0)
        return 1;
    const int64_t K = cols / 16;
    const int64_t m_pad = (rows + 127) / 128 * 128, k_pad = (K + 3) / 4 * 4;
    memset(sf, 0, (size_t)(m_pad * k_pad));
    uint16_t grp[16];
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            for (int i = 0; i < 16; ++i) {
                const int64_t c = 16 * k + i;
                grp[i] = c < a_cols ? a[r * a_cols + c] : m[r * m_cols + (c - a_cols)];
            }
            sf[orc_nvfp4_sf_offset(r, k, K)] = orc_nvfp4_group(grp, g, q + r * (cols / 2) + 8 * k);
        }
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* QKV epilogue: per-head RMSNorm + interleaved RoPE, V copy, joint [text, image] pack      */
/* ------------------------------------------------------------------------------------ */

/*
 * RMSNorm of one head vector of D BF16 values with a BF16 weight [QWEN-QKV implementation
 * breakdown item 3: Q/K RMS norm per head]: n_j = RN_bf16(x_j * w_j / sqrt(sum_i x_i^2 / D +
 * eps)), the exact value rounded once. fp64: the squares of BF16 values are exact, their sum
 * is exact unless the magnitudes span more than ~2^18, and the one division and square root
 * are correctly rounded, so the fp64 value is within a few 2^-53 of the exact one.
 */
ORC_API void orc_rms_norm_head(const uint16_t *x, const uint16_t *w, int64_t D, float eps,
                               uint16_t *n)
{
    double ss = 0.0;
    for (int64_t j = 0; j < D; ++j) {
        const double v = orc_bf16_to_f64(x[j]);
        ss += v * v;
    }
    const double rrms = 1.0 / sqrt(ss / (double)D + (double)eps);
    for (int64_t j = 0; j < D; ++j)
        n[j] = orc_bf16_from_f64(orc_bf16_to_f64(x[j]) * orc_bf16_to_f64(w[j]) * rrms);
}

/*
 * Interleaved (GPT-J style, is_neox=False) rotary embedding of one head vector [QWEN-QKV key
 * source snippets]: pair i = (n[2i], n[2i+1]) is rotated by (c_i, s_i) = (cos_sin[i],
 * cos_sin[D/2 + i]) from the fp32 cache row, each product and the sum rounded to fp32 as
 * separate operations (no fused multiply-add), then to BF16:
 *   o[2i]   = RN_bf16(RN32(RN32(n[2i]   * c) - RN32(n[2i+1] * s)))
 *   o[2i+1] = RN_bf16(RN32(RN32(n[2i+1] * c) + RN32(n[2i]   * s)))
 */
ORC_API void orc_rope_interleaved(const uint16_t *n, const float *cos_sin, int64_t D,
                                  uint16_t *o)
{
    for (int64_t i = 0; i < D / 2; ++i) {
        const float c = cos_sin[i], s = cos_sin[D / 2 + i];
        const float a = (float)orc_bf16_to_f64(n[2 * i]);
        const float b = (float)orc_bf16_to_f64(n[2 * i + 1]);
        const float ac = a * c, bs = b * s, bc = b * c, as = a * s;
        o[2 * i] = orc_bf16_from_f32(ac - bs);
        o[2 * i + 1] = orc_bf16_from_f32(bc + as);
    }
}

#define ORC_HEAD_DIM 128

/* One stream's Q or K head: RMSNorm then RoPE. */
static void qk_head(const uint16_t *x, const uint16_t *w, const float *cos_sin, float eps,
                    uint16_t *out)
{
    uint16_t n[ORC_HEAD_DIM];
    orc_rms_norm_head(x, w, ORC_HEAD_DIM, eps, n);
    orc_rope_interleaved(n, cos_sin, ORC_HEAD_DIM, out);
}

/*
 * The attention-input epilogue [QWEN-QKV implementation breakdown item 3; FLUX-QKV
 * implementation breakdown item 3]. Two streams (text, image), each with Q, K, V rows of
 * heads x 128 BF16 values at a row stride of ld elements (the packed GEMM output: Q, K, V
 * side by side), a cos/sin cache row per token ([tokens, 128] fp32: cos in 0..63, sin in
 * 64..127) and RMSNorm weights for Q and K ([128] BF16 each) and an eps. Output rows
 * [t_tokens + i_tokens, heads, 128], text first:
 *   joint_q[r, h] = RoPE(RMSNorm(q[h], wq), cache[r'])   (r' the token's row in its stream)
 *   joint_k[r, h] = RoPE(RMSNorm(k[h], wk), cache[r'])
 *   joint_v[r, h] = v[h]                                   (bit copy)
 */
ORC_API int orc_qkv_epilogue(uint16_t *jq, uint16_t *jk, uint16_t *jv,
                             const uint16_t *tq, const uint16_t *tk, const uint16_t *tv,
                             int64_t t_ld, int64_t t_tokens,
                             const uint16_t *iq, const uint16_t *ik, const uint16_t *iv,
                             int64_t i_ld, int64_t i_tokens,
                             const uint16_t *twq, const uint16_t *twk, const uint16_t *iwq,
                             const uint16_t *iwk, const float *t_cs, const float *i_cs,
                             int64_t heads, float t_eps, float i_eps)
{
    const int64_t D = ORC_HEAD_DIM, row = heads * D;
    for (int64_t r = 0; r < t_tokens + i_tokens; ++r) {
        const int txt = r < t_tokens;
        const int64_t rr = txt ? r : r - t_tokens;
        const int64_t ld = txt ? t_ld : i_ld;
        const uint16_t *q = (txt ? tq : iq) + rr * ld, *k = (txt ? tk : ik) + rr * ld,
                       *v = (txt ? tv : iv) + rr * ld;
        const uint16_t *wq = txt ? twq : iwq, *wk = txt ? twk : iwk;
        const float *cs = (txt ? t_cs : i_cs) + rr * D;
        const float eps = txt ? t_eps : i_eps;
        for (int64_t h = 0; h < heads; ++h) {
            qk_head(q + h * D, wq, cs, eps, jq + r * row + h * D);
            qk_head(k + h * D, wk, cs, eps, jk + r * row + h * D);
            memcpy(jv + r * row + h * D, v + h * D, D * sizeof(uint16_t));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Array forms of the scalar stages (same functions, looped; used by the pin tests)       */
/* ------------------------------------------------------------------------------------ */

ORC_API void orc_bf16_from_f32_n(const float *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_from_f32(v[i]);
}

ORC_API void orc_bf16_from_f64_n(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_from_f64(v[i]);
}

ORC_API void orc_e4m3_encode_n(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

ORC_API void orc_bf16_fma_n(const uint16_t *a, const uint16_t *b, const uint16_t *c,
                            uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_fma(a[i], b[i], c[i]);
}

ORC_API void orc_bf16_add_n(const uint16_t *a, const uint16_t *b, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_add(a[i], b[i]);
}

ORC_API void orc_quantize_n(const float *v, float inv, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_quantize(v[i], inv);
}

ORC_API void orc_e2m1_encode_n(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e2m1_encode(v[i]);
}
