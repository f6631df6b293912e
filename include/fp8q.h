/*
 * fp8q.h -- C ABI of libfp8q: fused row kernels for the DiT-block prologue on GB300 (sm_103a).
 *
 *   nss_fp8                 LayerNorm (no affine) -> AdaLN modulate -> dual output:
 *                           BF16 y and its static per-tensor FP8 E4M3 quantisation q.
 *   scale_residual_nss_fp8  gated residual update (optional input bias), then nss_fp8.
 *   bias_mul_add            deferred output-bias epilogue y = (x + bias) * gate + residual.
 *   token_cat_fp8           E4M3 quantisation of the row concat [a | m] without a BF16 concat.
 *   token_cat_nvfp4         NVFP4 quantisation (E2M1 codes + 128x4-tiled E4M3 block scales)
 *                           of the same row concat.
 *   qkv_epilogue            after the packed QKV GEMM: per-head Q/K RMSNorm + interleaved RoPE,
 *                           V copy, joint [text, image] attention inputs.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers to row-major, contiguous arrays on the current
 *     CUDA device. bf16 tensors are raw bfloat16 bits (uint16); E4M3 tensors are raw
 *     e4m3fn codes (uint8: no infinities, 0x7F/0xFF NaN, largest finite 448).
 *   - The caller owns every buffer. The library allocates nothing, never synchronises and
 *     only enqueues work on `stream` (0 = the legacy default stream). Outputs are complete
 *     when that stream reaches the launch.
 *   - Every tensor pointer must be 16-byte aligned (FP8Q_ERR_ALIGN otherwise); the NVFP4
 *     and QKV entry points need 32 bytes for their data pointers (see each call).
 *   - rows == 0 returns FP8Q_OK without touching any pointer or launching anything.
 *   - Argument errors are reported synchronously, before any launch, with a status code; a
 *     failed launch returns FP8Q_ERR_CUDA (fp8q_last_cuda_error() gives the cudaError_t).
 *   - input_scale is a device pointer to ONE fp32 value; it must be finite and > 0. That
 *     precondition is not checked (checking would need a device-to-host copy and a sync).
 *     The kernels use inv = RN_fp32(1 / *input_scale), a correctly rounded fp32 division.
 *   - Encode rule: q = E4M3(RN_fp32(v * inv)), saturating (|.| >= 448 -> +-448),
 *     round-to-nearest-even; NaN gives 0x7F.
 *   - Only compute capability 10.3 (GB300) is supported (FP8Q_ERR_UNSUPPORTED otherwise).
 *
 * Sources (page title and section):
 *   [QWEN-NQ]   "sglang #37156 - Qwen-Image FP8 norm + activation-quant fusion":
 *               implementation breakdown items 1-2, key source snippets (norm_scale_shift.cuh,
 *               norm_scale_shift_jit.py).
 *   [QWEN-BIAS] "sglang #37116 - Qwen-Image output-bias deferral": implementation breakdown
 *               item 3, key source snippets (bias_mul_add_kernel), review highlights.
 *   [FLUX-FP8]  "sglang #37162 - FLUX.2 FP8 LayerNorm/quant/QKV fusions": implementation
 *               breakdown items 2 and 4, key source snippets (_token_cat_fp8_kernel).
 *   [FLUX-FP4]  "sglang #37141 - FLUX.2 token-cat + NVFP4 fusion": features and motivation
 *               (attention 6144 + MLP 18432 -> NVFP4 without the concat), implementation
 *               breakdown items 1-3 (per-group conversion, 128x4-swizzled scale offsets,
 *               input_scale_inv as the global scale, 32-byte aligned dense BF16 inputs).
 *   [QWEN-QKV]  "sglang #37123 - Qwen-Image FP8 QKV fusion": implementation breakdown item 3
 *               (Q/K RMSNorm + RoPE, V copy, joint [text, image] output, head_dim 128, 32-byte
 *               aligned strided views of the packed GEMM output), key source snippets
 *               (per-stream norm weights, epsilons and cos/sin caches; is_neox=False).
 *   [FLUX-QKV]  "sglang #37162 - FLUX.2 FP8 LayerNorm/quant/QKV fusions": implementation
 *               breakdown item 3 (QK RMSNorm, RoPE, QKV pack, text/image concat).
 *   [NVFP4]     the public NVFP4 format: E2M1 elements, one E4M3 scale per 16 consecutive
 *               elements of a row, an fp32 per-tensor scale; 128x4 scale tiles of FP4 GEMMs.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8q_status {
    FP8Q_OK = 0,
    FP8Q_ERR_NULL = 1,        /* a required pointer is NULL (with rows > 0)                   */
    FP8Q_ERR_ALIGN = 2,       /* a tensor pointer is not 16-byte aligned (32 where stated)    */
    FP8Q_ERR_SHAPE = 3,       /* rows < 0, unsupported cols / a_cols / m_cols, mod_rows < 0   */
    FP8Q_ERR_UNSUPPORTED = 4, /* current device is not compute capability 10.3                */
    FP8Q_ERR_ALIAS = 5,       /* an output overlaps an input or another output (see per call) */
    FP8Q_ERR_CUDA = 6,        /* a CUDA runtime query or the kernel launch failed             */
    FP8Q_ERR_VALUE = 7        /* a scalar argument is out of range (eps < 0 or not finite)    */
} fp8q_status;

/*
 * LayerNorm -> modulate -> dual BF16 + E4M3 output, one row at a time [QWEN-NQ].
 *
 *   mu = mean(x[r,:]), var = mean((x[r,:] - mu)^2)       (population variance, no affine)
 *   n  = RN_bf16((x - mu) / sqrt(var + eps))             (normalised value, BF16-rounded)
 *   y  = RN_bf16(fma_fp32(n, RN_fp32(1 + scale[m,:]), shift[m,:]))     m = r / mod_rows
 *   q  = E4M3(RN_fp32(y * inv))
 *
 *   y_bf16      out  [rows, cols] bf16
 *   q_e4m3      out  [rows, cols] e4m3 codes
 *   x_bf16      in   [rows, cols] bf16
 *   scale_bf16  in   [n_mod, cols] bf16, n_mod = mod_rows ? ceil(rows / mod_rows) : 1
 *   shift_bf16  in   [n_mod, cols] bf16
 *   mod_rows    rows that share one scale/shift row (per-sample modulation); 0 = one row
 *               broadcast over all rows
 *   input_scale in   device pointer to one fp32 (finite, > 0)
 *   cols        multiple of 8, 8 <= cols <= 32768 (3072 and 6144 take the tuned path)
 *   eps         >= 0 and finite (1e-6 on the pages)
 *   Aliasing: no output may overlap any input or the other output (FP8Q_ERR_ALIAS).
 *   Value range: x must be finite with |x| < 2^56. The row sums (of x and of x^2) are kept in
 *   fp32-range double-float arithmetic, so larger magnitudes may overflow them; rows holding
 *   Inf or NaN, or values at or above 2^56, give unspecified y and q (no error is reported:
 *   checking would cost a pass over the data). With eps = 0 a row whose squares all underflow
 *   fp32 (|x| below about 1e-19) is also outside the contract.
 *   The row sums are formed error-free except for an fp32 sum of per-element rounding
 *   errors: the mean comes out exact on the workload rows and the variance within about
 *   2^-43 * (max|x| / sigma)^2 relative. Each normalised value is rounded to BF16 as the exact
 *   value would be, except when that value lies within about that relative distance of a
 *   BF16 rounding midpoint.
 *   Row slices (one call per GPU or per piece of a larger tensor): the modulation row of data
 *   row r is r / mod_rows counted from the call's own first row. A piece of rows [r0, r1)
 *   of a larger tensor is therefore passed as x + r0*cols with mod_rows = 0 and scale/shift
 *   pointing at the row of its modulation group, g = r0 / mod_rows, and every piece must lie
 *   inside one group (split a slice at multiples of mod_rows); the binding's row_pieces()
 *   makes such pieces.
 */
fp8q_status fp8q_nss_fp8(void* y_bf16, uint8_t* q_e4m3, const void* x_bf16,
                         const void* scale_bf16, const void* shift_bf16, int64_t mod_rows,
                         const float* input_scale, int64_t rows, int64_t cols, float eps,
                         cudaStream_t stream);

/*
 * Gated scale-residual with optional input bias, then nss_fp8 on the updated residual
 * [QWEN-NQ implementation breakdown item 1; QWEN-BIAS implementation breakdown item 3].
 *
 *   xb           = bias ? RN_bf16(x + bias) : x
 *   residual_out = RN_bf16(xb * gate[m,:] + residual)     (single rounding, BF16 FMA)
 *   (y, q)       = nss_fp8(residual_out, scale, shift, ...)
 *
 *   residual_out out [rows, cols] bf16; may be exactly the residual buffer (in-place update)
 *   y, q         out as in fp8q_nss_fp8
 *   x, residual  in  [rows, cols] bf16
 *   bias         in  [cols] bf16 or NULL (no input bias)
 *   gate, scale, shift in [n_mod, cols] bf16 (m = r / mod_rows as above)
 *   Aliasing: residual_out may equal residual exactly; every other overlap is rejected.
 *   Value range and row slices: as for fp8q_nss_fp8 (x, residual and the updated residual
 *   finite with magnitudes below 2^56; pieces inside one modulation group, gate offset like
 *   scale and shift).
 */
fp8q_status fp8q_scale_residual_nss_fp8(void* residual_out, void* y_bf16, uint8_t* q_e4m3,
                                        const void* x_bf16, const void* residual_bf16,
                                        const void* bias_bf16, const void* gate_bf16,
                                        const void* scale_bf16, const void* shift_bf16,
                                        int64_t mod_rows, const float* input_scale,
                                        int64_t rows, int64_t cols, float eps,
                                        cudaStream_t stream);

/*
 * Deferred output-bias epilogue [QWEN-BIAS key source snippets]:
 *   y = RN_bf16(RN_bf16(x + bias) * gate + residual), the second rounding single (BF16 FMA).
 *
 *   y        out [rows, cols] bf16; may equal x or residual exactly (elementwise in place)
 *   x        in  [rows, cols] bf16
 *   bias     in  [cols] bf16
 *   gate     in  [cols] bf16
 *   residual in  [rows, cols] bf16
 *   cols     multiple of 8, >= 8
 */
fp8q_status fp8q_bias_mul_add(void* y_bf16, const void* x_bf16, const void* bias_bf16,
                              const void* gate_bf16, const void* residual_bf16, int64_t rows,
                              int64_t cols, cudaStream_t stream);

/*
 * Token concat -> E4M3 [FLUX-FP8 implementation breakdown item 4, key source snippets]:
 *   q[r, c] = E4M3(RN_fp32(v * inv)),  v = a[r, c] (c < a_cols) else m[r, c - a_cols].
 * The BF16 concat [a | m] is never materialised.
 *
 *   q       out [rows, a_cols + m_cols] e4m3 codes (row stride a_cols + m_cols)
 *   a       in  [rows, a_cols] bf16 (attention output, 6144 wide on FLUX.2)
 *   m       in  [rows, m_cols] bf16 (SwiGLU output, 18432 wide on FLUX.2)
 *   a_cols, m_cols  multiples of 16, >= 16
 *   Aliasing: q may not overlap a or m.
 */
fp8q_status fp8q_token_cat_fp8(uint8_t* q_e4m3, const void* a_bf16, int64_t a_cols,
                               const void* m_bf16, int64_t m_cols, const float* input_scale,
                               int64_t rows, cudaStream_t stream);

/*
 * Token-concat -> NVFP4 [FLUX-FP4; NVFP4]: row r of cat(a, m) is quantised in 16-element
 * groups straight from the two sources (no BF16 concat). Per group, in IEEE fp32 with every
 * operation rounded to nearest even:
 *   amax = max |x_i|
 *   sf   = E4M3_satfinite(RN(g * RN(amax * RN(1/6))))                 (stored block scale)
 *   out  = sf == +-0 ? 0 : RN(1 / RN(E4M3(sf) * RN(1/g)))
 *   e_i  = E2M1_satfinite(RN(x_i * out))          E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6
 * so E2M1(e_i) * E4M3(sf) / g approximates x_i. g = *global_scale (the consuming GEMM's
 * input_scale_inv; finite and > 0, not checked). Sign of a zero result follows x_i * out.
 *
 *   q_fp4        out  [rows, (a_cols + m_cols) / 2] bytes; byte j of a row holds element 2j in
 *                     bits 0..3 and element 2j+1 in bits 4..7
 *   sf_e4m3      out  fp8q_nvfp4_scale_bytes(rows, a_cols + m_cols) bytes: block scale of
 *                     (row r, group k) of K = cols/16 groups at byte
 *                       ((r / 128) * ceil(K / 4) + k / 4) * 512
 *                       + (r % 32) * 16 + ((r % 128) / 32) * 4 + k % 4
 *                     (128-row x 4-group tiles of 512 bytes); entries of padding rows
 *                     (rows .. ceil(rows/128)*128 - 1) are written with 0
 *   a_bf16       in   [rows, a_cols] bf16 (attention part)
 *   m_bf16       in   [rows, m_cols] bf16 (MLP part)
 *   a_cols, m_cols    multiples of 64, >= 64 (FLUX.2: 6144 and 18432)
 *   global_scale in   device pointer to one fp32
 *   Alignment: q_fp4, a_bf16, m_bf16 32-byte aligned; sf_e4m3 16-byte aligned.
 *   Aliasing: q_fp4, sf_e4m3, a_bf16, m_bf16 and global_scale pairwise disjoint.
 *   Inputs containing NaN give unspecified codes in their group (no NaN in E2M1).
 */
fp8q_status fp8q_token_cat_nvfp4(uint8_t* q_fp4, uint8_t* sf_e4m3, const void* a_bf16,
                                 int64_t a_cols, const void* m_bf16, int64_t m_cols,
                                 const float* global_scale, int64_t rows, cudaStream_t stream);

/* Bytes of the padded block-scale buffer of fp8q_token_cat_nvfp4 for a [rows, cols] input:
 * ceil(rows/128)*128 * ceil(cols/64)*4. -1 for rows < 0 or cols not a positive multiple of 16.
 * Host-only arithmetic. */
int64_t fp8q_nvfp4_scale_bytes(int64_t rows, int64_t cols);

/* One input stream of fp8q_qkv_epilogue (all pointers device pointers, 32-byte aligned). */
typedef struct fp8q_qkv_stream {
    const void* q;         /* [tokens, ld] bf16; head h at values h*128 .. h*128+127        */
    const void* k;         /* same layout (the packed GEMM output: q, k, v side by side)    */
    const void* v;
    int64_t ld;            /* row stride in values: >= heads*128, a multiple of 16           */
    int64_t tokens;        /* rows of this stream (0 allowed: nothing read)                  */
    const void* q_weight;  /* [128] bf16 RMSNorm weight of Q                                 */
    const void* k_weight;  /* [128] bf16 RMSNorm weight of K                                 */
    const float* cos_sin;  /* [tokens, 128] fp32 RoPE cache: cos of pair i at i, sin at 64+i  */
    float eps;             /* RMSNorm epsilon, finite and > 0 (FP8Q_ERR_VALUE otherwise)     */
} fp8q_qkv_stream;

/*
 * Attention-input epilogue after the packed QKV GEMM [QWEN-QKV; FLUX-QKV], head_dim 128.
 * Joint row r < txt->tokens comes from text row r, the others from image row r - txt->tokens.
 * For every head h of a row (x = that head's 128 values of q or k, w the stream's weight):
 *   n_j    = RN_bf16(x_j * w_j / sqrt(sum_i x_i^2 / 128 + eps))        one rounding of the
 *                                                                       exact value
 *   o[2i]   = RN_bf16(RN32(RN32(n[2i] c_i) - RN32(n[2i+1] s_i)))        interleaved RoPE with
 *   o[2i+1] = RN_bf16(RN32(RN32(n[2i+1] c_i) + RN32(n[2i] s_i)))        c_i = cos_sin[row][i],
 *                                                                       s_i = cos_sin[row][64+i]
 *   joint_q[r, h, :] = o(q),  joint_k[r, h, :] = o(k),  joint_v[r, h, :] = v (bit copy)
 *
 *   joint_q, joint_k, joint_v  out  [txt->tokens + img->tokens, heads, 128] bf16, contiguous,
 *                                   32-byte aligned
 *   heads       1 .. 4096
 *   Aliasing: the three outputs are disjoint from each other and from every input.
 *   Values must be finite with |x| < 2^56; a head whose values are all below 2^-40 is
 *   normalised with eps dominating (its squares are not summed exactly).
 */
fp8q_status fp8q_qkv_epilogue(void* joint_q, void* joint_k, void* joint_v,
                              const fp8q_qkv_stream* txt, const fp8q_qkv_stream* img,
                              int64_t heads, cudaStream_t stream);

/* Bits of the device error word (fp8q_device_error). */
#define FP8Q_DEVERR_WAIT_TIMEOUT 1u /* a kernel gave up on a bounded shared-memory wait */

/*
 * Reads and clears the device error word of the current device. Every wait inside the
 * library's kernels is bounded (about two seconds of SM clock); a wait that runs out sets
 * FP8Q_DEVERR_WAIT_TIMEOUT, and the kernel stops taking work and returns with its outputs
 * incomplete. Only a defect can cause this: every phase a kernel waits for is completed by
 * the same CTA (a bulk copy landing, or another warp's arrival), never by the host or another
 * kernel. Diagnostic call, not for the hot path: it synchronises with the device
 * (cudaMemcpyFromSymbol) and is not capturable in a CUDA graph.
 *   bits  out  host pointer; receives the word (0: no wait ran out since the last call)
 */
fp8q_status fp8q_device_error(unsigned int* bits);

/* Human-readable name of a status code (static string; never NULL). */
const char* fp8q_status_string(int status);

/* cudaError_t of the last FP8Q_ERR_CUDA returned on the calling host thread (0 if none). */
int fp8q_last_cuda_error(void);

/* Which runtime call produced that error, e.g. "cudaLaunchKernel(98560): cudaErrorInvalidValue"
 * (thread-local static string, "" if none; overwritten by the next failure). */
const char* fp8q_last_error_detail(void);

/* Library ABI version: 0x00MMmmpp (0.2.0: token_cat_nvfp4 and qkv_epilogue added; 0.3.0:
 * fp8q_device_error added). */
int fp8q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
