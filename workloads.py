"""Seeded synthetic inputs for the fused LayerNorm -> modulate -> FP8 row path.

This module only draws random numbers and casts them to bf16 host arrays; it holds none of
the method's arithmetic. The same host bytes feed both the CPU oracle and the CUDA path.

Every draw uses ``torch.Generator('cpu').manual_seed(seed)``: values are drawn in fp32,
scaled, then cast to bf16 (round-to-nearest-even) by torch. Arrays are returned as numpy
``uint16`` bit patterns (row-major, contiguous).

Workload shapes follow the pages' models: Qwen-Image hidden size 3072 with 4096 image + 512
text tokens, FLUX.2 attention width 6144 and SwiGLU width 18432 (4608 tokens per sample).
No model weights or datasets exist here; these synthetic draws stand in for the activations
of those checkpoints.
"""
from __future__ import annotations

import numpy as np
import torch

EPS = 1e-6

#: Real checkpoint input scale printed in the review notes of "sglang #37156 - Qwen-Image
#: FP8 norm + activation-quant fusion" (midpoint-sensitive under a 1-ulp reciprocal change).
QWEN_CHECKPOINT_INPUT_SCALE = 0.4754464328

#: The five input scales of the Qwen-Image sweep: the checkpoint value, two powers of two
#: (y / s then lands exactly on E4M3 rounding midpoints for ~1/16 of normal-range values),
#: and two generic values.
QWEN_INPUT_SCALES = (QWEN_CHECKPOINT_INPUT_SCALE, 0.0625, 0.25, 0.05, 0.0123)

CONFIGS = {
    "nss_tiny": dict(op="nss_fp8", rows=127, cols=3072, input_scale=0.0123, seed=0),
    "nss_qwen": dict(op="nss_fp8", rows=4608, cols=3072, input_scale=QWEN_CHECKPOINT_INPUT_SCALE,
                     input_scales=QWEN_INPUT_SCALES, rows_sweep=(1, 127, 1024), seed=0,
                     outlier_channels=30, outlier_gain=20.0),
    "scale_residual_qwen": dict(op="scale_residual_nss_fp8", rows=4096, cols=3072,
                                input_scale=0.05, seed=0),
    "bias_mul_add_qwen": dict(op="bias_mul_add", rows=4096, cols=3072, seed=0),
    "nss_flux": dict(op="nss_fp8", rows=9216, cols=6144, n_samples=2, mod_rows=4608,
                     input_scale=0.02, seed=0),
    "token_cat_flux": dict(op="token_cat_fp8", rows=4608, a_cols=6144, m_cols=18432,
                           input_scale=0.1, seed=0),
    # Same activations quantised to NVFP4; global scale = 448 * 6 / 44.8, the amax that the
    # FP8 configuration's input_scale 0.1 stands for.
    "token_cat_nvfp4_flux": dict(op="token_cat_nvfp4", rows=4608, a_cols=6144, m_cols=18432,
                                 global_scale=60.0, seed=0),
    # Attention-input epilogue after the packed QKV GEMM: 1024x1024 image -> 64x64 = 4096
    # image tokens; text tokens 256 (Qwen-Image) / 512 (FLUX.2); head_dim 128.
    "qkv_qwen": dict(op="qkv_epilogue", txt_tokens=256, img_tokens=4096, heads=24, eps=1e-6,
                     seed=0),
    "qkv_flux": dict(op="qkv_epilogue", txt_tokens=512, img_tokens=4096, heads=48, eps=1e-6,
                     seed=1),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def to_bf16_bits(t: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> bf16 (RNE, by torch) -> numpy uint16 bit patterns."""
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def normal_bf16(shape, std: float, g: torch.Generator) -> np.ndarray:
    return to_bf16_bits(torch.randn(*shape, generator=g, dtype=torch.float32) * std)


def nss_inputs(rows: int, cols: int, seed: int = 0, n_mod: int = 1, outlier_channels: int = 0,
               outlier_gain: float = 20.0, x_std: float = 1.0, mod_std: float = 0.1):
    """x [rows, cols] ~ N(0, x_std) (optional outlier channels x gain), scale/shift
    [n_mod, cols] ~ N(0, mod_std)."""
    g = _gen(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32) * x_std
    if outlier_channels:
        ch = torch.randperm(cols, generator=g)[:outlier_channels]
        x[:, ch] *= outlier_gain
    scale = torch.randn(n_mod, cols, generator=g, dtype=torch.float32) * mod_std
    shift = torch.randn(n_mod, cols, generator=g, dtype=torch.float32) * mod_std
    return dict(x=to_bf16_bits(x), scale=to_bf16_bits(scale), shift=to_bf16_bits(shift))


def residual_inputs(rows: int, cols: int, seed: int = 0, n_mod: int = 1):
    """x, residual [rows, cols] ~ N(0,1); bias [cols] ~ N(0, 0.05); gate/scale/shift
    [n_mod, cols] ~ N(0, 0.1)."""
    g = _gen(seed)
    x = normal_bf16((rows, cols), 1.0, g)
    residual = normal_bf16((rows, cols), 1.0, g)
    bias = normal_bf16((cols,), 0.05, g)
    gate = normal_bf16((n_mod, cols), 0.1, g)
    scale = normal_bf16((n_mod, cols), 0.1, g)
    shift = normal_bf16((n_mod, cols), 0.1, g)
    return dict(x=x, residual=residual, bias=bias, gate=gate, scale=scale, shift=shift)


def token_cat_inputs(rows: int, a_cols: int = 6144, m_cols: int = 18432, seed: int = 0,
                     tail_prob: float = 0.001, tail_gain: float = 50.0):
    """attention a [rows, a_cols] ~ N(0,1); SwiGLU m [rows, m_cols] ~ N(0, 0.5) with a
    heavy tail: entries with probability tail_prob are multiplied by tail_gain."""
    g = _gen(seed)
    a = torch.randn(rows, a_cols, generator=g, dtype=torch.float32)
    m = torch.randn(rows, m_cols, generator=g, dtype=torch.float32) * 0.5
    mask = torch.rand(rows, m_cols, generator=g) < tail_prob
    m[mask] *= tail_gain
    return dict(a=to_bf16_bits(a), m=to_bf16_bits(m))


def rope_cache(positions: np.ndarray, head_dim: int = 128, theta: float = 10000.0) -> np.ndarray:
    """fp32 [tokens, head_dim] cache rows (cos of the head_dim/2 pair angles, then sin).
    positions: [tokens, head_dim/2] position index used by each pair."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    ang = positions.astype(np.float64) * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def qkv_inputs(txt_tokens: int, img_tokens: int, heads: int, seed: int = 0, eps: float = 1e-6,
               head_dim: int = 128, extra_cols: int = 0):
    """Two streams of packed QKV GEMM output, [tokens, 3*heads*head_dim (+extra_cols)] BF16
    (q | k | v side by side). q, k ~ N(0,1) times a per-channel gain exp(N(0, 0.5)) shared by
    all heads (trained projections have uneven channels); v ~ N(0,1). RMSNorm weights ~
    N(1, 0.3). cos/sin caches: text token t uses position t for every pair; image token
    (y, x) of a square grid uses y for the first half of the pairs and x for the second."""
    g = _gen(seed)
    out = {}
    side = int(round(img_tokens ** 0.5))
    for name, n in (("txt", txt_tokens), ("img", img_tokens)):
        width = 3 * heads * head_dim + extra_cols
        gain = torch.exp(torch.randn(head_dim, generator=g) * 0.5)
        qk = torch.randn(n, 2, heads, head_dim, generator=g) * gain
        v = torch.randn(n, heads * head_dim, generator=g)
        packed = torch.cat([qk.reshape(n, 2 * heads * head_dim), v,
                            torch.randn(n, extra_cols, generator=g)], dim=1)
        assert packed.shape[1] == width
        bits = to_bf16_bits(packed)
        hd = heads * head_dim
        if name == "txt" or side * side != n:
            pos = np.repeat(np.arange(n)[:, None], head_dim // 2, axis=1)
        else:
            yy, xx = np.divmod(np.arange(n), side)
            pos = np.concatenate([np.repeat(yy[:, None], head_dim // 4, axis=1),
                                  np.repeat(xx[:, None], head_dim // 4, axis=1)], axis=1)
        out[name] = dict(packed=bits, q=bits[:, :hd], k=bits[:, hd:2 * hd], v=bits[:, 2 * hd:3 * hd],
                         ld=width,
                         wq=to_bf16_bits(1.0 + 0.3 * torch.randn(head_dim, generator=g)),
                         wk=to_bf16_bits(1.0 + 0.3 * torch.randn(head_dim, generator=g)),
                         cos_sin=rope_cache(pos, head_dim), eps=eps)
    return out


def config_inputs(name: str, rows: int | None = None, seed: int | None = None):
    """Inputs of a named configuration (optionally with fewer rows / another seed)."""
    c = CONFIGS[name]
    r = c.get("rows") if rows is None else rows
    s = c["seed"] if seed is None else seed
    if c["op"] == "nss_fp8":
        n_mod = c.get("n_samples", 1)
        return nss_inputs(r, c["cols"], seed=s, n_mod=n_mod,
                          outlier_channels=c.get("outlier_channels", 0),
                          outlier_gain=c.get("outlier_gain", 20.0))
    if c["op"] in ("scale_residual_nss_fp8", "bias_mul_add"):
        return residual_inputs(r, c["cols"], seed=s)
    if c["op"] in ("token_cat_fp8", "token_cat_nvfp4"):
        return token_cat_inputs(r, c["a_cols"], c["m_cols"], seed=s)
    if c["op"] == "qkv_epilogue":
        return qkv_inputs(c["txt_tokens"], c["img_tokens"], c["heads"], seed=s, eps=c["eps"])
    raise KeyError(name)
