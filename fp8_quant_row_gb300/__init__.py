"""fp8_quant_row_gb300: fused LayerNorm -> AdaLN modulate -> FP8 E4M3 row kernels for GB300.

Python binding of the C ABI in include/fp8q.h. This layer only marshals arguments: it checks
tensor dtypes/devices, allocates outputs with torch when the caller passes none, and calls
the library on the current torch CUDA stream. Every step of the computation runs in the
library's sm_103a kernels; there is no CPU or eager fallback.

    y, q = nss_fp8(x, scale, shift, input_scale)                      # q: float8_e4m3fn
    r, y, q = scale_residual_nss_fp8(x, residual, gate, scale, shift, input_scale, bias=b)
    y = bias_mul_add(x, bias, gate, residual)
    q = token_cat_fp8(attention, mlp, input_scale)
    q4, sf = token_cat_nvfp4(attention, mlp, global_scale)            # uint8 codes / scales
    jq, jk, jv = qkv_epilogue(txt, img, heads)      # per-head QK RMSNorm + RoPE, joint pack
    bits = device_error()                           # 0 unless a bounded kernel wait ran out
"""
from __future__ import annotations

import torch

from . import _capi
from ._build import build
from ._capi import Fp8qError

__all__ = ["nss_fp8", "scale_residual_nss_fp8", "bias_mul_add", "token_cat_fp8",
           "token_cat_nvfp4", "nvfp4_scale_bytes", "qkv_epilogue", "device_error",
           "row_pieces", "build",
           "Fp8qError", "library_path"]

EPS = 1e-6


def library_path() -> str:
    return _capi.LIB


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA bfloat16 tensor, got "
                        f"{t.dtype} on {t.device} (contiguous={t.is_contiguous()})")
    return t


def _scale_ptr(input_scale: torch.Tensor) -> int:
    if input_scale.dtype != torch.float32 or not input_scale.is_cuda or input_scale.numel() != 1:
        raise TypeError("input_scale: expected a one-element float32 CUDA tensor")
    return input_scale.data_ptr()


def _out(out, shape, dtype, like: torch.Tensor, name: str) -> torch.Tensor:
    if out is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    if out.dtype != dtype or tuple(out.shape) != tuple(shape) or not out.is_contiguous():
        raise TypeError(f"{name}: expected contiguous {dtype} {tuple(shape)}")
    return out


def _rows_cols(x: torch.Tensor):
    cols = x.shape[-1]
    return (x.numel() // cols if cols else 0), cols


def nss_fp8(x, scale, shift, input_scale, *, mod_rows: int = 0, eps: float = EPS, y=None,
            q=None, stream=None):
    """LayerNorm (no affine) -> modulate -> (bf16 y, float8_e4m3fn q). x: [..., cols]."""
    _bf16(x, "x"), _bf16(scale, "scale"), _bf16(shift, "shift")
    rows, cols = _rows_cols(x)
    y = _out(y, x.shape, torch.bfloat16, x, "y")
    q = _out(q, x.shape, torch.float8_e4m3fn, x, "q")
    st = _capi.lib().fp8q_nss_fp8(y.data_ptr(), q.data_ptr(), x.data_ptr(), scale.data_ptr(),
                                  shift.data_ptr(), int(mod_rows), _scale_ptr(input_scale),
                                  rows, cols, float(eps), _stream_handle(stream))
    _capi.check(st, "fp8q_nss_fp8")
    return y, q


def scale_residual_nss_fp8(x, residual, gate, scale, shift, input_scale, *, bias=None,
                           mod_rows: int = 0, eps: float = EPS, residual_out=None, y=None,
                           q=None, stream=None):
    """residual_out = RN(RN(x + bias) * gate + residual); (y, q) = nss_fp8(residual_out)."""
    for t, n in ((x, "x"), (residual, "residual"), (gate, "gate"), (scale, "scale"),
                 (shift, "shift")):
        _bf16(t, n)
    if bias is not None:
        _bf16(bias, "bias")
    rows, cols = _rows_cols(x)
    residual_out = _out(residual_out, x.shape, torch.bfloat16, x, "residual_out")
    y = _out(y, x.shape, torch.bfloat16, x, "y")
    q = _out(q, x.shape, torch.float8_e4m3fn, x, "q")
    st = _capi.lib().fp8q_scale_residual_nss_fp8(
        residual_out.data_ptr(), y.data_ptr(), q.data_ptr(), x.data_ptr(), residual.data_ptr(),
        None if bias is None else bias.data_ptr(), gate.data_ptr(), scale.data_ptr(),
        shift.data_ptr(), int(mod_rows), _scale_ptr(input_scale), rows, cols, float(eps),
        _stream_handle(stream))
    _capi.check(st, "fp8q_scale_residual_nss_fp8")
    return residual_out, y, q


def bias_mul_add(x, bias, gate, residual, *, y=None, stream=None):
    """y = RN(RN(x + bias) * gate + residual), the last rounding single (BF16 FMA)."""
    for t, n in ((x, "x"), (bias, "bias"), (gate, "gate"), (residual, "residual")):
        _bf16(t, n)
    rows, cols = _rows_cols(x)
    y = _out(y, x.shape, torch.bfloat16, x, "y")
    st = _capi.lib().fp8q_bias_mul_add(y.data_ptr(), x.data_ptr(), bias.data_ptr(),
                                       gate.data_ptr(), residual.data_ptr(), rows, cols,
                                       _stream_handle(stream))
    _capi.check(st, "fp8q_bias_mul_add")
    return y


def token_cat_fp8(a, m, input_scale, *, q=None, stream=None):
    """float8_e4m3fn q = E4M3(cat(a, m, dim=-1) * RN(1/input_scale)), no BF16 concat."""
    _bf16(a, "a"), _bf16(m, "m")
    rows, a_cols = _rows_cols(a)
    m_cols = m.shape[-1]
    if m.numel() != rows * m_cols:
        raise TypeError("a and m must have the same number of rows")
    q = _out(q, (*a.shape[:-1], a_cols + m_cols), torch.float8_e4m3fn, a, "q")
    st = _capi.lib().fp8q_token_cat_fp8(q.data_ptr(), a.data_ptr(), a_cols, m.data_ptr(),
                                        m_cols, _scale_ptr(input_scale), rows,
                                        _stream_handle(stream))
    _capi.check(st, "fp8q_token_cat_fp8")
    return q


def nvfp4_scale_bytes(rows: int, cols: int) -> int:
    """Size of the padded 128x4-tiled block-scale buffer for a [rows, cols] NVFP4 tensor."""
    n = _capi.lib().fp8q_nvfp4_scale_bytes(int(rows), int(cols))
    if n < 0:
        raise ValueError(f"no NVFP4 layout for rows={rows}, cols={cols}")
    return n


def token_cat_nvfp4(a, m, global_scale, *, q=None, sf=None, stream=None):
    """NVFP4 of cat(a, m, dim=-1) without a BF16 concat: (q, sf), both uint8.

    q [..., (a_cols + m_cols) / 2] holds two E2M1 codes per byte (first element in the low
    nibble); sf is the flat 128x4-tiled E4M3 block-scale buffer (nvfp4_scale_bytes bytes,
    padding rows zero). global_scale: one-element float32 CUDA tensor (input_scale_inv)."""
    _bf16(a, "a"), _bf16(m, "m")
    rows, a_cols = _rows_cols(a)
    m_cols = m.shape[-1]
    if m.numel() != rows * m_cols:
        raise TypeError("a and m must have the same number of rows")
    cols = a_cols + m_cols
    q = _out(q, (*a.shape[:-1], cols // 2), torch.uint8, a, "q")
    n_sf = _capi.lib().fp8q_nvfp4_scale_bytes(rows, cols)
    sf = _out(sf, (max(n_sf, 0),), torch.uint8, a, "sf")
    st = _capi.lib().fp8q_token_cat_nvfp4(q.data_ptr(), sf.data_ptr(), a.data_ptr(), a_cols,
                                          m.data_ptr(), m_cols, _scale_ptr(global_scale), rows,
                                          _stream_handle(stream))
    _capi.check(st, "fp8q_token_cat_nvfp4")
    return q, sf


HEAD_DIM = 128


def _qkv_stream(st: dict, heads: int) -> "_capi.QkvStream":
    q, k, v = st["q"], st["k"], st["v"]
    tokens = q.shape[0]
    if tokens == 0:  # an empty stream: nothing is read from it
        return _capi.QkvStream(None, None, None, heads * HEAD_DIM, 0, None, None, None,
                               float(st.get("eps", EPS)))
    for name in ("q", "k", "v"):
        t = st[name]
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise TypeError(f"{name}: expected a 2-D CUDA bfloat16 tensor with unit column stride")
        if t.shape[0] != tokens or t.shape[1] < heads * HEAD_DIM or t.stride(0) != q.stride(0):
            raise TypeError(f"{name}: rows, width or row stride differ from q")
    for name in ("q_weight", "k_weight"):
        _bf16(st[name], name)
        if st[name].numel() != HEAD_DIM:
            raise TypeError(f"{name}: expected {HEAD_DIM} values")
    cs = st["cos_sin"]
    if cs.dtype != torch.float32 or not cs.is_cuda or not cs.is_contiguous() or \
            tuple(cs.shape) != (tokens, HEAD_DIM):
        raise TypeError(f"cos_sin: expected a contiguous CUDA float32 [{tokens}, {HEAD_DIM}]")
    return _capi.QkvStream(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.stride(0), tokens,
                           st["q_weight"].data_ptr(), st["k_weight"].data_ptr(), cs.data_ptr(),
                           float(st.get("eps", EPS)))


def qkv_epilogue(txt: dict, img: dict, heads: int, *, out=None, stream=None):
    """Attention inputs after the packed QKV GEMM: returns joint (q, k, v), each bfloat16
    [txt_tokens + img_tokens, heads, 128], text first. Per head of q and k: RMSNorm with the
    stream's weight and eps, then interleaved RoPE with the stream's fp32 cos/sin cache; v is
    copied. `txt` / `img`: dicts with q, k, v (2-D views of the GEMM output, e.g. column
    slices of one [tokens, 3*heads*128] tensor), q_weight, k_weight, cos_sin and eps."""
    ts, ims = _qkv_stream(txt, heads), _qkv_stream(img, heads)
    total = ts.tokens + ims.tokens
    like = txt["q"]
    if out is None:
        out = tuple(torch.empty(total, heads, HEAD_DIM, dtype=torch.bfloat16, device=like.device)
                    for _ in range(3))
    for t in out:
        _out(t, (total, heads, HEAD_DIM), torch.bfloat16, like, "out")
    st = _capi.lib().fp8q_qkv_epilogue(out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
                                       ts, ims, heads, _stream_handle(stream))
    _capi.check(st, "fp8q_qkv_epilogue")
    return out


def device_error() -> int:
    """Reads and clears the current device's error word (fp8q_device_error): 0 unless a
    bounded wait inside a kernel ran out since the last call. Synchronises with the device."""
    import ctypes
    bits = ctypes.c_uint(0)
    _capi.check(_capi.lib().fp8q_device_error(ctypes.byref(bits)), "fp8q_device_error")
    return int(bits.value)


def row_pieces(rows: int, mod_rows: int, world: int, rank: int):
    """The pieces of rank `rank`'s share when `rows` rows are split over `world` processes:
    a list of (r0, r1, group). The rows are cut into `world` contiguous slices of near-equal
    size (the first rows % world slices one row longer), and a slice is cut again wherever
    it crosses a modulation-group boundary (a multiple of mod_rows), so every piece lies in
    one group. Each piece is one call on x[r0:r1] with mod_rows = 0 and the scale/shift (and
    gate) rows of `group` (0 when mod_rows is 0). Rows are independent, so the pieces of all
    ranks together give exactly the single call's outputs; no data is exchanged."""
    if rows < 0 or mod_rows < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("row_pieces: need rows >= 0, mod_rows >= 0, 0 <= rank < world")
    base, extra = divmod(rows, world)
    r0 = rank * base + min(rank, extra)
    r1 = r0 + base + (1 if rank < extra else 0)
    pieces = []
    while r0 < r1:
        if mod_rows:
            g = r0 // mod_rows
            end = min(r1, (g + 1) * mod_rows)
        else:
            g, end = 0, r1
        pieces.append((r0, end, g))
        r0 = end
    return pieces
