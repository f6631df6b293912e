"""CPU oracle for the fused LayerNorm -> modulate -> FP8 E4M3 row path (test infrastructure).

This package is the correctness reference, and nothing else: only ``tests/``, the
``__graft_entry__.smoke()`` check and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import it. The CUDA product path neither imports nor links it, and the two
share no code.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp64 where the pages leave the
precision open); this module compiles it with gcc on first use and wraps it with ctypes over
numpy arrays. bf16 tensors are passed as ``numpy.uint16`` bit patterns and E4M3 tensors as
``numpy.uint8`` codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fvisibility=hidden", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc; no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        f32 = ctypes.c_float
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        lib.orc_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.orc_bf16_from_f64.restype = ctypes.c_uint16
        lib.orc_bf16_from_f32.argtypes = [f32]
        lib.orc_bf16_from_f32.restype = ctypes.c_uint16
        lib.orc_bf16_fma.argtypes = [ctypes.c_uint16] * 3
        lib.orc_bf16_fma.restype = ctypes.c_uint16
        lib.orc_bf16_add.argtypes = [ctypes.c_uint16] * 2
        lib.orc_bf16_add.restype = ctypes.c_uint16
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_encode.argtypes = [f32]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_recip_f32.argtypes = [f32]
        lib.orc_recip_f32.restype = f32
        lib.orc_quantize.argtypes = [f32, f32]
        lib.orc_quantize.restype = ctypes.c_uint8
        lib.orc_modulate.argtypes = [ctypes.c_uint16] * 3
        lib.orc_modulate.restype = ctypes.c_uint16
        lib.orc_ln_row_t.argtypes = [u16p, i64, f32, f64p]
        lib.orc_ln_row_t.restype = None
        lib.orc_nss_fp8.argtypes = [u16p, u8p, u16p, u16p, u16p, i64, f32, i64, i64, f32, f64p]
        lib.orc_nss_fp8.restype = ctypes.c_int
        lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e2m1_decode.restype = ctypes.c_double
        lib.orc_e2m1_encode.argtypes = [f32]
        lib.orc_e2m1_encode.restype = ctypes.c_uint8
        lib.orc_e2m1_encode_n.argtypes = [ctypes.POINTER(f32), u8p, i64]
        lib.orc_e2m1_encode_n.restype = None
        lib.orc_nvfp4_group.argtypes = [u16p, f32, u8p]
        lib.orc_nvfp4_group.restype = ctypes.c_uint8
        lib.orc_nvfp4_sf_offset.argtypes = [i64, i64, i64]
        lib.orc_nvfp4_sf_offset.restype = i64
        lib.orc_token_cat_nvfp4.argtypes = [u8p, u8p, u16p, i64, u16p, i64, f32, i64]
        lib.orc_token_cat_nvfp4.restype = ctypes.c_int
        f32p = ctypes.POINTER(f32)
        lib.orc_rms_norm_head.argtypes = [u16p, u16p, i64, f32, u16p]
        lib.orc_rms_norm_head.restype = None
        lib.orc_rope_interleaved.argtypes = [u16p, f32p, i64, u16p]
        lib.orc_rope_interleaved.restype = None
        lib.orc_qkv_epilogue.argtypes = [u16p, u16p, u16p, u16p, u16p, u16p, i64, i64,
                                         u16p, u16p, u16p, i64, i64, u16p, u16p, u16p, u16p,
                                         f32p, f32p, i64, f32, f32]
        lib.orc_qkv_epilogue.restype = ctypes.c_int
        lib.orc_bias_mul_add.argtypes = [u16p, u16p, u16p, u16p, u16p, i64, i64]
        lib.orc_bias_mul_add.restype = ctypes.c_int
        lib.orc_scale_residual_nss_fp8.argtypes = [u16p, u16p, u8p, u16p, u16p, u16p, u16p, u16p,
                                                   u16p, i64, f32, i64, i64, f32, f64p]
        lib.orc_scale_residual_nss_fp8.restype = ctypes.c_int
        lib.orc_token_cat_fp8.argtypes = [u8p, u16p, i64, u16p, i64, f32, i64]
        lib.orc_token_cat_fp8.restype = ctypes.c_int
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.orc_bf16_from_f32_n.argtypes = [f32p, u16p, i64]
        lib.orc_bf16_from_f64_n.argtypes = [f64p, u16p, i64]
        lib.orc_e4m3_encode_n.argtypes = [f32p, u8p, i64]
        lib.orc_bf16_fma_n.argtypes = [u16p, u16p, u16p, u16p, i64]
        lib.orc_bf16_add_n.argtypes = [u16p, u16p, u16p, i64]
        lib.orc_quantize_n.argtypes = [f32p, f32, u8p, i64]
        for name in ("orc_bf16_from_f32_n", "orc_bf16_from_f64_n", "orc_e4m3_encode_n",
                     "orc_bf16_fma_n", "orc_bf16_add_n", "orc_quantize_n"):
            getattr(lib, name).restype = None
        _lib = lib
        return lib


def _u16(a):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _ptr(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


# ---- scalar stages (exposed for the pin tests) ---------------------------------------------

def bf16_to_f64(b: int) -> float:
    return _load().orc_bf16_to_f64(int(b))


def bf16_from_f64(v: float) -> int:
    return int(_load().orc_bf16_from_f64(float(v)))


def bf16_from_f32(v) -> int:
    return int(_load().orc_bf16_from_f32(float(np.float32(v))))


def bf16_fma(a: int, b: int, c: int) -> int:
    return int(_load().orc_bf16_fma(int(a), int(b), int(c)))


def bf16_add(a: int, b: int) -> int:
    return int(_load().orc_bf16_add(int(a), int(b)))


def e4m3_decode(c: int) -> float:
    return _load().orc_e4m3_decode(int(c))


def e4m3_encode(v) -> int:
    return int(_load().orc_e4m3_encode(float(np.float32(v))))


def recip_f32(s) -> np.float32:
    return np.float32(_load().orc_recip_f32(float(np.float32(s))))


def quantize(v, inv) -> int:
    return int(_load().orc_quantize(float(np.float32(v)), float(np.float32(inv))))


def modulate(n: int, scale: int, shift: int) -> int:
    return int(_load().orc_modulate(int(n), int(scale), int(shift)))


def ln_row_t(x_row, eps: float = 1e-6) -> np.ndarray:
    """fp64 normalised values (x - mu) / sqrt(var + eps) of one bf16 row (before rounding)."""
    x, xp = _u16(x_row)
    t = np.empty(x.size, dtype=np.float64)
    _load().orc_ln_row_t(xp, x.size, float(np.float32(eps)), _ptr(t, ctypes.c_double))
    return t


# ---- vectorised helpers over arrays (loops run in C) ----------------------------------------

def bf16_from_f32_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    _load().orc_bf16_from_f32_n(_ptr(v, ctypes.c_float), _ptr(out, ctypes.c_uint16), v.size)
    return out


def bf16_from_f64_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().orc_bf16_from_f64_n(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16), v.size)
    return out


def e4m3_encode_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().orc_e4m3_encode_n(_ptr(v, ctypes.c_float), _ptr(out, ctypes.c_uint8), v.size)
    return out


def bf16_fma_array(a, b, c) -> np.ndarray:
    a, ap = _u16(a)
    b, bp = _u16(b)
    c, cp = _u16(c)
    out = np.empty(a.shape, np.uint16)
    _load().orc_bf16_fma_n(ap, bp, cp, _ptr(out, ctypes.c_uint16), a.size)
    return out


def bf16_add_array(a, b) -> np.ndarray:
    a, ap = _u16(a)
    b, bp = _u16(b)
    out = np.empty(a.shape, np.uint16)
    _load().orc_bf16_add_n(ap, bp, _ptr(out, ctypes.c_uint16), a.size)
    return out


def quantize_array(v, inv) -> np.ndarray:
    """E4M3(RN_fp32(v * inv)) elementwise; v float32 array."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().orc_quantize_n(_ptr(v, ctypes.c_float), float(np.float32(inv)),
                           _ptr(out, ctypes.c_uint8), v.size)
    return out


def e2m1_decode(c: int) -> float:
    return _load().orc_e2m1_decode(int(c) & 0xFF)


def e2m1_encode(v) -> int:
    return _load().orc_e2m1_encode(float(np.float32(v)))


def e2m1_encode_array(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().orc_e2m1_encode_n(_ptr(v, ctypes.c_float), _ptr(out, ctypes.c_uint8), v.size)
    return out


def nvfp4_group(x16, g) -> tuple[int, np.ndarray]:
    """One 16-element group: (E4M3 block-scale code, 8 packed E2M1 bytes)."""
    x, xp = _u16(x16)
    assert x.size == 16
    packed = np.zeros(8, np.uint8)
    code = _load().orc_nvfp4_group(xp, float(np.float32(g)), _ptr(packed, ctypes.c_uint8))
    return code, packed


def nvfp4_sf_offset(m: int, k: int, k_groups: int) -> int:
    return _load().orc_nvfp4_sf_offset(int(m), int(k), int(k_groups))


def nvfp4_sf_shape(rows: int, cols: int) -> tuple[int, int]:
    """(padded rows, padded groups) of the 128x4-tiled block-scale buffer."""
    k = cols // 16
    return (rows + 127) // 128 * 128, (k + 3) // 4 * 4


# ---- whole operations ------------------------------------------------------------------------

def nss_fp8(x, scale, shift, input_scale, mod_rows=0, eps=1e-6):
    """LayerNorm (no affine) -> modulate -> (bf16 y, E4M3 q). x: uint16 [rows, cols]."""
    x, xp = _u16(x)
    rows, cols = x.shape
    scale, sp = _u16(scale)
    shift, hp = _u16(shift)
    y = np.empty((rows, cols), np.uint16)
    q = np.empty((rows, cols), np.uint8)
    t = np.empty(max(cols, 1), np.float64)
    _load().orc_nss_fp8(_ptr(y, ctypes.c_uint16), _ptr(q, ctypes.c_uint8), xp, sp, hp,
                        int(mod_rows), float(np.float32(input_scale)), rows, cols,
                        float(np.float32(eps)), _ptr(t, ctypes.c_double))
    return y, q


def bias_mul_add(x, bias, gate, residual):
    """y = RN_bf16(RN_bf16(x + bias) * gate + residual) (single-rounded BF16 FMA)."""
    x, xp = _u16(x)
    rows, cols = x.shape
    bias, bp = _u16(bias)
    gate, gp = _u16(gate)
    residual, rp = _u16(residual)
    y = np.empty((rows, cols), np.uint16)
    _load().orc_bias_mul_add(_ptr(y, ctypes.c_uint16), xp, bp, gp, rp, rows, cols)
    return y


def scale_residual_nss_fp8(x, residual, bias, gate, scale, shift, input_scale, mod_rows=0,
                           eps=1e-6):
    """residual_out = RN_bf16(RN_bf16(x + bias) * gate + residual); (y, q) = nss_fp8(residual_out).

    bias may be None (then x is used as is)."""
    x, xp = _u16(x)
    rows, cols = x.shape
    residual, rp = _u16(residual)
    if bias is None:
        bp = ctypes.POINTER(ctypes.c_uint16)()
    else:
        bias, bp = _u16(bias)
    gate, gp = _u16(gate)
    scale, sp = _u16(scale)
    shift, hp = _u16(shift)
    ro = np.empty((rows, cols), np.uint16)
    y = np.empty((rows, cols), np.uint16)
    q = np.empty((rows, cols), np.uint8)
    t = np.empty(max(cols, 1), np.float64)
    _load().orc_scale_residual_nss_fp8(_ptr(ro, ctypes.c_uint16), _ptr(y, ctypes.c_uint16),
                                       _ptr(q, ctypes.c_uint8), xp, rp, bp, gp, sp, hp,
                                       int(mod_rows), float(np.float32(input_scale)), rows, cols,
                                       float(np.float32(eps)), _ptr(t, ctypes.c_double))
    return ro, y, q


def token_cat_fp8(a, m, input_scale):
    """q[r] = E4M3(cat(a[r], m[r]) * RN_fp32(1/input_scale)), without a bf16 concat."""
    a, ap = _u16(a)
    m, mp = _u16(m)
    rows, a_cols = a.shape
    m_cols = m.shape[1]
    assert m.shape[0] == rows
    q = np.empty((rows, a_cols + m_cols), np.uint8)
    _load().orc_token_cat_fp8(_ptr(q, ctypes.c_uint8), ap, a_cols, mp, m_cols,
                              float(np.float32(input_scale)), rows)
    return q


def token_cat_nvfp4(a, m, global_scale):
    """(q, sf): q [rows, cols/2] packed E2M1 of cat(a[r], m[r]) per 16-element group, sf the
    128x4-tiled E4M3 block scales (flat, padded rows/groups zero)."""
    a, ap = _u16(a)
    m, mp = _u16(m)
    rows, a_cols = a.shape
    m_cols = m.shape[1]
    assert m.shape[0] == rows and (a_cols + m_cols) % 16 == 0
    cols = a_cols + m_cols
    mp_, kp_ = nvfp4_sf_shape(rows, cols)
    q = np.empty((rows, cols // 2), np.uint8)
    sf = np.empty(mp_ * kp_, np.uint8)
    rc = _load().orc_token_cat_nvfp4(_ptr(q, ctypes.c_uint8), _ptr(sf, ctypes.c_uint8), ap, a_cols,
                                     mp, m_cols, float(np.float32(global_scale)), rows)
    assert rc == 0
    return q, sf


HEAD_DIM = 128


def rms_norm_head(x, w, eps=1e-6) -> np.ndarray:
    """n = RN_bf16(x * w / sqrt(mean(x^2) + eps)) for one head vector (uint16 bf16 bits)."""
    x, xp = _u16(x)
    w, wp = _u16(w)
    assert x.size == w.size
    out = np.empty(x.size, np.uint16)
    _load().orc_rms_norm_head(xp, wp, x.size, float(np.float32(eps)), _ptr(out, ctypes.c_uint16))
    return out


def rope_interleaved(n, cos_sin) -> np.ndarray:
    """Interleaved RoPE of one head vector with an fp32 cache row (cos first, then sin)."""
    n, np_ = _u16(n)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    assert cs.size == n.size
    out = np.empty(n.size, np.uint16)
    _load().orc_rope_interleaved(np_, _ptr(cs, ctypes.c_float), n.size, _ptr(out, ctypes.c_uint16))
    return out


def qkv_epilogue(txt, img, heads):
    """txt / img: dicts with q, k, v ([tokens, ld] uint16 arrays, head h at columns
    h*128 .. h*128+127 of each row), wq, wk ([128] uint16), cos_sin ([tokens, 128] float32)
    and eps. Returns joint (q, k, v), each [t_tokens + i_tokens, heads, 128] uint16."""
    def prep(st):
        arrs = {}
        for key in ("q", "k", "v", "wq", "wk"):
            arrs[key] = _u16(st[key])
        cs = np.ascontiguousarray(st["cos_sin"], dtype=np.float32)
        arrs["cs"] = (cs, _ptr(cs, ctypes.c_float))
        return arrs
    t, i = prep(txt), prep(img)
    tt, it = txt["q"].shape[0], img["q"].shape[0]
    for st, n in ((txt, tt), (img, it)):
        assert st["q"].shape[1] >= heads * HEAD_DIM and st["cos_sin"].shape == (n, HEAD_DIM)
        assert st["q"].shape == st["k"].shape == st["v"].shape
    out = [np.empty((tt + it, heads, HEAD_DIM), np.uint16) for _ in range(3)]
    rc = _load().orc_qkv_epilogue(
        *[_ptr(o, ctypes.c_uint16) for o in out],
        t["q"][1], t["k"][1], t["v"][1], txt["q"].shape[1], tt,
        i["q"][1], i["k"][1], i["v"][1], img["q"].shape[1], it,
        t["wq"][1], t["wk"][1], i["wq"][1], i["wk"][1], t["cs"][1], i["cs"][1], heads,
        float(np.float32(txt["eps"])), float(np.float32(img["eps"])))
    assert rc == 0
    return tuple(out)
