"""ctypes view of the C ABI declared in include/fp8q.h (libfp8q.so, built in-tree).

There is no fallback: if the library is missing or does not load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB

_lock = threading.Lock()
_lib = None

STATUS = {0: "FP8Q_OK", 1: "FP8Q_ERR_NULL", 2: "FP8Q_ERR_ALIGN", 3: "FP8Q_ERR_SHAPE",
          4: "FP8Q_ERR_UNSUPPORTED", 5: "FP8Q_ERR_ALIAS", 6: "FP8Q_ERR_CUDA",
          7: "FP8Q_ERR_VALUE"}

#: every function include/fp8q.h declares
SYMBOLS = ("fp8q_nss_fp8", "fp8q_scale_residual_nss_fp8", "fp8q_bias_mul_add",
           "fp8q_token_cat_fp8", "fp8q_token_cat_nvfp4", "fp8q_nvfp4_scale_bytes",
           "fp8q_qkv_epilogue", "fp8q_device_error",
           "fp8q_status_string", "fp8q_last_cuda_error",
           "fp8q_last_error_detail", "fp8q_version")


class QkvStream(ctypes.Structure):
    """struct fp8q_qkv_stream of include/fp8q.h."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("ld", ctypes.c_int64), ("tokens", ctypes.c_int64),
                ("q_weight", ctypes.c_void_p), ("k_weight", ctypes.c_void_p),
                ("cos_sin", ctypes.c_void_p), ("eps", ctypes.c_float)]


class Fp8qError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = lib().fp8q_status_string(self.status).decode()
        if self.status == 6:
            msg += (f" (cudaError_t {lib().fp8q_last_cuda_error()}: "
                    f"{lib().fp8q_last_error_detail().decode()})")
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)}: {msg}")


def lib():
    """Load libfp8q.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: build it with __graft_entry__.build() "
                               "(nvcc, sm_103a); there is no non-CUDA fallback")
        L = ctypes.CDLL(LIB)
        vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
        L.fp8q_nss_fp8.argtypes = [vp, vp, vp, vp, vp, i64, vp, i64, i64, f32, vp]
        L.fp8q_scale_residual_nss_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, vp,
                                                  i64, i64, f32, vp]
        L.fp8q_bias_mul_add.argtypes = [vp, vp, vp, vp, vp, i64, i64, vp]
        L.fp8q_token_cat_fp8.argtypes = [vp, vp, i64, vp, i64, vp, i64, vp]
        L.fp8q_token_cat_nvfp4.argtypes = [vp, vp, vp, i64, vp, i64, vp, i64, vp]
        L.fp8q_qkv_epilogue.argtypes = [vp, vp, vp, ctypes.POINTER(QkvStream),
                                         ctypes.POINTER(QkvStream), i64, vp]
        L.fp8q_nvfp4_scale_bytes.argtypes = [i64, i64]
        L.fp8q_nvfp4_scale_bytes.restype = i64
        for name in ("fp8q_nss_fp8", "fp8q_scale_residual_nss_fp8", "fp8q_bias_mul_add",
                     "fp8q_token_cat_fp8", "fp8q_token_cat_nvfp4", "fp8q_qkv_epilogue"):
            getattr(L, name).restype = i32
        L.fp8q_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.fp8q_device_error.restype = i32
        L.fp8q_status_string.argtypes = [i32]
        L.fp8q_status_string.restype = ctypes.c_char_p
        L.fp8q_last_cuda_error.argtypes = []
        L.fp8q_last_cuda_error.restype = i32
        L.fp8q_last_error_detail.argtypes = []
        L.fp8q_last_error_detail.restype = ctypes.c_char_p
        L.fp8q_version.argtypes = []
        L.fp8q_version.restype = i32
        _lib = L
        return L


def check(status: int, where: str) -> None:
    if status != 0:
        raise Fp8qError(status, where)
