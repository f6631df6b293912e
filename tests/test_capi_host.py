"""Host-only checks of the C ABI (no GPU): the library builds for sm_103a, loads, exports
every function include/fp8q.h declares, and rejects bad arguments synchronously with the
documented status codes before touching any device."""
from __future__ import annotations

import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")

OK, NULL, ALIGN, SHAPE, UNSUPPORTED, ALIAS, CUDA, VALUE = range(8)


@pytest.fixture(scope="module")
def L():
    import fp8_quant_row_gb300 as fq
    fq.build()
    return fq._capi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8q_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("fp8q_nss_fp8", "fp8q_scale_residual_nss_fp8", "fp8q_bias_mul_add",
              "fp8q_token_cat_fp8"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    import fp8_quant_row_gb300._capi as capi
    names = declared_functions()
    assert sorted(capi.SYMBOLS) == names
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB], capture_output=True,
                         text=True, check=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), n


def test_library_is_built_for_sm_103a_only(L):
    import fp8_quant_row_gb300._capi as capi
    out = subprocess.run(["cuobjdump", "--list-elf", capi.LIB], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    elfs = [l for l in out.stdout.splitlines() if ".cubin" in l]
    assert elfs and all("sm_103a" in l for l in elfs), out.stdout


def test_status_strings_and_version(L):
    assert L.fp8q_version() == 0x000300
    for s in range(8):
        assert L.fp8q_status_string(s)
    assert L.fp8q_status_string(99) == b"unknown status"
    assert L.fp8q_last_cuda_error() == 0


A = 1 << 20  # fake, 16-byte aligned, non-overlapping "device" addresses (never dereferenced)


def nss(L, y=A, q=2 * A, x=3 * A, sc=4 * A, sh=5 * A, mod_rows=0, s=6 * A, rows=4, cols=3072,
        eps=1e-6):
    return L.fp8q_nss_fp8(y, q, x, sc, sh, mod_rows, s, rows, cols, eps, None)


def test_nss_argument_checks(L):
    assert nss(L, rows=-1) == SHAPE
    assert nss(L, cols=3070) == SHAPE
    assert nss(L, cols=0) == SHAPE
    assert nss(L, cols=32768 + 8) == SHAPE
    assert nss(L, mod_rows=-2) == SHAPE
    assert nss(L, eps=-1.0) == VALUE
    assert nss(L, eps=float("nan")) == VALUE
    assert nss(L, eps=float("inf")) == VALUE
    assert nss(L, rows=0, y=None, q=None, x=None) == OK  # nothing to do, nothing touched
    assert nss(L, y=None) == NULL
    assert nss(L, s=None) == NULL
    assert nss(L, x=3 * A + 8) == ALIGN
    assert nss(L, q=2 * A + 1) == ALIGN
    assert nss(L, y=3 * A) == ALIAS                    # y on top of x
    assert nss(L, q=A + 4096) == ALIAS                 # q inside y
    assert nss(L, sc=A + 16) == ALIAS                  # scale inside y
    assert nss(L, s=2 * A + 64) == ALIAS               # input_scale inside q


def test_scale_residual_argument_checks(L):
    def call(ro=A, y=2 * A, q=3 * A, x=4 * A, res=5 * A, b=6 * A, g=7 * A, sc=8 * A, sh=9 * A,
             s=10 * A, rows=4, cols=3072):
        return L.fp8q_scale_residual_nss_fp8(ro, y, q, x, res, b, g, sc, sh, 0, s, rows, cols,
                                             1e-6, None)
    assert call(rows=-5) == SHAPE
    assert call(g=None) == NULL
    assert call(b=6 * A + 2) == ALIGN
    assert call(ro=4 * A) == ALIAS                     # residual_out on x
    assert call(y=5 * A) == ALIAS                      # y on residual
    assert call(ro=5 * A, y=5 * A + 8192) == ALIAS     # in-place residual but y overlaps it


def test_bias_mul_add_argument_checks(L):
    def call(y=A, x=2 * A, b=3 * A, g=4 * A, r=5 * A, rows=4, cols=3072):
        return L.fp8q_bias_mul_add(y, x, b, g, r, rows, cols, None)
    assert call(cols=12) == SHAPE
    assert call(cols=0) == SHAPE
    assert call(rows=0, y=None) == OK
    assert call(r=None) == NULL
    assert call(g=4 * A + 4) == ALIGN
    assert call(y=2 * A + 16) == ALIAS                 # partial overlap with x
    assert call(y=3 * A) == ALIAS                      # y over bias


def test_token_cat_argument_checks(L):
    def call(q=A, a=8 * A, ac=6144, m=16 * A, mc=18432, s=40 * A, rows=4):
        return L.fp8q_token_cat_fp8(q, a, ac, m, mc, s, rows, None)
    assert call(ac=6136) == SHAPE
    assert call(mc=8) == SHAPE
    assert call(rows=-1) == SHAPE
    assert call(rows=0, q=None) == OK
    assert call(m=None) == NULL
    assert call(a=8 * A + 8) == ALIGN
    assert call(q=16 * A) == ALIAS


def test_binding_fails_loudly_without_the_library(tmp_path):
    code = (
        "import fp8_quant_row_gb300._capi as c, fp8_quant_row_gb300._build as b\n"
        f"c.LIB = {str(tmp_path / 'missing.so')!r}\n"
        "c._lib = None\n"
        "try:\n"
        "    c.lib()\n"
        "except RuntimeError as e:\n"
        "    print('raised', e)\n"
    )
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert "raised" in out.stdout and "no non-CUDA fallback" in out.stdout, out.stderr


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "fp8_quant_row_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text), f
    code = ("import sys, fp8_quant_row_gb300\n"
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert out.stdout.strip() == "False", out.stderr


def test_token_cat_nvfp4_argument_checks(L):
    def call(q=A, sf=4 * A, a=8 * A, ac=6144, m=16 * A, mc=18432, s=40 * A, rows=4):
        return L.fp8q_token_cat_nvfp4(q, sf, a, ac, m, mc, s, rows, None)
    assert call(ac=6144 - 16) == SHAPE       # parts must be multiples of 64 columns
    assert call(mc=32) == SHAPE
    assert call(rows=-1) == SHAPE
    assert call(rows=0, q=None, sf=None) == OK
    assert call(sf=None) == NULL
    assert call(s=None) == NULL
    assert call(a=8 * A + 16) == ALIGN       # 16-byte aligned is not enough for the data
    assert call(q=A + 16) == ALIGN
    assert call(sf=4 * A + 8) == ALIGN
    assert call(sf=8 * A + 64) == ALIAS      # scales inside a
    assert call(q=16 * A) == ALIAS
    assert call(sf=A + 32) == ALIAS         # scales inside q
    assert call(s=4 * A + 4) == ALIAS        # global scale inside the scale buffer


def test_nvfp4_scale_bytes(L):
    f = L.fp8q_nvfp4_scale_bytes
    assert f(4608, 24576) == 4608 * 1536
    assert f(17, 24576) == 128 * 1536          # rows padded to 128
    assert f(1, 16) == 128 * 4                 # groups padded to 4
    assert f(129, 80) == 256 * 8
    assert f(0, 64) == 0
    assert f(-1, 64) == -1 and f(4, 24) == -1 and f(4, 0) == -1


def test_qkv_epilogue_argument_checks(L):
    import fp8_quant_row_gb300._capi as capi

    def stream(base, tokens=4, ld=3 * 24 * 128, eps=1e-6):
        return capi.QkvStream(base, base + 24 * 256, base + 48 * 256, ld, tokens,
                              base + 100 * A, base + 100 * A + 4096, base + 101 * A, eps)

    def call(jq=A, jk=2 * A, jv=3 * A, txt=None, img=None, heads=24):
        txt = txt or stream(10 * A)
        img = img or stream(20 * A)
        return L.fp8q_qkv_epilogue(jq, jk, jv, txt, img, heads, None)

    assert call(heads=0) == SHAPE
    assert call(txt=stream(10 * A, ld=24 * 128 - 16)) == SHAPE      # row narrower than heads
    assert call(img=stream(20 * A, ld=3 * 24 * 128 + 8)) == SHAPE   # stride not 16 values
    assert call(txt=stream(10 * A, tokens=-1)) == SHAPE
    assert call(txt=stream(10 * A, tokens=0), img=stream(20 * A, tokens=0), jq=None) == OK
    assert call(img=stream(20 * A, eps=0.0)) == VALUE
    assert call(img=stream(20 * A, eps=float("nan"))) == VALUE
    assert call(jk=None) == NULL
    assert call(jq=A + 16) == ALIGN
    assert call(txt=stream(10 * A + 16)) == ALIGN
    assert call(jk=A + 4096) == ALIAS                                # outputs overlap
    assert call(jv=10 * A + 256) == ALIAS                            # output over text q
    assert call(jq=20 * A + 100 * A + 64) == ALIAS                  # output over a weight
