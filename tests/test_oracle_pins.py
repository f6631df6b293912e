"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each stage of the oracle is checked against an independent source: the E4M3 format
definition and torch's float8_e4m3fn cast, torch's bfloat16 cast, exact rational arithmetic
with a brute-force nearest-value search (tests/exact.py), closed forms of LayerNorm, and the
page's printed worked example. The checks are chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign or index, a transposed operand, a wrong tie rule, eps outside
the square root, sample instead of population variance) fails at least one of them.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F = Fraction


def bf(v) -> int:
    """bf16 bits of an fp32 value via torch's cast (round-to-nearest-even)."""
    return int(torch.tensor([float(v)], dtype=torch.float32).to(torch.bfloat16)
               .view(torch.int16).item()) & 0xFFFF


# ------------------------------------------------------------------------------------------
# E4M3
# ------------------------------------------------------------------------------------------

def test_e4m3_decode_matches_format_and_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        ov = oracle.e4m3_decode(c)
        ev = exact.e4m3_value(c)
        if (c & 0x7F) == 0x7F:
            assert math.isnan(ov) and math.isnan(tv[c]) and math.isnan(ev)
        else:
            assert ov == tv[c] == ev, hex(c)
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_roundtrip_all_codes():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00


def test_e4m3_midpoints_go_to_even_code():
    for c in range(0x00, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exactly representable in fp32
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want, hex(c)
        assert oracle.e4m3_encode(-mid) == want | 0x80
        # just off the midpoint goes to the nearer code
        above = np.nextafter(mid, np.float32(np.inf))
        below = np.nextafter(mid, np.float32(-np.inf))
        assert oracle.e4m3_encode(above) == c + 1
        assert oracle.e4m3_encode(below) == c


def test_e4m3_saturation_and_special_values():
    for v in (448.0, 449.0, 464.0, 479.9, 480.0, 1e30, float(np.finfo(np.float32).max), np.inf):
        assert oracle.e4m3_encode(v) == 0x7E, v
        assert oracle.e4m3_encode(-v) == 0xFE, v
    assert oracle.e4m3_encode(np.nan) == 0x7F
    # subnormal edges: 2^-10 is the tie between 0 and 2^-9 -> even (0);
    # 3*2^-10 is the tie between 2^-9 (0x01) and 2^-8 (0x02) -> even (0x02)
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02
    assert oracle.e4m3_encode(-(2.0 ** -11)) == 0x80
    assert oracle.e4m3_encode(-(2.0 ** -9)) == 0x81
    assert oracle.e4m3_encode(1.0) == 0x38
    assert oracle.e4m3_encode(-1.0) == 0xB8


def _torch_satfinite_e4m3(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return torch.clamp(t, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_on_random_and_constructed_values():
    rng = np.random.default_rng(1234)
    parts = [
        rng.standard_normal(2_000_000).astype(np.float32) * np.float32(30.0),
        (rng.standard_normal(500_000) * 2.0 ** rng.integers(-14, 12, 500_000)).astype(np.float32),
        rng.uniform(-500, 500, 200_000).astype(np.float32),
        # random fp32 bit patterns with exponents around the E4M3 range
        (rng.integers(0, 2 ** 23, 300_000) | ((rng.integers(100, 140, 300_000)) << 23)
         | (rng.integers(0, 2, 300_000) << 31)).astype(np.uint32).view(np.float32),
    ]
    # all midpoints and their fp32 neighbours
    mids = []
    for c in range(0x7E):
        m = np.float32((oracle.e4m3_decode(c) + oracle.e4m3_decode(c + 1)) / 2)
        mids += [m, np.nextafter(m, np.float32(1e9)), np.nextafter(m, np.float32(-1e9))]
    mids = np.array(mids, dtype=np.float32)
    parts += [mids, -mids]
    v = np.concatenate(parts)
    ours = oracle.e4m3_encode_array(v)
    ref = _torch_satfinite_e4m3(v)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:10]]


def test_e4m3_encode_matches_exact_nearest_search():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(4000) * 2.0 ** rng.integers(-12, 10, 4000)).astype(np.float32)
    ours = oracle.e4m3_encode_array(v)
    for i in range(v.size):
        assert ours[i] == exact.nearest_e4m3_satfinite(F(float(v[i]))), float(v[i])


# ------------------------------------------------------------------------------------------
# BF16 rounding
# ------------------------------------------------------------------------------------------

def test_bf16_from_f32_matches_torch_on_all_low_halves():
    """Rounding depends only on the low 16 bits given the high 16: take every low half for a
    sample of high halves (all exponents, both signs, edge mantissas)."""
    rng = np.random.default_rng(99)
    highs = set(int(h) for h in rng.integers(0, 0x10000, 200))
    for e in range(256):
        for m in (0x00, 0x01, 0x3F, 0x40, 0x7E, 0x7F):
            for s in (0, 1):
                highs.add((s << 15) | (e << 7) | m)
    highs = np.array(sorted(highs), dtype=np.uint32)
    low = np.arange(0x10000, dtype=np.uint32)
    for chunk in np.array_split(highs, 8):
        bits = ((chunk[:, None] << 16) | low[None, :]).ravel()
        f = bits.view(np.float32)
        ours = oracle.bf16_from_f32_array(f)
        ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(f)
        assert np.array_equal(ours[~nan], ref[~nan])
        # NaN stays NaN (payload is not part of the contract)
        assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)


@pytest.mark.slow
def test_bf16_from_f32_exhaustive_against_torch():
    """Every one of the 2^32 fp32 bit patterns (NaNs: still NaN)."""
    low = np.arange(0x10000, dtype=np.uint32)
    for h0 in range(0, 0x10000, 0x200):
        highs = np.arange(h0, h0 + 0x200, dtype=np.uint32)
        f = ((highs[:, None] << 16) | low[None, :]).ravel().view(np.float32)
        ours = oracle.bf16_from_f32_array(f)
        ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(f)
        assert np.array_equal(ours[~nan], ref[~nan]), hex(h0)
        assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)


@pytest.mark.slow
def test_e4m3_encode_exhaustive_against_torch():
    """Every finite fp32 bit pattern: clamp to +-448 and cast with torch, vs the oracle."""
    low = np.arange(0x10000, dtype=np.uint32)
    for h0 in range(0, 0x10000, 0x200):
        highs = np.arange(h0, h0 + 0x200, dtype=np.uint32)
        f = ((highs[:, None] << 16) | low[None, :]).ravel().view(np.float32)
        f = f[np.isfinite(f)]
        ours = oracle.e4m3_encode_array(f)
        assert np.array_equal(ours, _torch_satfinite_e4m3(f)), hex(h0)


def test_bf16_from_f64_matches_exact_nearest_search():
    rng = np.random.default_rng(5)
    vals = list(rng.standard_normal(3000) * 2.0 ** rng.integers(-140, 128, 3000))
    # exact midpoints between neighbouring bf16 values and values just around them
    for b in rng.integers(0, 0x7F7F, 500):
        lo, hi = exact.bf16_value(int(b)), exact.bf16_value(int(b) + 1)
        mid = (lo + hi) / 2  # exact in fp64
        vals += [mid, -mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)]
    vals += [3.3895313892515355e38, 3.3961775292304846e38, 3.4e38, 1e39, 2.0 ** -133, 2.0 ** -134,
             3 * 2.0 ** -135, 2.0 ** -150, 0.0, -0.0]
    for v in vals:
        want = exact.nearest_bf16(F(v)) if v != 0 else (0x8000 if math.copysign(1, v) < 0 else 0)
        assert oracle.bf16_from_f64(v) == want, v


# ------------------------------------------------------------------------------------------
# BF16 add and single-rounded BF16 FMA
# ------------------------------------------------------------------------------------------

def _golden_fma_example():
    with open(os.path.join(GOLDEN, "bias_fma_tie_example.json")) as fh:
        return json.load(fh)


def test_page_worked_example_bias_then_single_rounded_fma():
    g = _golden_fma_example()["inputs"]
    x, b, gate, r = (bf(g[k]) for k in ("x", "bias", "gate", "residual"))
    # the printed inputs are bf16 values
    assert [exact.bf16_value(v) for v in (x, b, gate, r)] == [g["x"], g["bias"], g["gate"], g["residual"]]
    xb = oracle.bf16_add(x, b)
    xb_exact = exact.nearest_bf16(F(g["x"]) + F(g["bias"]))
    assert xb == xb_exact
    y = oracle.bf16_fma(xb, gate, r)
    want = exact.nearest_bf16(F(exact.bf16_value(xb)) * F(g["gate"]) + F(g["residual"]))
    assert y == want
    assert exact.bf16_value(y) == -5079040.0
    # The product alone is an exact bf16 tie (154.5 quanta of 32768); rounding through fp32
    # first would land on the even neighbour instead. The oracle must not do that.
    p = F(exact.bf16_value(xb)) * F(g["gate"])
    assert p / 32768 == F(-309, 2)
    via_fp32 = bf(np.float32(np.float32(exact.bf16_value(xb)) * np.float32(g["gate"]))
                  + np.float32(g["residual"]))
    assert exact.bf16_value(via_fp32) == -5046272.0 and via_fp32 != y


def _random_bf16(rng, n, lo_exp=-30, hi_exp=30):
    v = rng.standard_normal(n) * 2.0 ** rng.integers(lo_exp, hi_exp, n)
    return np.array([bf(x) for x in v], dtype=np.uint16)


def test_bf16_fma_matches_exact_arithmetic():
    rng = np.random.default_rng(11)
    n = 3000
    a, b, c = _random_bf16(rng, n), _random_bf16(rng, n), _random_bf16(rng, n)
    # constructed ties: a*b exactly on a bf16 midpoint, c tiny (+, -, 0)
    ties = exact.bf16_product_ties()
    assert len(ties) > 100
    ta, tb, tc = [], [], []
    for i in range(600):
        m1, m2 = ties[int(rng.integers(len(ties)))]
        e1, e2 = int(rng.integers(-20, 20)), int(rng.integers(-20, 20))
        sgn = float(rng.choice([1.0, -1.0]))
        ta.append(bf(sgn * m1 * 2.0 ** e1))
        tb.append(bf(m2 * 2.0 ** e2))
        tc.append(bf(float([1.0, -1.0, 0.0][i % 3]) * 2.0 ** (e1 + e2 - 10)))
    # the constructed products really are ties
    for i in range(20):
        p = F(exact.bf16_value(ta[i])) * F(exact.bf16_value(tb[i]))
        lo = exact.nearest_bf16(p)
        assert exact.nearest_bf16(p + p / 2 ** 40) != exact.nearest_bf16(p - p / 2 ** 40)
    a = np.concatenate([a, ta]).astype(np.uint16)
    b = np.concatenate([b, tb]).astype(np.uint16)
    c = np.concatenate([c, tc]).astype(np.uint16)
    ours = oracle.bf16_fma_array(a, b, c)
    for i in range(a.size):
        v = F(exact.bf16_value(a[i])) * F(exact.bf16_value(b[i])) + F(exact.bf16_value(c[i]))
        if v == 0:
            continue  # sign-of-zero checked below
        assert ours[i] == exact.nearest_bf16(v), (hex(a[i]), hex(b[i]), hex(c[i]))
    # IEEE exact-zero sums: +0 unless both addends are -0
    pz, nz, one = bf(0.0), 0x8000, bf(1.0)
    assert oracle.bf16_fma(one, one, bf(-1.0)) == 0x0000
    assert oracle.bf16_fma(nz, one, nz) == 0x8000
    assert oracle.bf16_fma(nz, one, pz) == 0x0000


def test_bf16_add_matches_exact_and_the_pages_fp32_route():
    """RN_bf16(x + bias): the oracle rounds the exact sum once; the pages add in fp32 and
    cast. For two bf16 operands both are the same value -- check both."""
    rng = np.random.default_rng(3)
    n = 200_000
    a = _random_bf16(rng, 4000, -40, 40)
    b = _random_bf16(rng, 4000, -40, 40)
    ours = oracle.bf16_add_array(a, b)
    for i in range(a.size):
        v = F(exact.bf16_value(a[i])) + F(exact.bf16_value(b[i]))
        if v != 0:
            assert ours[i] == exact.nearest_bf16(v)
    # the page's fp32 route, via torch, on many more pairs (wide exponent gaps included)
    x = torch.randn(n, dtype=torch.float32) * torch.exp2(torch.randint(-30, 30, (n,)).float())
    y = torch.randn(n, dtype=torch.float32) * torch.exp2(torch.randint(-30, 30, (n,)).float())
    xb, yb = x.to(torch.bfloat16), y.to(torch.bfloat16)
    ref = (xb.float() + yb.float()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = oracle.bf16_add_array(xb.view(torch.int16).numpy().view(np.uint16),
                                 yb.view(torch.int16).numpy().view(np.uint16))
    nz = (ref & 0x7FFF) != 0
    assert np.array_equal(ours[nz], ref[nz])


# ------------------------------------------------------------------------------------------
# reciprocal, quantise, modulate
# ------------------------------------------------------------------------------------------

def test_reciprocal_is_correctly_rounded():
    with open(os.path.join(GOLDEN, "checkpoint_input_scale.json")) as fh:
        ck = json.load(fh)["input_scale"]
    rng = np.random.default_rng(17)
    scales = [ck, 0.0625, 0.25, 0.05, 0.0123, 0.02, 0.1, 1.0, 3.0, 1e-3, 448.0]
    scales += list(rng.uniform(1e-4, 10.0, 2000))
    for s in scales:
        s32 = np.float32(s)
        assert oracle.recip_f32(s32) == np.float32(exact.nearest_f32(1 / F(float(s32)))), s


def test_quantize_matches_torch_fp32_multiply_and_cast():
    rng = np.random.default_rng(23)
    v = np.array([exact.bf16_value(b) for b in _random_bf16(rng, 20000, -12, 10)], np.float32)
    for s in (0.4754464328, 0.0625, 0.25, 0.05, 0.0123):
        inv = oracle.recip_f32(s)
        ours = oracle.quantize_array(v, inv)
        prod = (torch.from_numpy(v) * torch.tensor(inv, dtype=torch.float32)).numpy()
        ref = _torch_satfinite_e4m3(prod)
        assert np.array_equal(ours, ref), s


def test_power_of_two_scales_put_many_values_on_e4m3_midpoints():
    """With s a power of two, y * (1/s) is exact and lands on an E4M3 midpoint whenever the
    fifth significant bit of y is set and the rest below is clear (~1/16 of values)."""
    rng = np.random.default_rng(29)
    y = np.array([exact.bf16_value(b) for b in _random_bf16(rng, 20000, -6, 3)], np.float32)
    for s in (0.0625, 0.25):
        inv = oracle.recip_f32(s)
        prod = y * inv
        on_mid = 0
        for p in prod[:4000]:
            a = abs(F(float(p)))
            if a == 0 or a >= 448:
                continue
            q = exact.nearest_e4m3_satfinite(a)
            # a is a midpoint iff distance to the chosen code equals distance to the other
            vq = abs(F(exact.e4m3_value(q)))
            other = [abs(F(exact.e4m3_value(c))) for c in (q - 1, q + 1) if 0 <= c < 0x7F]
            if any(abs(a - o) == abs(a - vq) for o in other):
                on_mid += 1
        assert on_mid > 150, (s, on_mid)


def test_modulate_is_one_fp32_fma_then_bf16():
    rng = np.random.default_rng(31)
    n = _random_bf16(rng, 3000, -8, 3)
    sc = _random_bf16(rng, 3000, -8, 0)
    sh = _random_bf16(rng, 3000, -8, 0)
    for i in range(n.size):
        one_plus = np.float32(np.float32(1.0) + np.float32(exact.bf16_value(sc[i])))
        exact_fma = F(exact.bf16_value(n[i])) * F(float(one_plus)) + F(exact.bf16_value(sh[i]))
        r32 = exact.nearest_f32(exact_fma) if exact_fma != 0 else 0.0
        want = bf(r32)
        got = oracle.modulate(int(n[i]), int(sc[i]), int(sh[i]))
        if exact_fma == 0:
            assert (got & 0x7FFF) == 0
        else:
            assert got == want, (hex(n[i]), hex(sc[i]), hex(sh[i]))


# ------------------------------------------------------------------------------------------
# LayerNorm stage: brute force on tiny rows, closed forms on wide rows
# ------------------------------------------------------------------------------------------

EPS32 = F(float(np.float32(1e-6)))


def _exact_nss_row(xbits, scb, shb, input_scale):
    """Exact reference for one row: exact mean / population variance, RN_bf16 of
    (x - mu)/sqrt(var + eps) decided by squared comparisons, then the fp32 FMA modulate,
    bf16 cast and fp32 quantise (torch's float8 cast)."""
    xs = [F(exact.bf16_value(b)) for b in xbits]
    C = len(xs)
    mu = sum(xs) / C
    var = sum((v - mu) ** 2 for v in xs) / C
    w = var + EPS32
    inv = np.float32(exact.nearest_f32(1 / F(float(np.float32(input_scale)))))
    ys, qs = [], []
    for j, v in enumerate(xs):
        nb = exact.rnb_of_quotient(v - mu, w)
        one_plus = np.float32(np.float32(1.0) + np.float32(exact.bf16_value(scb[j])))
        fm = F(exact.bf16_value(nb)) * F(float(one_plus)) + F(exact.bf16_value(shb[j]))
        r32 = exact.nearest_f32(fm) if fm != 0 else 0.0
        yb = bf(r32)
        ys.append(yb)
        prod = np.float32(np.float32(exact.bf16_value(yb)) * inv)
        qs.append(int(_torch_satfinite_e4m3(np.array([prod]))[0]))
    return ys, qs


def _small_rows(rng):
    rows = []
    for C in (1, 2, 3, 4):
        for _ in range(60):
            rows.append([bf(v) for v in rng.standard_normal(C) * 2.0 ** int(rng.integers(-6, 6))])
    rows += [
        [bf(1.0)] * 4,                       # constant row: t = 0 exactly
        [bf(1e-3), bf(-1e-3)],               # var comparable to eps: eps placement matters
        [bf(2e-3), bf(-2e-3), bf(1e-3), bf(0.0)],
        [bf(100.0), bf(100.5), bf(99.5), bf(100.25)],  # large mean, small spread
        [bf(-3.0), bf(5.0)],
        [bf(1.0), bf(2.0), bf(4.0)],         # asymmetric row: catches sample-vs-population var
        [bf(0.5), bf(-7.0), bf(3.0), bf(0.0)],
    ]
    return rows


def test_ln_stage_matches_exact_brute_force_on_tiny_rows():
    rng = np.random.default_rng(41)
    for xr in _small_rows(rng):
        C = len(xr)
        scb = [bf(v) for v in rng.standard_normal(C) * 0.1]
        shb = [bf(v) for v in rng.standard_normal(C) * 0.1]
        for s in (0.4754464328, 0.0625, 0.0123):
            y, q = oracle.nss_fp8(np.array([xr], np.uint16), np.array([scb], np.uint16),
                                  np.array([shb], np.uint16), s)
            ye, qe = _exact_nss_row(xr, scb, shb, s)
            assert list(y[0]) == ye, (xr, s)
            assert list(q[0]) == qe, (xr, s)


def test_ln_normalised_value_rounding_matches_exact_decision():
    """n = RN_bf16((x - mu)/sqrt(var + eps)) with scale = shift = 0 (so y == n) on rows of
    a few elements, exact decision by squared comparisons."""
    rng = np.random.default_rng(43)
    zero = np.zeros((1, 4), np.uint16)
    for _ in range(300):
        xr = [bf(v) for v in rng.standard_normal(4) * 2.0 ** int(rng.integers(-10, 10))]
        xs = [F(exact.bf16_value(b)) for b in xr]
        mu = sum(xs) / 4
        w = sum((v - mu) ** 2 for v in xs) / 4 + EPS32
        want = [exact.rnb_of_quotient(v - mu, w) for v in xs]
        y, _ = oracle.nss_fp8(np.array([xr], np.uint16), zero, zero, 1.0)
        got = [int(v) for v in y[0]]
        # y = RN_bf16(fma(n, 1, 0)) = n except for the sign of an exact zero
        assert [g & 0xFFFF if (g & 0x7FFF) else 0 for g in got] == \
               [w_ & 0xFFFF if (w_ & 0x7FFF) else 0 for w_ in want], xr


def test_ln_closed_forms_on_wide_rows():
    from workloads import nss_inputs
    inp = nss_inputs(16, 3072, seed=5)
    zero = np.zeros((1, 3072), np.uint16)
    y, _ = oracle.nss_fp8(inp["x"], zero, zero, 1.0)
    n = np.array([[exact.bf16_value(b) for b in row] for row in y[:4]], np.float64)
    for row in n:
        assert abs(row.mean()) < 2e-3
        assert abs(row.var() - 1.0) < 5e-3
    # constant rows: n == 0 exactly, y == shift, q == E4M3(shift * inv)
    xc = np.full((3, 3072), bf(0.75), np.uint16)
    y, q = oracle.nss_fp8(xc, inp["scale"], inp["shift"], 0.05)
    assert np.array_equal(y, np.broadcast_to(inp["shift"], y.shape))
    sh = np.array([exact.bf16_value(b) for b in inp["shift"][0]], np.float32)
    inv = oracle.recip_f32(0.05)
    qe = _torch_satfinite_e4m3((torch.from_numpy(sh) * torch.tensor(inv)).numpy())
    assert np.array_equal(q, np.broadcast_to(qe, q.shape))


def test_ln_stats_track_an_fp64_numpy_layernorm():
    """torch's LayerNorm (fp64, no affine) as a library check of the statistics: the fp64
    normalised values agree to ~1e-12 on rows with outlier channels."""
    from workloads import nss_inputs
    inp = nss_inputs(8, 3072, seed=9, outlier_channels=30)
    x = np.array([[exact.bf16_value(b) for b in row] for row in inp["x"]], np.float64)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (3072,), eps=float(np.float32(1e-6))).numpy()
    for r in range(8):
        t = oracle.ln_row_t(inp["x"][r])
        assert np.max(np.abs(t - ref[r])) < 1e-10


# ------------------------------------------------------------------------------------------
# whole operations: composition invariants
# ------------------------------------------------------------------------------------------

def test_scale_residual_is_bias_mul_add_then_nss():
    from workloads import residual_inputs
    inp = residual_inputs(64, 3072, seed=3)
    ro, y, q = oracle.scale_residual_nss_fp8(inp["x"], inp["residual"], inp["bias"], inp["gate"],
                                             inp["scale"], inp["shift"], 0.05)
    ro2 = oracle.bias_mul_add(inp["x"], inp["bias"], inp["gate"][0], inp["residual"])
    assert np.array_equal(ro, ro2)
    y2, q2 = oracle.nss_fp8(ro, inp["scale"], inp["shift"], 0.05)
    assert np.array_equal(y, y2) and np.array_equal(q, q2)
    # no bias: x is used as is, i.e. residual_out = RN_bf16(x * gate + residual)
    ro3, _, _ = oracle.scale_residual_nss_fp8(inp["x"], inp["residual"], None, inp["gate"],
                                              inp["scale"], inp["shift"], 0.05)
    ro4 = oracle.bf16_fma_array(inp["x"], np.broadcast_to(inp["gate"], inp["x"].shape),
                                inp["residual"])
    assert np.array_equal(ro3, ro4)


def test_bias_mul_add_elementwise_against_exact():
    from workloads import residual_inputs
    inp = residual_inputs(4, 256, seed=8)
    y = oracle.bias_mul_add(inp["x"], inp["bias"], inp["gate"][0], inp["residual"])
    for r in range(4):
        for j in range(0, 256, 3):
            xb = exact.nearest_bf16(F(exact.bf16_value(inp["x"][r, j])) + F(exact.bf16_value(inp["bias"][j])))
            v = F(exact.bf16_value(xb)) * F(exact.bf16_value(inp["gate"][0, j])) + \
                F(exact.bf16_value(inp["residual"][r, j]))
            if v != 0:
                assert y[r, j] == exact.nearest_bf16(v)


def test_per_sample_modulation_uses_row_div_mod_rows():
    from workloads import nss_inputs
    inp = nss_inputs(6, 64, seed=2, n_mod=3)
    y, q = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], 0.02, mod_rows=2)
    for r in range(6):
        m = r // 2
        y1, q1 = oracle.nss_fp8(inp["x"][r:r + 1], inp["scale"][m:m + 1], inp["shift"][m:m + 1], 0.02)
        assert np.array_equal(y[r], y1[0]) and np.array_equal(q[r], q1[0])


def test_token_cat_is_quantised_concat():
    from workloads import token_cat_inputs
    inp = token_cat_inputs(5, 48, 80, seed=4)
    q = oracle.token_cat_fp8(inp["a"], inp["m"], 0.1)
    cat = np.concatenate([inp["a"], inp["m"]], axis=1)
    v = (cat.astype(np.uint32) << 16).view(np.float32)
    inv = oracle.recip_f32(0.1)
    ref = _torch_satfinite_e4m3((torch.from_numpy(v) * torch.tensor(inv)).numpy())
    assert np.array_equal(q, ref)


# ------------------------------------------------------------------------------------------
# Token-concat -> NVFP4
# ------------------------------------------------------------------------------------------

def test_e2m1_decode_matches_format_definition():
    for c in range(16):
        assert Fraction(oracle.e2m1_decode(c)) == exact.e2m1_value(c), c
        assert math.copysign(1.0, oracle.e2m1_decode(c)) == (-1.0 if c & 8 else 1.0)
    assert [oracle.e2m1_decode(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def _e2m1_probe_values(rng):
    grid = [float(exact.e2m1_value(c)) for c in range(8)]
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])]
    vals = grid + mids + [6.5, 7.0, 1e30, 3.4e38, 1e-30, 0.0]
    for v in mids + grid[1:]:
        vals += [float(np.nextafter(np.float32(v), np.float32(0))),
                 float(np.nextafter(np.float32(v), np.float32(np.inf)))]
    vals += list(rng.uniform(0, 8, 2000).astype(np.float32))
    vals += list((2.0 ** rng.uniform(-12, 4, 2000)).astype(np.float32))
    vals = np.array(vals, np.float32)
    return np.concatenate([vals, -vals, np.array([-0.0], np.float32)])


def test_e2m1_encode_matches_exact_nearest_search():
    v = _e2m1_probe_values(np.random.default_rng(7))
    got = oracle.e2m1_encode_array(v)
    want = np.array([exact.nearest_e2m1_satfinite(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, want)
    # spot values of the tie rule and of saturation, from the definition
    for x, c in [(0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6),
                 (5.0, 0x6), (5.01, 0x7), (1e9, 0x7), (-0.2, 0x8), (-0.0, 0x8), (-5.0, 0xE)]:
        assert oracle.e2m1_encode(x) == c, (x, c)


def test_nvfp4_sf_offset_matches_hand_worked_layout():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_sf_layout.json")))
    for m, k, kk, off in g["cases"]:
        assert oracle.nvfp4_sf_offset(m, k, kk) == off, (m, k, kk)


@pytest.mark.parametrize("rows,groups", [(1, 4), (128, 4), (129, 6), (300, 12), (256, 1)])
def test_nvfp4_sf_offset_matches_reshape_construction(rows, groups):
    m_pad, k_pad = oracle.nvfp4_sf_shape(rows, 16 * groups)
    pos = exact.blocked_scale_positions(m_pad, k_pad)
    got = np.array([[oracle.nvfp4_sf_offset(m, k, groups) for k in range(k_pad)]
                    for m in range(m_pad)])
    assert np.array_equal(got, pos)
    assert sorted(got.ravel()) == list(range(m_pad * k_pad))  # a permutation of the buffer


def _group_bits(vals):
    return np.array([bf(v) for v in vals], np.uint16)


def _unpack(packed):
    out = []
    for b in packed:
        out += [int(b) & 0xF, int(b) >> 4]
    return out


@pytest.mark.parametrize("e", [-6, -3, 0, 2, 8])
def test_nvfp4_group_is_exact_on_representable_groups(e):
    # Every element an E2M1 value times 2^e with amax 6 * 2^e and global scale 1: the block
    # scale must come out as 2^e and every element as its own E2M1 code (closed form).
    rng = np.random.default_rng(100 + e)
    codes = rng.integers(0, 16, 16)
    codes[rng.integers(0, 16)] = 7
    vals = [float(exact.e2m1_value(int(c))) * 2.0 ** e for c in codes]
    code, packed = oracle.nvfp4_group(_group_bits(vals), 1.0)
    assert Fraction(exact.e4m3_value(code)) == Fraction(2) ** e
    got = _unpack(packed)
    for c, g_ in zip(codes, got):
        assert exact.e2m1_value(g_) == exact.e2m1_value(int(c))  # -0 and +0 both allowed only if equal


def test_nvfp4_group_nibble_order_and_zero_groups():
    code, packed = oracle.nvfp4_group(_group_bits([6.0, 0.0] + [0.0] * 14), 1.0)
    assert code == 0x38 and packed[0] == 0x07 and not packed[1:].any()  # element 0 low nibble
    code, packed = oracle.nvfp4_group(_group_bits([0.0, -6.0] + [0.0] * 14), 1.0)
    assert code == 0x38 and packed[0] == 0xF0
    code, packed = oracle.nvfp4_group(_group_bits([0.0] * 16), 3.0)
    assert code == 0 and not packed.any()
    code, packed = oracle.nvfp4_group(np.full(16, 0x8000, np.uint16), 3.0)   # all -0
    assert code == 0 and (packed == 0x88).all()
    # block scale below half the smallest E4M3 subnormal: code 0, every element a signed zero
    code, packed = oracle.nvfp4_group(_group_bits([1e-4, -1e-4] * 8), 1.0)
    assert code == 0 and (packed == 0x80).all()


def _exact_group(xbits, g):
    """Brute-force evaluation of the group reading with exact rationals and nearest-value
    searches (tests/exact.py); shares no rounding code with the oracle."""
    g = np.float32(g)
    xs = [exact.bf16_value(int(b)) for b in xbits]
    amax = max(abs(Fraction(x)) for x in xs)
    inv6 = exact.nearest_f32(Fraction(1, 6))
    s = exact.nearest_f32(Fraction(float(g)) * Fraction(exact.nearest_f32(amax * Fraction(inv6))))
    code = exact.nearest_e4m3_satfinite(Fraction(s))
    if code & 0x7F == 0:
        out = 0.0
    else:
        inv_g = exact.nearest_f32(1 / Fraction(float(g)))
        d = exact.nearest_f32(Fraction(exact.e4m3_value(code)) * Fraction(inv_g))
        out = exact.nearest_f32(1 / Fraction(d))
    elems = []
    for x in xs:
        p = Fraction(x) * Fraction(out)
        v = exact.nearest_f32(p) if p != 0 else math.copysign(0.0, x) * (1.0 if out >= 0 else -1.0)
        elems.append(exact.nearest_e2m1_satfinite(v))
    return code, elems


def test_nvfp4_group_matches_exact_brute_force():
    rng = np.random.default_rng(11)
    for trial in range(300):
        scale_exp = rng.uniform(-8, 8)
        x = (rng.standard_normal(16) * 2.0 ** scale_exp).astype(np.float32)
        if trial % 7 == 0:
            x[rng.integers(0, 16)] *= 40.0         # an outlier sets the block scale
        g = np.float32(2.0 ** rng.uniform(-4, 12))
        if trial % 11 == 0:
            g = np.float32(2688.0 / 7.5)            # a typical input_scale_inv
        bits = _group_bits(x)
        code, packed = oracle.nvfp4_group(bits, g)
        want_code, want_elems = _exact_group(bits, g)
        assert code == want_code, trial
        assert _unpack(packed) == want_elems, trial


def test_nvfp4_group_amax_element_lands_on_six():
    # Invariant of the format: with a normal, unsaturated block scale (relative rounding
    # error <= 2^-4), amax * out lies within [6/(1+2^-4), 6/(1-2^-4)], which rounds to 6.
    rng = np.random.default_rng(12)
    hits = 0
    for _ in range(2000):
        x = (rng.standard_normal(16) * 2.0 ** rng.uniform(-6, 6)).astype(np.float32)
        g = np.float32(2.0 ** rng.uniform(-3, 6))
        bits = _group_bits(x)
        code, packed = oracle.nvfp4_group(bits, g)
        if not (0x08 <= code <= 0x7D):          # normal and below the 448 clamp
            continue
        xv = np.array([exact.bf16_value(int(b)) for b in bits])
        i = int(np.argmax(np.abs(xv)))
        e = _unpack(packed)[i]
        assert e & 7 == 7, (code, xv[i])
        hits += 1
        # every element dequantises within half an E2M1 step (x the block scale) of x
        dq = np.array([float(exact.e2m1_value(c)) for c in _unpack(packed)])
        unit = float(exact.e4m3_value(code)) / float(g)
        assert np.all(np.abs(dq * unit - xv) <= 1.0 * unit * 1.07 + 1e-30)
    assert hits > 1500


def test_nvfp4_group_saturates_the_block_scale():
    x = _group_bits([1000.0] + [1.0] * 15)
    code, packed = oracle.nvfp4_group(x, 1000.0)    # s = 1000 * 1000 / 6 >> 448
    assert code == 0x7E
    assert _unpack(packed)[0] == 7


@pytest.mark.parametrize("rows,a_cols,m_cols", [(5, 48, 80), (130, 40, 88), (128, 64, 64),
                                                (1, 16, 16)])
def test_token_cat_nvfp4_is_grouped_concat(rows, a_cols, m_cols):
    rng = np.random.default_rng(rows + a_cols)
    a = np.array([bf(v) for v in rng.standard_normal(rows * a_cols)], np.uint16).reshape(rows, a_cols)
    m = np.array([bf(v) for v in 3 * rng.standard_normal(rows * m_cols)], np.uint16).reshape(rows, m_cols)
    g = np.float32(2688.0 / 12.0)
    q, sf = oracle.token_cat_nvfp4(a, m, g)
    cols = a_cols + m_cols
    K = cols // 16
    m_pad, k_pad = oracle.nvfp4_sf_shape(rows, cols)
    pos = exact.blocked_scale_positions(m_pad, k_pad)
    cat = np.concatenate([a, m], axis=1)
    seen = np.zeros(sf.size, bool)
    for r in range(rows):
        for k in range(K):
            code, packed = oracle.nvfp4_group(cat[r, 16 * k:16 * k + 16], g)
            assert sf[pos[r, k]] == code
            assert np.array_equal(q[r, 8 * k:8 * k + 8], packed)
            seen[pos[r, k]] = True
    assert not sf[~seen].any()          # padding rows and groups hold zero scales


# ------------------------------------------------------------------------------------------
# QKV epilogue: per-head RMSNorm, interleaved RoPE, joint pack
# ------------------------------------------------------------------------------------------

def _exact_rms_head(xb, wb, eps):
    xs = [F(exact.bf16_value(int(b))) for b in xb]
    ws = [F(exact.bf16_value(int(b))) for b in wb]
    W_ = sum(x * x for x in xs) / len(xs) + F(float(np.float32(eps)))
    return [exact.rnb_of_quotient(x * w, W_) for x, w in zip(xs, ws)]


def _rand_bits(rng, n, lo=-8, hi=8):
    v = rng.standard_normal(n) * 2.0 ** rng.uniform(lo, hi, n)
    return np.array([bf(x) for x in v], np.uint16)


@pytest.mark.parametrize("D", [2, 4, 8, 128])
def test_rms_norm_head_matches_exact_brute_force(D):
    rng = np.random.default_rng(D)
    for trial in range(60 if D < 128 else 12):
        x = _rand_bits(rng, D, -6, 6) if trial % 3 else _rand_bits(rng, D, -1, 1)
        w = _rand_bits(rng, D, -2, 2)
        if trial % 5 == 0:
            x[:] = x[0]                            # constant vector
        eps = [1e-6, 0.0, 1e-2][trial % 3]
        if eps == 0.0 and not any(exact.bf16_value(int(b)) for b in x):
            continue
        got = [int(v) for v in oracle.rms_norm_head(x, w, eps)]
        want = _exact_rms_head(x, w, eps)
        # exact zeros: the oracle keeps the IEEE sign of x * w, the exact search returns +0
        got = [0 if (g & 0x7FFF) == 0 else g for g in got]
        want = [0 if (v & 0x7FFF) == 0 else v for v in want]
        assert got == want, (D, trial)


def test_rms_norm_head_closed_forms():
    one = np.full(128, bf(1.0), np.uint16)
    # constant vector a, weight 1, eps 0: every value is sign(a) exactly
    for a in (3.0, -0.125, 1e-10, 6e4):
        n = oracle.rms_norm_head(np.full(128, bf(a), np.uint16), one, 0.0)
        assert (n == bf(math.copysign(1.0, a))).all()
    # scale invariance with eps = 0 (a power-of-two rescale is exact in BF16)
    rng = np.random.default_rng(5)
    x = _rand_bits(rng, 128, -3, 3)
    x2 = np.array([bf(exact.bf16_value(int(b)) * 2.0 ** 20) for b in x], np.uint16)
    assert np.array_equal(oracle.rms_norm_head(x, one, 0.0), oracle.rms_norm_head(x2, one, 0.0))
    # the weight multiplies: w = 2 doubles every value exactly
    two = np.full(128, bf(2.0), np.uint16)
    a = oracle.rms_norm_head(x, one, 1e-6)
    b = oracle.rms_norm_head(x, two, 1e-6)
    assert all(exact.bf16_value(int(v)) * 2 == exact.bf16_value(int(u)) for v, u in zip(a, b))
    # eps dominates a tiny vector: n is x / sqrt(eps) to within one BF16 step
    tiny = np.array([bf(1e-9)] * 128, np.uint16)
    n = oracle.rms_norm_head(tiny, one, 1e-2)
    approx = exact.bf16_value(int(tiny[0])) / math.sqrt(float(np.float32(1e-2)))
    assert abs(exact.bf16_value(int(n[0])) - approx) <= approx * 2.0 ** -8


def test_rms_norm_head_matches_torch_fp64_rms_norm():
    rms_norm = getattr(torch.nn.functional, "rms_norm", None)
    if rms_norm is None:
        pytest.skip("torch without rms_norm")
    rng = np.random.default_rng(9)
    for _ in range(200):
        x = _rand_bits(rng, 128, -4, 4)
        w = _rand_bits(rng, 128, -1, 1)
        xt = torch.tensor([exact.bf16_value(int(b)) for b in x], dtype=torch.float64)
        wt = torch.tensor([exact.bf16_value(int(b)) for b in w], dtype=torch.float64)
        ref = rms_norm(xt, (128,), wt, float(np.float32(1e-6))).numpy()
        # fp64 -> BF16 with one rounding (torch's own cast goes through fp32)
        ref = np.array([exact.nearest_bf16(F(float(v))) for v in ref], np.uint16)
        assert np.array_equal(oracle.rms_norm_head(x, w, 1e-6), ref)


def _torch_rope(nb, cs):
    """Interleaved RoPE in eager fp32 torch ops (each op rounded separately)."""
    n = torch.from_numpy(nb.view(np.int16)).view(torch.bfloat16).float()
    c = torch.from_numpy(cs[:64].copy())
    s = torch.from_numpy(cs[64:].copy())
    a, b = n[0::2], n[1::2]
    o = torch.empty(128, dtype=torch.float32)
    o[0::2] = a * c - b * s
    o[1::2] = b * c + a * s
    return o.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rope_matches_torch_eager_fp32_and_exact_steps():
    rng = np.random.default_rng(21)
    for trial in range(300):
        nb = _rand_bits(rng, 128, -6, 6)
        ang = rng.uniform(-1e4, 1e4, 64)
        cs = np.concatenate([np.cos(ang), np.sin(ang)]).astype(np.float32)
        got = oracle.rope_interleaved(nb, cs)
        assert np.array_equal(got, _torch_rope(nb, cs)), trial
        if trial < 20:
            for i in range(64):
                a, b = F(exact.bf16_value(int(nb[2 * i]))), F(exact.bf16_value(int(nb[2 * i + 1])))
                c, s = F(float(cs[i])), F(float(cs[64 + i]))
                r0 = F(exact.nearest_f32(a * c)) - F(exact.nearest_f32(b * s))
                r1 = F(exact.nearest_f32(b * c)) + F(exact.nearest_f32(a * s))
                for r, g in ((r0, got[2 * i]), (r1, got[2 * i + 1])):
                    want = exact.nearest_bf16(F(exact.nearest_f32(r))) if r != 0 else 0
                    assert (int(g) & 0x7FFF) == (want & 0x7FFF) and (r == 0 or int(g) == want)


def test_rope_closed_forms():
    rng = np.random.default_rng(22)
    nb = _rand_bits(rng, 128, -6, 6)
    ident = np.concatenate([np.ones(64), np.zeros(64)]).astype(np.float32)
    assert np.array_equal(oracle.rope_interleaved(nb, ident), nb)
    quarter = np.concatenate([np.zeros(64), np.ones(64)]).astype(np.float32)   # 90 degrees
    o = oracle.rope_interleaved(nb, quarter)
    assert np.array_equal(o[0::2], nb[1::2] ^ 0x8000) and np.array_equal(o[1::2], nb[0::2])
    half = np.concatenate([-np.ones(64), np.zeros(64)]).astype(np.float32)     # 180 degrees
    assert np.array_equal(oracle.rope_interleaved(nb, half) & 0x7FFF, nb & 0x7FFF)


def test_qkv_epilogue_is_per_head_norm_rope_and_joint_text_first():
    import workloads as W
    d = W.qkv_inputs(3, 4, heads=2, seed=4, extra_cols=16)   # row stride > 3*heads*128
    d["txt"]["eps"], d["img"]["eps"] = 1e-6, 1e-5
    jq, jk, jv = oracle.qkv_epilogue(d["txt"], d["img"], heads=2)
    assert jq.shape == (7, 2, 128)
    for r in range(7):
        st, rr = (d["txt"], r) if r < 3 else (d["img"], r - 3)
        for h in range(2):
            sl = slice(h * 128, h * 128 + 128)
            for x, w, out in ((st["q"], st["wq"], jq), (st["k"], st["wk"], jk)):
                n = oracle.rms_norm_head(x[rr, sl], w, st["eps"])
                assert np.array_equal(out[r, h], oracle.rope_interleaved(n, st["cos_sin"][rr]))
            assert np.array_equal(jv[r, h], st["v"][rr, sl])
