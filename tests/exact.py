"""Exact-arithmetic brute-force helpers for the oracle pin tests.

Nothing here shares code with the oracle: rounding is decided by a nearest-neighbour search
over the sorted list of all finite values of the target format, with exact rational
distances (``fractions.Fraction``), ties broken toward the even bit pattern. That is the
textbook definition of round-to-nearest-even, evaluated by enumeration rather than by the
quantum arithmetic the oracle uses.
"""
from __future__ import annotations

import bisect
import math
import struct
from fractions import Fraction
from functools import lru_cache

import numpy as np


def f32_bits(v) -> int:
    return struct.unpack("<I", struct.pack("<f", float(np.float32(v))))[0]


def f32_from_bits(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", int(u) & 0xFFFFFFFF))[0]


def bf16_value(b: int) -> float:
    return f32_from_bits((int(b) & 0xFFFF) << 16)


@lru_cache(maxsize=1)
def _bf16_table():
    """Sorted non-negative finite bf16 values (as Fractions) with their bit patterns."""
    vals, bits = [], []
    for b in range(0x0000, 0x7F80):  # +0 .. largest finite
        vals.append(Fraction(bf16_value(b)))
        bits.append(b)
    return vals, bits


def nearest_bf16(v: Fraction) -> int:
    """bf16 bit pattern of RNE(v) for an exact rational v (overflow -> +-Inf)."""
    vals, bits = _bf16_table()
    neg = v < 0
    a = -v if neg else v
    sign = 0x8000 if neg else 0
    top = vals[-1]
    # Overflow threshold: halfway between the largest finite value and 2^128; a tie there
    # goes to the "even" pattern, which is the infinity encoding (largest finite is odd).
    ovf = top + (Fraction(2) ** 128 - top) / 2
    if a >= ovf:
        return sign | 0x7F80
    i = bisect.bisect_left(vals, a)
    if i < len(vals) and vals[i] == a:
        return sign | bits[i]
    if i == len(vals):
        return sign | bits[-1]
    lo, hi = i - 1, i
    dlo, dhi = a - vals[lo], vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if bits[lo] % 2 == 0 else hi
    return sign | bits[pick]


def nearest_f32(v: Fraction) -> float:
    """RNE of an exact rational to binary32 (finite range only): neighbours by nextafter,
    decided with exact distances."""
    guess = np.float32(float(v))  # within one ulp of the answer
    cands = {guess, np.nextafter(guess, np.float32(np.inf)),
             np.nextafter(guess, np.float32(-np.inf))}
    best = None
    for c in cands:
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - v)
        key = (d, f32_bits(c) & 1)  # tie -> even significand
        if best is None or key < best[0]:
            best = (key, c)
    return float(best[1])


@lru_cache(maxsize=1)
def _e4m3_table():
    """Non-negative finite E4M3 (fn) values from the format definition: 1 sign bit, 4
    exponent bits with bias 7, 3 mantissa bits, exponent field 0 subnormal, S.1111.111 NaN."""
    vals, codes = [], []
    for c in range(0x00, 0x7F):
        e, m = (c >> 3) & 0xF, c & 7
        v = Fraction(m, 8) * Fraction(2) ** (-6) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        vals.append(v)
        codes.append(c)
    return vals, codes


def e4m3_value(c: int) -> float:
    vals, _ = _e4m3_table()
    if (c & 0x7F) == 0x7F:
        return math.nan
    v = float(vals[c & 0x7F])
    return -v if c & 0x80 else v


def nearest_e4m3_satfinite(v: Fraction) -> int:
    """Saturating RNE to E4M3: |v| >= 448 -> +-448, else the nearest code, ties to even."""
    vals, codes = _e4m3_table()
    neg = v < 0
    a = -v if neg else v
    sign = 0x80 if neg else 0
    if a >= vals[-1]:
        return sign | codes[-1]
    i = bisect.bisect_left(vals, a)
    if vals[i] == a:
        return sign | codes[i]
    lo, hi = i - 1, i
    dlo, dhi = a - vals[lo], vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if codes[lo] % 2 == 0 else hi
    return sign | codes[pick]


def rnb_of_quotient(d: Fraction, w: Fraction) -> int:
    """RNE to bf16 of t = d / sqrt(w) (w > 0), decided without any square-root error:
    t is compared with candidate bf16 values and midpoints b through d^2 vs b^2 * w."""
    if d == 0:
        return 0x0000
    neg = d < 0
    ad = -d if neg else d
    approx = float(ad) / math.sqrt(float(w))
    vals, bits = _bf16_table()

    def cmp_t(b: Fraction) -> int:  # sign(|t| - b) for b >= 0
        lhs, rhs = ad * ad, b * b * w
        return (lhs > rhs) - (lhs < rhs)

    i = bisect.bisect_left(vals, Fraction(approx))
    i = min(max(i, 1), len(vals) - 1)
    # walk to the bracket vals[i-1] <= |t| < vals[i]
    while i > 1 and cmp_t(vals[i - 1]) < 0:
        i -= 1
    while i < len(vals) - 1 and cmp_t(vals[i]) >= 0:
        i += 1
    lo, hi = i - 1, i
    if cmp_t(vals[lo]) == 0:
        pick = lo
    else:
        mid = (vals[lo] + vals[hi]) / 2
        c = cmp_t(mid)
        if c < 0:
            pick = lo
        elif c > 0:
            pick = hi
        else:
            pick = lo if bits[lo] % 2 == 0 else hi
    return (0x8000 if neg else 0) | bits[pick]


@lru_cache(maxsize=1)
def bf16_product_ties():
    """All pairs (m1, m2) of 8-bit significands (128..255) whose exact product lies exactly
    on a midpoint between two adjacent bf16 values (integer enumeration)."""
    out = []
    for m1 in range(128, 256):
        for m2 in range(128, 256):
            p = m1 * m2
            low = p.bit_length() - 8
            if low > 0 and p % (1 << low) == (1 << (low - 1)):
                out.append((m1, m2))
    return out


@lru_cache(maxsize=1)
def _e2m1_table():
    """Non-negative E2M1 values from the format definition: 1 sign bit, 2 exponent bits with
    bias 1, 1 mantissa bit, exponent field 0 subnormal; no infinities or NaN."""
    vals, codes = [], []
    for c in range(0, 8):
        e, m = (c >> 1) & 3, c & 1
        v = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
        vals.append(v)
        codes.append(c)
    return vals, codes


def e2m1_value(c: int) -> Fraction:
    vals, _ = _e2m1_table()
    v = vals[c & 7]
    return -v if c & 8 else v


def nearest_e2m1_satfinite(v: float) -> int:
    """Saturating RNE of a finite float to E2M1 by nearest-value search with exact
    distances; the sign bit follows the sign of v (so -0.1 and -0.0 give 0x8)."""
    vals, codes = _e2m1_table()
    sign = 8 if math.copysign(1.0, v) < 0 else 0
    a = abs(Fraction(v))
    if a >= vals[-1]:
        return sign | codes[-1]
    i = bisect.bisect_left(vals, a)
    if vals[i] == a:
        return sign | codes[i]
    lo, hi = i - 1, i
    dlo, dhi = a - vals[lo], vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if codes[lo] % 2 == 0 else hi
    return sign | codes[pick]


def blocked_scale_positions(m_pad: int, k_pad: int) -> np.ndarray:
    """Position of every (row, group) block scale in the 128x4-tiled layout, built by array
    reshapes rather than by an offset formula: the padded [m_pad, k_pad] scale matrix is cut
    into 128x4 tiles (row-tile-major), each tile's 128 rows are split as 4 bands of 32 and
    stored as 32 lines of 16 bytes (line = row within its band; a line holds the 4 bands
    side by side, 4 groups each). Returns pos[m, k]."""
    ids = np.arange(m_pad * k_pad, dtype=np.int64).reshape(m_pad, k_pad)
    t = ids.reshape(m_pad // 128, 4, 32, k_pad // 4, 4)  # (row tile, band, line, group tile, c)
    t = t.transpose(0, 3, 2, 1, 4)                        # (row tile, group tile, line, band, c)
    stored = t.reshape(-1)                                # stored[p] = id of the scale at p
    pos = np.empty(m_pad * k_pad, np.int64)
    pos[stored] = np.arange(stored.size)
    return pos.reshape(m_pad, k_pad)
