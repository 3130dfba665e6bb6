"""Inputs planted at rounding boundaries (test infrastructure; no arithmetic of the method).

double_rounding_keys: indexer keys for the cache-append step whose fp32 quotient
x / scale (scale = amax / 448 in fp32) lands exactly on the midpoint between two
neighbouring e4m3 values, while the exact quotient lies just beside that midpoint, on the
side of the neighbour with the odd mantissa.  Rounding the fp32 quotient again (ties to
even) then gives the even neighbour; rounding the exact quotient once gives the odd one.
"""
from fractions import Fraction

import numpy as np

# midpoints between neighbouring e4m3 values, at several binades (including a
# subnormal-free small one and a large one); the side the exact quotient is planted on is
# that of the neighbour with the odd code
MIDPOINTS = [Fraction(17, 16), Fraction(19, 16), Fraction(17, 8), Fraction(27, 8),
             Fraction(25, 2), Fraction(21, 32), Fraction(100, 1)]


def _e4m3_values():
    """(value, code) of every non-negative finite e4m3 code, from the format's definition."""
    out = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out.append((v, code))
    return out


def _neighbours(mid):
    vals = _e4m3_values()
    below = max((v, c) for v, c in vals if v < mid)
    above = min((v, c) for v, c in vals if v > mid)
    return below, above


def double_rounding_keys(n, Di, seed):
    rng = np.random.default_rng(seed)
    keys = np.zeros((n, Di), np.float32)
    for i in range(n):
        while True:
            row = (rng.standard_normal(Di) * 0.05).astype(np.float32)
            amax = np.float32(rng.uniform(1.0, 2.0))
            row[0] = amax
            scale = np.float32(amax) / np.float32(448.0)
            planted = 0
            for j, mid in enumerate(MIDPOINTS):
                (lo, clo), (hi, chi) = _neighbours(mid)
                assert (lo + hi) / 2 == mid and all(v != mid for v, _ in _e4m3_values())
                side = +1 if (chi & 1) else -1      # the odd neighbour's side
                base = np.float32(float(mid) * float(scale))
                for k in range(-16, 17):
                    x = base
                    for _ in range(abs(k)):
                        x = np.nextafter(x, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
                    q32 = np.float32(x) / scale
                    exact = Fraction(float(x)) / Fraction(float(scale))
                    if Fraction(float(q32)) == mid and (exact - mid) * side > 0:
                        row[1 + j] = x
                        planted += 1
                        break
            if planted >= 3:
                keys[i] = row
                break
    return keys


def nearest_e4m3_code(value):
    """Code of the e4m3 value nearest to the exact rational `value` (ties to the even
    code, saturating at 448), found by comparing with every code: the definition."""
    sign = 0x80 if value < 0 else 0
    a = abs(value)
    best = None
    for v, c in _e4m3_values():
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1] | sign
