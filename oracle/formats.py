"""8-bit number formats: E4M3 ("fn"), E8M0, and bf16 output rounding.

TEST INFRASTRUCTURE ONLY (see the package docstring).

E4M3 follows the OCP 8-bit floating point definition: 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits; exponent field 0 holds subnormals
sign * 2^-6 * m/8; there are no infinities and the single NaN pattern per sign
is S.1111.111.  The largest finite magnitude is 448 (S.1111.110).

Encoding is "round to nearest representable value, ties to the even code,
saturating to +-448" -- the cast the FP8 linear layer applies after scaling
(LoKA, section II-C and section III-C recipes; rounding and saturation fixed by
the layer definition this library implements).  Infinity saturates to +-448
and NaN maps to the NaN code of the same sign.

E8M0 is the MX v1.0 shared-scale format: 8 exponent bits, bias 127, value
2^(c-127), code 255 is NaN.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
E4M3_MAX_CODE = 0x7E
E4M3_NAN_CODE = 0x7F


def e4m3_decode_code(c: int) -> float:
    """Value of one E4M3 code, from the bit-field definition."""
    s = -1.0 if (c >> 7) & 1 else 1.0
    e = (c >> 3) & 0xF
    m = c & 0x7
    if e == 0xF and m == 0x7:
        return math.copysign(float("nan"), s)
    if e == 0:
        return s * 2.0 ** -6 * (m / 8.0)
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


# Magnitudes of the 127 non-negative finite codes 0x00..0x7E, which are
# strictly increasing in the code; index == code.
_POS = np.array([e4m3_decode_code(c) for c in range(0x7F)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_decode_code(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Decode an array of uint8 E4M3 codes to float64."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Round-to-nearest-even, saturating E4M3 encode of float values.

    ``v`` is taken exactly (float32 values convert to float64 exactly).  For a
    magnitude a below 448 the two neighbouring codes lo < a <= hi are found in
    the table of all non-negative finite values and the nearer one is taken;
    at an exact midpoint the even code wins.  a >= 448 (including infinity)
    gives 448.  The sign bit is copied, so -0.0 and negative values that round
    to zero give 0x80.
    """
    v64 = np.asarray(v, dtype=np.float64)
    a = np.abs(v64)
    nan = np.isnan(v64)
    a_fin = np.where(nan, 0.0, a)
    hi = np.clip(np.searchsorted(_POS, a_fin, side="left"), 1, 0x7E)
    lo = hi - 1
    d_lo = a_fin - _POS[lo]
    d_hi = _POS[hi] - a_fin
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a_fin >= E4M3_MAX, E4M3_MAX_CODE, mag)
    mag = np.where(nan, E4M3_NAN_CODE, mag)
    sign = np.signbit(v64).astype(np.int64) << 7
    return (mag | sign).astype(np.uint8)


def e8m0_decode(codes: np.ndarray) -> np.ndarray:
    """Value 2^(c-127) of E8M0 codes; code 255 is NaN."""
    c = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, out)


def floor_log2(a) -> np.ndarray:
    """floor(log2(a)) of non-negative float32 magnitudes, through frexp.

    frexp writes a = f * 2^p with f in [0.5, 1), so floor(log2 a) = p - 1;
    this holds for subnormals too.  Zero gives a very small sentinel (-1000),
    infinity and NaN give 128 (the exponent an fp32 Inf/NaN encodes).
    """
    a64 = np.asarray(a, dtype=np.float64)
    _, p = np.frexp(a64)
    out = p.astype(np.int64) - 1
    out = np.where(a64 == 0.0, -1000, out)
    out = np.where(~np.isfinite(a64), 128, out)
    return out


def bf16_round(v) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    A bf16 keeps 8 significant bits; the rounding quantum at binade 2^e is
    2^(e-7) for normal numbers and 2^-133 in the subnormal range.  Values
    beyond the largest bf16 become infinities.  Returns float64 values that
    are exactly representable in bf16.
    """
    v64 = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v64)
    fin = np.isfinite(v64) & (v64 != 0.0)
    x = v64[fin]
    _, p = np.frexp(x)              # |x| in [2^(p-1), 2^p)
    e = np.maximum(p - 1, -126)     # binade, clamped at the subnormal range
    q = np.ldexp(1.0, e - 7)        # quantum
    r = np.rint(x / q) * q          # x / q is exact (power-of-two division)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    out[fin] = r
    out[~fin] = v64[~fin]
    return out


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 values at the magnitude of v (float64 in, float64 out)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, p = np.frexp(np.where(a == 0.0, 1.0, a))
    e = np.maximum(p - 1, -126)
    return np.where(a == 0.0, 2.0 ** -133, np.ldexp(1.0, e - 7))
