"""Oracle: OCP FP8-E4M3 from its bit-level definition (test infrastructure only).

[KV缓存机制解析] §8 ("混合精度缓存") stores history K/V as FP8/INT8 together with a
scaling factor.  Its snippet divides an amax by 127, which is the INT8 constant;
for E4M3 the plain reading used here is ``scale = amax / 448`` with 448 the
largest finite E4M3 value, and quantisation ``code = RNE_satfinite(x / scale)``.

E4M3 ("fn" variant of the OCP 8-bit floating point spec): 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits.  No infinities; S.1111.111 is NaN.

* exponent field e in 1..15:  value = (-1)^S * 2^(e-7) * (1 + m/8)
  (e = 15 with m = 7 is NaN, so the largest finite value is 1.75 * 2^8 = 448)
* exponent field 0:           value = (-1)^S * 2^-6 * (m/8)   (subnormals, and 0)

Encoding rounds to the nearest representable value, ties to the even mantissa,
then saturates anything beyond +-448 to +-448 ("satfinite"); NaN stays NaN.
"""

from __future__ import annotations

import math

import numpy as np

MAX_FINITE = 448.0
NAN_CODE = 0x7F


def decode_code(code: int) -> float:
    """Value of one E4M3 code (0..255) as a Python float (exact)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * math.ldexp(m / 8.0, -6)
    return sign * math.ldexp(1.0 + m / 8.0, e - 7)


DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)


def decode(codes) -> np.ndarray:
    """Vectorised decode of a uint8 array to float64 (exact)."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode_scalar(x: float) -> int:
    """E4M3 code of a real number: round to nearest, ties to even, saturate finite."""
    if math.isnan(x):
        return NAN_CODE
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0x00
    a = abs(x)
    if a == 0.0:
        return sign
    if math.isinf(a):
        return sign | 0x7E                              # saturate to 448
    if a >= math.ldexp(1.0, -6):
        # normal range: a = 2^E * f with f in [1, 2)
        E = math.floor(math.log2(a))
        # guard against log2 rounding at exact powers of two
        if math.ldexp(1.0, E) > a:
            E -= 1
        elif math.ldexp(1.0, E + 1) <= a:
            E += 1
        scaled = a / math.ldexp(1.0, E) * 8.0          # in [8, 16): 8 + mantissa
        q = _round_half_even(scaled)                    # 8 .. 16
        if q == 16:
            q = 8
            E += 1
        mant = q - 8
        efield = E + 7
        if efield > 15 or (efield == 15 and mant == 7):
            return sign | 0x7E                          # saturate to 448
        return sign | (efield << 3) | mant
    # subnormal range: a = k * 2^-9, k in [0, 8)
    k = _round_half_even(a / math.ldexp(1.0, -9))       # 0 .. 8 (8 == smallest normal)
    return sign | k


def _round_half_even(v: float) -> int:
    f = math.floor(v)
    r = v - f
    if r > 0.5:
        return f + 1
    if r < 0.5:
        return f
    return f if f % 2 == 0 else f + 1


def encode(x) -> np.ndarray:
    """Vectorised encode, same rule as ``encode_scalar``.

    The non-negative codes 0x00..0x7E are increasing in value, so for a = |x| the
    candidates are the two neighbouring table entries; the nearer wins, and on a tie
    the even code (even mantissa) wins.  Beyond 448 the code saturates to 0x7E.
    """
    xf = np.asarray(x, dtype=np.float64)
    flat = xf.reshape(-1)
    mags = DECODE_TABLE[:0x7F]                         # values of codes 0x00..0x7E
    a = np.abs(flat)
    hi = np.clip(np.searchsorted(mags, a, side="left"), 1, 0x7E)
    lo = hi - 1
    d_lo = a - mags[lo]
    d_hi = mags[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= MAX_FINITE, 0x7E, code)
    code = np.where(a == 0.0, 0, code)
    sign = np.signbit(flat).astype(np.int64) << 7
    out = (code | sign).astype(np.uint8)
    out = np.where(np.isnan(flat), NAN_CODE, out).astype(np.uint8)
    return out.reshape(xf.shape)


def quantize(x, scale) -> np.ndarray:
    """Codes for ``x`` stored with ``scale``: ``RNE_satfinite(fp32(x) / fp32(scale))``.

    The division is the single IEEE float32 division of the stored value by the
    stored scale (both float32); the quotient is then encoded exactly as above.
    """
    x32 = np.asarray(x, dtype=np.float32)
    s32 = np.asarray(scale, dtype=np.float32)
    quot = (x32 / s32).astype(np.float32)
    return encode(quot)
