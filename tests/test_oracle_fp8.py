"""Pins for the oracle's FP8-E4M3 encode/decode (CPU only)."""

import math

import numpy as np
import torch

from oracle import fp8


def test_decode_table_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.DECODE_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert nan.sum() == 2                      # 0x7F and 0xFF
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def _brute_force(x):
    """Nearest finite E4M3 value, ties to the even code (even mantissa), +-448 saturation."""
    if math.isnan(x):
        return fp8.NAN_CODE
    best, best_err = None, None
    for c in range(256):
        v = fp8.DECODE_TABLE[c]
        if math.isnan(v):
            continue
        if (c & 0x80) != (0x80 if math.copysign(1.0, x) < 0 else 0):
            continue                           # same sign (keeps -0 for negative zero)
        err = abs(v - x)
        if best is None or err < best_err or (err == best_err and (c & 1) == 0 and (best & 1) == 1):
            best, best_err = c, err
    return best


def test_encode_matches_brute_force_nearest_even():
    rng = np.random.default_rng(7)
    vals = list(fp8.DECODE_TABLE[np.isfinite(fp8.DECODE_TABLE)])
    finite = sorted(set(abs(v) for v in vals))
    # exact midpoints between neighbours (ties), values near them, random values
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    xs = vals + mids + [m * (1 + 1e-9) for m in mids] + [m * (1 - 1e-9) for m in mids]
    xs += list(rng.standard_normal(2000) * 50) + list(rng.uniform(-1e-2, 1e-2, 500))
    xs += [460.0, 464.0, 465.0, 500.0, 1e6, -1e6, 0.0, -0.0, 2.0 ** -10, 2.0 ** -11]
    for x in xs:
        assert fp8.encode_scalar(x) == _brute_force(x), x
    assert fp8.encode_scalar(math.inf) == 0x7E and fp8.encode_scalar(-math.inf) == 0xFE
    assert fp8.encode_scalar(math.nan) == 0x7F


def test_encode_matches_torch_in_range():
    """torch's float8_e4m3fn cast rounds to nearest-even; inside +-448 it must agree."""
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 100,
                        rng.uniform(-448, 448, 20000).astype(np.float32),
                        rng.uniform(-0.02, 0.02, 5000).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = fp8.encode(x)
    inside = np.abs(x) <= 448
    assert np.array_equal(ours[inside], ref[inside])
    assert np.all(ours[x > 448] == 0x7E) and np.all(ours[x < -448] == 0xFE)


def test_quantize_divides_in_float32_then_rounds():
    rng = np.random.default_rng(9)
    x = rng.standard_normal(4000).astype(np.float16)
    for scale in (np.float32(1.0), np.float32(0.0123), np.float32(3.7)):
        q = fp8.quantize(x, scale)
        quot = torch.from_numpy(x.astype(np.float32)) / torch.tensor(scale, dtype=torch.float32)
        ref = quot.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q, ref)
        # dequantised error within half an E4M3 step (relative 2^-4) for in-range values
        deq = fp8.decode(q) * float(scale)
        xf = x.astype(np.float64)
        ok = np.abs(xf) / float(scale) <= 448
        assert np.all(np.abs(deq[ok] - xf[ok]) <= np.maximum(np.abs(xf[ok]) * 2.0 ** -4,
                                                              float(scale) * 2.0 ** -10) * (1 + 1e-6))


def test_vectorised_encode_equals_scalar_definition():
    rng = np.random.default_rng(10)
    finite = fp8.DECODE_TABLE[np.isfinite(fp8.DECODE_TABLE)]
    mags = np.sort(np.unique(np.abs(finite)))
    mids = (mags[:-1] + mags[1:]) / 2
    xs = np.concatenate([finite, mids, -mids, mids * (1 + 1e-12), mids * (1 - 1e-12),
                         rng.standard_normal(20000) * 60, rng.uniform(-3e-3, 3e-3, 5000),
                         [448.0, 464.0, -464.0, 470.0, 1e9, -1e9, 0.0, -0.0, np.inf, -np.inf, np.nan]])
    vec = fp8.encode(xs)
    ref = np.array([fp8.encode_scalar(float(v)) for v in xs], dtype=np.uint8)
    assert np.array_equal(vec, ref)
