"""Pins for the oracle's own format conversion (double -> fp32 / fp16 / bf16, RNE).

Checked against: exhaustive bit-pattern round trips; numpy's float16/float32
conversions and torch's bfloat16 decode (independent library routines); and an
exhaustive walk over every pair of adjacent bf16 / fp16 values with inputs at,
just below and just above each midpoint, whose correct result is known by
construction (ties go to the even pattern).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.exact import BF16, F16, F32, bits_value, nearest_bits


def _all16():
    return np.arange(0, 1 << 16, dtype=np.int64)


@pytest.mark.parametrize("fmt", [F16, BF16])
def test_decode_matches_library_for_every_pattern(fmt):
    L = oracle.lib()
    for b in range(1 << 16):
        want = bits_value(b, fmt)
        got = L.orc_decode(b, fmt)
        if math.isnan(want):
            assert math.isnan(got), hex(b)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), hex(b)


@pytest.mark.parametrize("fmt", [F16, BF16])
def test_round_trip_every_pattern(fmt):
    L = oracle.lib()
    for b in range(1 << 16):
        v = L.orc_decode(b, fmt)
        e = L.orc_encode(v, fmt)
        if math.isnan(v):
            assert math.isnan(L.orc_decode(e, fmt))
        else:
            assert e == b, (hex(b), hex(e))


def _sorted_positive_finite(fmt):
    vals = []
    for b in range(0, 1 << 15):
        v = bits_value(b, fmt)
        if math.isfinite(v):
            vals.append((v, b))
    vals.sort()
    return vals


@pytest.mark.parametrize("fmt", [F16, BF16])
def test_midpoints_and_neighbours_exhaustive(fmt):
    """For every adjacent pair (a, b): a midpoint ties to even, nudges go to the nearer."""
    L = oracle.lib()
    vals = _sorted_positive_finite(fmt)
    for (a, ba), (b, bb) in zip(vals, vals[1:]):
        if a == b:
            continue  # +0 / -0 never both appear here (positive patterns only)
        m = (a + b) / 2.0  # exact in double: both are short binary fractions
        tie = ba if ba % 2 == 0 else bb
        delta = (b - a) * 2.0 ** -20
        for v, want in ((m, tie), (m - delta, ba), (m + delta, bb), (a, ba), (b, bb)):
            for sgn in (1.0, -1.0):
                got = L.orc_encode(sgn * v, fmt)
                w = want | (0x8000 if sgn < 0 else 0)
                assert got == w, (fmt, sgn * v, hex(got), hex(w))


def test_overflow_boundaries():
    L = oracle.lib()
    # fp16: max 65504, next would be 65536; midpoint 65520 ties to "even" = 65536 -> inf
    assert L.orc_encode(65504.0, F16) == 0x7BFF
    assert L.orc_encode(65519.99, F16) == 0x7BFF
    assert L.orc_encode(65520.0, F16) == 0x7C00
    assert L.orc_encode(-1e9, F16) == 0xFC00
    # bf16: max (2 - 2^-7) * 2^127; the midpoint to 2^128 overflows
    mx = (2 - 2 ** -7) * 2.0 ** 127
    assert L.orc_encode(mx, BF16) == 0x7F7F
    assert L.orc_encode((2 - 2 ** -8) * 2.0 ** 127, BF16) == 0x7F80
    assert L.orc_encode(1e300, F32) == 0x7F800000
    assert L.orc_encode(float("inf"), BF16) == 0x7F80
    assert L.orc_encode(float("-inf"), F16) == 0xFC00


def test_subnormals():
    L = oracle.lib()
    assert L.orc_encode(2.0 ** -24, F16) == 0x0001
    assert L.orc_encode(2.0 ** -25, F16) == 0x0000          # tie -> even (0)
    assert L.orc_encode(3 * 2.0 ** -25, F16) == 0x0002      # tie between 1 and 2 -> 2
    assert L.orc_encode(2.0 ** -133, BF16) == 0x0001
    assert L.orc_encode(2.0 ** -149, F32) == 0x00000001
    assert L.orc_encode(2.0 ** -150, F32) == 0x00000000
    assert L.orc_encode(-(2.0 ** -14), F16) == 0x8400


def test_random_doubles_match_numpy_and_search():
    """fp16 / fp32 against numpy's direct float64 conversion; bf16 against the search."""
    L = oracle.lib()
    g = np.random.default_rng(7)
    mant = g.uniform(1.0, 2.0, 20000)
    expo = g.integers(-30, 20, 20000)
    vals = np.ldexp(mant, expo) * np.where(g.random(20000) < 0.5, -1.0, 1.0)
    h = vals.astype(np.float16).view(np.uint16)
    f = vals.astype(np.float32).view(np.uint32)
    for i, v in enumerate(vals):
        assert L.orc_encode(float(v), F16) == int(h[i]), v
        assert L.orc_encode(float(v), F32) == int(f[i]), v
    for v in vals[:3000]:
        assert L.orc_encode(float(v), BF16) == nearest_bits(float(v), BF16), v


def test_bf16_matches_torch_on_fp32_inputs():
    """For fp32-representable inputs torch's float->bfloat16 conversion is RNE."""
    L = oracle.lib()
    g = np.random.default_rng(8)
    bits = g.integers(0, 0x7F7FFFFF, 50000, dtype=np.int64).astype(np.uint32)
    f = bits.view(np.float32)
    tb = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    for i in range(len(f)):
        assert L.orc_encode(float(f[i]), BF16) == int(tb[i]), float(f[i])


def test_nan_stays_nan():
    L = oracle.lib()
    for fmt in (F32, F16, BF16):
        assert math.isnan(L.orc_decode(L.orc_encode(float("nan"), fmt), fmt))


def test_search_helper_agrees_with_numpy():
    """The test-side search itself, against numpy on a few values (sanity of the pin)."""
    for v in (1.0, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 0.1, -3.3e-6, 6.0e4):
        assert nearest_bits(v, F16) == int(np.float16(v).view(np.uint16))
        assert nearest_bits(v, F32) == int(np.float32(v).view(np.uint32))
