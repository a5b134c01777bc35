"""Exact reference values for the oracle's pins (test-only helpers).

``nearest_bits`` rounds an exact value (Fraction or Decimal) to a format by
brute force: it decodes a handful of neighbouring bit patterns with torch /
numpy, measures each one's exact distance to the value, and keeps the nearest
(ties to the even pattern). It shares no code or algorithm with the oracle's
own rounding, which rescales and inspects the fraction.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

getcontext().prec = 80

F32, F16, BF16 = 0, 1, 2
TORCH_DT = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
MAXFIN = {F32: Fraction(2 ** 24 - 1) * Fraction(2) ** (127 - 23),
          F16: Fraction(65504),
          BF16: Fraction(2 ** 8 - 1) * Fraction(2) ** (127 - 7)}


def bits_value(bits: int, fmt: int) -> float:
    """Exact value of a bit pattern, decoded by numpy (fp16, fp32) or torch (bf16)."""
    if fmt == F16:
        return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])
    if fmt == F32:
        return float(np.array([bits], dtype=np.uint32).view(np.float32)[0])
    t = torch.tensor([bits - 0x10000 if bits >= 0x8000 else bits], dtype=torch.int16)
    return float(t.view(torch.bfloat16).to(torch.float64)[0])


def _ordered(bits: int, fmt: int) -> int:
    width = 32 if fmt == F32 else 16
    sign = 1 << (width - 1)
    return -(bits & (sign - 1)) if bits & sign else bits


def _from_ordered(o: int, fmt: int) -> int:
    width = 32 if fmt == F32 else 16
    return ((1 << (width - 1)) | (-o)) if o < 0 else o


def ulp_distance(a_bits: int, b_bits: int, fmt: int) -> int:
    """Number of representable steps between two finite patterns (+0 and -0 are 0 apart)."""
    return abs(_ordered(a_bits, fmt) - _ordered(b_bits, fmt))


def _estimate_bits(x: float, fmt: int) -> int:
    if fmt == F16:
        return int(np.array([x], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
    f32 = int(np.array([x], dtype=np.float64).astype(np.float32).view(np.uint32)[0])
    return f32 if fmt == F32 else f32 >> 16


def nearest_bits(value, fmt: int) -> int:
    """Bits of the representable value nearest to ``value`` (ties to even), by search."""
    q = Fraction(value) if not isinstance(value, Decimal) else Fraction(value)
    if abs(q) > MAXFIN[fmt] + (MAXFIN[fmt] - Fraction(bits_value(_prev_max(fmt), fmt))) / 2:
        inf = {F32: 0x7F800000, F16: 0x7C00, BF16: 0x7F80}[fmt]
        sign = {F32: 0x80000000, F16: 0x8000, BF16: 0x8000}[fmt]
        return inf | (sign if q < 0 else 0)
    est = _estimate_bits(float(q), fmt)
    o = _ordered(est, fmt)
    best = None
    for d in range(-3, 4):
        b = _from_ordered(o + d, fmt)
        v = bits_value(b, fmt)
        if math.isinf(v) or math.isnan(v):
            continue
        dist = abs(Fraction(v) - q)
        key = (dist, b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def _prev_max(fmt: int) -> int:
    return {F32: 0x7F7FFFFE, F16: 0x7BFE, BF16: 0x7F7E}[fmt]


def dsqrt(x) -> Decimal:
    return Decimal(x).sqrt() if not isinstance(x, Decimal) else x.sqrt()


def dexp(x) -> Decimal:
    return Decimal(x).exp() if not isinstance(x, Decimal) else x.exp()


def tensor_bits(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a CPU tensor as int64 numpy array."""
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().astype(np.int64) & 0xFFFFFFFF
    return t.view(torch.int16).numpy().astype(np.int64) & 0xFFFF


def from_bits(bits, fmt: int, shape=None) -> torch.Tensor:
    a = np.asarray(bits, dtype=np.int64)
    if fmt == F32:
        t = torch.from_numpy(a.astype(np.uint32).view(np.int32).copy()).view(torch.float32)
    else:
        t = torch.from_numpy(a.astype(np.uint16).view(np.int16).copy()).view(TORCH_DT[fmt])
    return t.reshape(shape) if shape is not None else t
