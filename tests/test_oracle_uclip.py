"""Pins for the oracle's UClip / DyHT "norm".

DyHT(x) = y * clamp(a x, -1, 1) replaces every RMSNorm of the AsyncT model
(mer.dev "AsyncT vllm 适配加速笔记（一）" section 0); the uclip kernel of section
3.3 of the same page generalises it to clamp(a x, clip_min, clip_max) * g with
a scalar or per-channel alpha and gamma, over 3-D [N, H, D] views whose middle
stride is free (narrow Q/K views of a fused QKV projection).

The page's kernel evaluates in float, so the oracle keeps its two fp32
roundings (a * x, then * g) and fp32 bounds. The pins: exhaustive identity and
plain-clip cases checked against torch's own clamp, closed forms for
power-of-two scales, the special values, exact-rational brute force of the
kernel's steps (fp32 roundings by search) with per-channel parameters and
asymmetric bounds, a case where the fp32 rounding of a * x decides the output,
and stride invariance on narrow views.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.exact import BF16, F16, F32, TORCH_DT, bits_value, from_bits, nearest_bits, tensor_bits

FMTS = [F32, F16, BF16]


def _all_finite_patterns(fmt):
    """Every non-NaN pattern of a 16-bit format; 200 000 random fp32 patterns plus specials."""
    if fmt == F32:
        g = np.random.default_rng(71)
        bits = g.integers(0, 2 ** 32, size=200_000, dtype=np.int64)
        bits = np.concatenate([bits, [0, 0x80000000, 0x7F800000, 0xFF800000, 1, 0x807FFFFF]])
    else:
        bits = np.arange(0, 2 ** 16, dtype=np.int64)
    t = from_bits(bits, fmt)
    return t[~torch.isnan(t)]


def _scalar(v):
    return torch.tensor([v], dtype=torch.float32)


def _run(x, alpha, gamma, lo, hi):
    out = torch.empty_like(x)
    oracle.uclip(x, alpha, gamma, out, lo, hi)
    return out


@pytest.mark.parametrize("fmt", FMTS)
def test_unit_scales_and_open_bounds_are_the_identity(fmt):
    x = _all_finite_patterns(fmt).reshape(1, -1)
    out = _run(x, _scalar(1.0), _scalar(1.0), -math.inf, math.inf)
    assert np.array_equal(tensor_bits(out), tensor_bits(x))


@pytest.mark.parametrize("fmt", FMTS)
def test_dyht_with_unit_scales_is_torch_clamp(fmt):
    x = _all_finite_patterns(fmt).reshape(1, -1)
    out = torch.empty_like(x)
    oracle.dyht(x, _scalar(1.0), _scalar(1.0), out)
    want = torch.clamp(x, -1.0, 1.0)
    assert np.array_equal(tensor_bits(out), tensor_bits(want))


@pytest.mark.parametrize("fmt", FMTS)
def test_power_of_two_scales_closed_form(fmt):
    """alpha = 1/2, gamma = 4, bounds (-1, 1): 2x where |x| < 2, else 4 sign(x).
    alpha = -2, gamma = 1/4, bounds (-1/2, 3/4): -x/2 inside, the bound * 1/4 outside."""
    dt = TORCH_DT[fmt]
    x = torch.tensor([0.0, 0.5, -0.5, 1.75, -1.9375, 2.0, -2.0, 3.0, -100.0, 1e-3, -7e-4], dtype=dt).reshape(1, -1)
    out = _run(x, _scalar(0.5), _scalar(4.0), -1.0, 1.0)
    xd = x.double()
    want = torch.where(xd.abs() < 2, 2 * xd, 4 * torch.sign(xd)).to(dt)
    assert np.array_equal(tensor_bits(out), tensor_bits(want))
    out = _run(x, _scalar(-2.0), _scalar(0.25), -0.5, 0.75)
    v = -2 * xd
    want = torch.where(v < -0.5, torch.full_like(v, -0.125),
                       torch.where(v > 0.75, torch.full_like(v, 0.1875), v * 0.25)).to(dt)
    assert torch.equal(out, want)


@pytest.mark.parametrize("fmt", FMTS)
def test_special_values(fmt):
    dt = TORCH_DT[fmt]
    x = torch.tensor([math.nan, math.inf, -math.inf, 0.0, -0.0], dtype=dt).reshape(1, -1)
    out = _run(x, _scalar(3.0), _scalar(-2.0), -1.0, 1.0)
    assert out[0, 0].item() == -1.0 * -2.0            # a NaN product takes the lower bound, times g
    assert out[0, 1].item() == -2.0 and out[0, 2].item() == 2.0   # +-inf clip to the bounds, times g
    assert out[0, 3].item() == 0.0 and out[0, 4].item() == 0.0
    z = _run(x[:, 1:3], _scalar(0.0), _scalar(0.5), -1.0, 1.0)   # 0 * inf = NaN -> the lower bound
    assert (z == -0.5).all()
    with pytest.raises(ValueError):
        _run(x, _scalar(1.0), _scalar(1.0), 1.0, -1.0)   # lo > hi
    with pytest.raises(ValueError):
        _run(x, _scalar(1.0), _scalar(1.0), math.nan, 1.0)


def _f32(v: Fraction) -> Fraction:
    """v rounded to fp32 by the brute-force nearest search."""
    return Fraction(bits_value(nearest_bits(v, F32), F32))


def _exact_bits(x, alpha, gamma, lo, hi, fmt):
    """The page's kernel steps on exact rationals: fp32(a x), the clamp against
    fp32 bounds, fp32(* g), then the nearest value of the format."""
    N, H, D = x.shape
    xs = x.double().numpy()
    a = alpha.double().numpy()
    g = gamma.double().numpy()
    flo, fhi = _f32(Fraction(lo)), _f32(Fraction(hi))
    bits = np.zeros((N, H, D), dtype=np.int64)
    for n in range(N):
        for h in range(H):
            for d in range(D):
                v = _f32(Fraction(float(a[d if a.size > 1 else 0])) * Fraction(float(xs[n, h, d])))
                v = min(max(v, flo), fhi)
                y = _f32(v * Fraction(float(g[d if g.size > 1 else 0])))
                bits[n, h, d] = nearest_bits(y, fmt)
    return bits


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("a_pc,g_pc", [(True, True), (True, False), (False, True), (False, False)])
def test_brute_force_per_channel_asymmetric_bounds(fmt, a_pc, g_pc):
    gen = torch.Generator().manual_seed(72 + 4 * fmt + 2 * a_pc + g_pc)
    N, H, D = 3, 4, 7
    x = (torch.randn(N, H, D, generator=gen, dtype=torch.float64) * 2).to(TORCH_DT[fmt])
    alpha = (torch.rand(D if a_pc else 1, generator=gen, dtype=torch.float64) * 3 - 1).float()
    gamma = (torch.randn(D if g_pc else 1, generator=gen, dtype=torch.float64)).float()
    lo, hi = -0.7, 1.3
    out = torch.empty_like(x)
    oracle.uclip(x, alpha, gamma, out, lo, hi)
    got = tensor_bits(out).reshape(N, H, D)
    want = _exact_bits(x, alpha, gamma, lo, hi, fmt)
    zero = (from_bits(want.reshape(-1), fmt) == 0).numpy().reshape(N, H, D)
    assert np.array_equal(got[~zero], want[~zero])
    assert (out.reshape(-1)[torch.from_numpy(zero.reshape(-1))] == 0).all()


def test_channel_index_is_the_last_dimension():
    """x = 1 everywhere: out[n, h, d] = clamp(alpha_d, lo, hi) * gamma_d, the same for every n and h."""
    D = 16
    alpha = torch.tensor([(d - 8) / 4 for d in range(D)], dtype=torch.float32)   # -2 .. 1.75
    gamma = torch.tensor([2.0 ** (d % 5) for d in range(D)], dtype=torch.float32)
    x = torch.ones(3, 5, D, dtype=torch.float32)
    out = _run(x, alpha, gamma, -1.0, 1.5)
    want = torch.tensor([min(max((d - 8) / 4, -1.0), 1.5) * 2.0 ** (d % 5) for d in range(D)])
    assert torch.equal(out, want.expand(3, 5, D))


@pytest.mark.parametrize("fmt", FMTS)
def test_narrow_views_match_contiguous(fmt):
    """Q/K views of a fused [N, 16, 64] QKV buffer (middle stride 64 and token stride 1024),
    and a padded [N, 3, 64 + 8] buffer (middle stride 72): values as on a contiguous copy,
    padding and the other heads untouched."""
    dt = TORCH_DT[fmt]
    gen = torch.Generator().manual_seed(73)
    N, D = 5, 64
    alpha = torch.rand(D, generator=gen) + 0.5
    gamma = torch.randn(D, generator=gen)
    qkv = torch.randn(N, 16, D, generator=gen).to(dt)
    k = qkv[:, 12:14, :]
    ref = _run(k.contiguous(), alpha, gamma, -1.0, 1.0)
    before = qkv.clone()
    oracle.uclip(k, alpha, gamma, k, -1.0, 1.0)          # in place on the view
    assert torch.equal(tensor_bits_t(qkv[:, 12:14]), tensor_bits_t(ref))
    assert torch.equal(tensor_bits_t(qkv[:, :12]), tensor_bits_t(before[:, :12]))
    assert torch.equal(tensor_bits_t(qkv[:, 14:]), tensor_bits_t(before[:, 14:]))
    buf = torch.randn(N, 3, D + 8, generator=gen).to(dt)
    xv = buf[:, :, :D]
    obuf = torch.zeros(N, 3, D + 8, dtype=dt)
    oracle.uclip(xv, alpha, gamma, obuf[:, :, :D], -1.0, 1.0)
    assert torch.equal(tensor_bits_t(obuf[:, :, :D]), tensor_bits_t(_run(xv.contiguous(), alpha, gamma, -1.0, 1.0)))
    assert (obuf[:, :, D:] == 0).all()


def tensor_bits_t(t):
    return torch.from_numpy(tensor_bits(t))


def test_fp32_product_rounding_is_kept():
    """Inputs (found by search) where the kernel's two fp32 roundings move the fp16
    result by one ulp against a single rounding of the exact a * x * g: the oracle
    must give the fp32-step value 0xb838, not the exact value's 0xb837."""
    x = torch.tensor([[-1.8701171875]], dtype=torch.float16)
    a = torch.tensor([0.280250608921051], dtype=torch.float32)
    g = torch.tensor([1.0057204961776733], dtype=torch.float32)
    exact = Fraction(float(a[0])) * Fraction(float(x[0, 0])) * Fraction(float(g[0]))
    assert nearest_bits(exact, F16) == 0xB837
    out = _run(x, a, g, -math.inf, math.inf)
    assert int(tensor_bits(out)[0, 0]) == 0xB838
    assert int(tensor_bits(out)[0, 0]) == int(_exact_bits(x.reshape(1, 1, 1), a, g, -4.0, 4.0, F16)[0, 0, 0])
