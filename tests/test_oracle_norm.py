"""Pins for the oracle's RMSNorm and residual-add + RMSNorm.

Each expected value is built outside the oracle: exact arithmetic in Python
(Fraction / 80-digit Decimal) followed by the brute-force nearest-value search
in tests/exact.py. The closed forms are those of the RMSNorm definition the
pages state (koas-w.github.io "preformanceimprovement", section 3:
x.pow(2).mean(-1).add(eps).rsqrt().mul(x).mul(weight); agent.csdn.net
"使用Triton实现RMSNorm算子": rsqrt(sum_sq / D + eps)).
"""
import itertools
from decimal import Decimal
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from swiglu_rmsnorm_add_gb300 import synthetic
from tests.exact import BF16, F16, F32, TORCH_DT, dsqrt, from_bits, nearest_bits, tensor_bits

EPS = float(np.float32(1e-6))  # the fp32 value a caller passes
FMTS = [F32, F16, BF16]


def _t(vals, fmt):
    return torch.tensor(vals, dtype=torch.float64).to(TORCH_DT[fmt])


def _exact_rms_out(x_vals, w_vals, eps):
    D = len(x_vals)
    ms = sum(Decimal(v) * Decimal(v) for v in x_vals) / D
    r = 1 / dsqrt(ms + Decimal(eps))
    return [Decimal(xv) * r * Decimal(wv) for xv, wv in zip(x_vals, w_vals)]


@pytest.mark.parametrize("fmt", FMTS)
def test_constant_row_closed_form(fmt):
    # a row of constant c with w = 1 gives c / sqrt(c^2 + eps); c = 1e-3 makes eps matter
    for c in (1.0, -2.5, 1e-3, 0.1875):
        D = 37
        x = _t([c] * D, fmt).reshape(1, D)
        cq = float(x[0, 0].double())
        w = _t([1.0] * D, fmt)
        out = torch.empty_like(x)
        oracle.rmsnorm(x, w, out, EPS)
        want = nearest_bits(Decimal(cq) / dsqrt(Decimal(cq) ** 2 + Decimal(EPS)), fmt)
        assert (tensor_bits(out) == want).all(), (c, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_zero_row_is_zero(fmt):
    x = torch.zeros(3, 64, dtype=TORCH_DT[fmt])
    w = synthetic.normal((64,), 1.0, 0.1, TORCH_DT[fmt], 5, 1)
    out = torch.full_like(x, 7.0)
    oracle.rmsnorm(x, w, out, EPS)
    assert (out.double() == 0).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_one_hot_closed_form(fmt):
    # e_k * a -> a * sqrt(D) / sqrt(a^2 + D * eps) * w[k] at k, 0 elsewhere
    D, k, a = 100, 17, 3.0
    x = torch.zeros(1, D, dtype=TORCH_DT[fmt])
    x[0, k] = a
    w = synthetic.normal((D,), 1.0, 0.1, TORCH_DT[fmt], 6, 2)
    out = torch.empty_like(x)
    oracle.rmsnorm(x, w, out, EPS)
    wk = Decimal(float(w[k].double()))
    want = nearest_bits(Decimal(a) * dsqrt(Decimal(D)) / dsqrt(Decimal(a) ** 2 + D * Decimal(EPS)) * wk, fmt)
    assert int(tensor_bits(out)[0, k]) == want
    others = torch.cat([out[0, :k], out[0, k + 1:]])
    assert (others.double() == 0).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_weight_doubling_doubles_output(fmt):
    x, w = synthetic.rms_inputs(8, 96, TORCH_DT[fmt], 9)
    o1, o2 = torch.empty_like(x), torch.empty_like(x)
    oracle.rmsnorm(x, w, o1, EPS)
    oracle.rmsnorm(x, w * 2, o2, EPS)  # x2 is exact in every format
    assert torch.equal(o2, o1 * 2)


@pytest.mark.parametrize("fmt", FMTS)
def test_brute_force_tiny(fmt):
    grid = [-2.0, -0.5, 0.0, 0.25, 1.0, 3.0]
    wgrid = [1.0, -0.5, 1.5]
    for D in (1, 2, 3, 4):
        combos = list(itertools.product(grid, repeat=D))[::max(1, 6 ** D // 60)]
        for xs in combos:
            ws = [wgrid[j % 3] for j in range(D)]
            x = _t(list(xs), fmt).reshape(1, D)
            w = _t(ws, fmt)
            out = torch.empty_like(x)
            oracle.rmsnorm(x, w, out, EPS)
            want = [nearest_bits(v, fmt) for v in _exact_rms_out(xs, ws, EPS)]
            got = [int(b) for b in tensor_bits(out)[0]]
            # signed zeros compare as values
            for g, wv in zip(got, want):
                assert g == wv or (g & 0x7FFF == 0 and wv & 0x7FFF == 0) or \
                    (fmt == F32 and (g & 0x7FFFFFFF) == 0 and (wv & 0x7FFFFFFF) == 0), (xs, D)


@pytest.mark.parametrize("fmt", FMTS)
def test_random_rows_match_exact(fmt):
    """Random rows: the oracle's double result rounds to the exactly computed value."""
    x, w = synthetic.rms_inputs(4, 48, TORCH_DT[fmt], 10)
    out = torch.empty_like(x)
    oracle.rmsnorm(x, w, out, EPS)
    ob = tensor_bits(out)
    wv = [float(v) for v in w.double()]
    for r in range(4):
        xs = [float(v) for v in x[r].double()]
        want = [nearest_bits(v, fmt) for v in _exact_rms_out(xs, wv, EPS)]
        assert [int(b) for b in ob[r]] == want


def test_row_strides_and_padding_untouched():
    fmt = BF16
    rows, D, xs, os_ = 5, 40, 56, 64
    xbuf = synthetic.normal((rows, xs), 0, 1, torch.bfloat16, 11, 1)
    obuf = torch.full((rows, os_), -7.0, dtype=torch.bfloat16)
    w = synthetic.normal((D,), 1.0, 0.1, torch.bfloat16, 11, 2)
    oracle.rmsnorm(xbuf[:, :D], w, obuf[:, :D], EPS)
    assert (obuf[:, D:].double() == -7.0).all()
    dense = torch.empty(rows, D, dtype=torch.bfloat16)
    oracle.rmsnorm(xbuf[:, :D].contiguous(), w, dense, EPS)
    assert torch.equal(dense, obuf[:, :D])
    # each row is normalised by its own statistics: row r equals the one-row call
    for r in range(rows):
        one = torch.empty(1, D, dtype=torch.bfloat16)
        oracle.rmsnorm(xbuf[r:r + 1, :D].contiguous(), w, one, EPS)
        assert torch.equal(one[0], obuf[r, :D])


@pytest.mark.parametrize("fmt", FMTS)
def test_add_rmsnorm_sum_is_correctly_rounded(fmt):
    x, res, w = synthetic.add_rms_inputs(6, 33, TORCH_DT[fmt], 12)
    x0 = x.clone()
    out = torch.empty_like(x)
    oracle.add_rmsnorm(x, res, w, out, EPS)
    xb = tensor_bits(x)
    for r in range(6):
        for j in range(33):
            exact = Fraction(float(x0[r, j].double())) + Fraction(float(res[r, j].double()))
            assert int(xb[r, j]) == nearest_bits(exact, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_add_rmsnorm_out_is_norm_of_rounded_sum(fmt):
    x, res, w = synthetic.add_rms_inputs(3, 29, TORCH_DT[fmt], 13)
    out = torch.empty_like(x)
    oracle.add_rmsnorm(x, res, w, out, EPS)
    ob = tensor_bits(out)
    wv = [float(v) for v in w.double()]
    for r in range(3):
        s = [float(v) for v in x[r].double()]  # the stored, rounded sum
        want = [nearest_bits(v, fmt) for v in _exact_rms_out(s, wv, EPS)]
        assert [int(b) for b in ob[r]] == want


@pytest.mark.parametrize("fmt", FMTS)
def test_add_rmsnorm_zero_residual_is_rmsnorm(fmt):
    x, res, w = synthetic.add_rms_inputs(4, 70, TORCH_DT[fmt], 14)
    res.zero_()
    x0 = x.clone()
    out, ref = torch.empty_like(x), torch.empty_like(x)
    oracle.add_rmsnorm(x, res, w, out, EPS)
    oracle.rmsnorm(x0, w, ref, EPS)
    assert torch.equal(x, x0) and torch.equal(out, ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_add_rmsnorm_constant_rows(fmt):
    a, b, D = 0.75, -2.0, 24
    x = _t([a] * D, fmt).reshape(1, D)
    res = _t([b] * D, fmt).reshape(1, D)
    w = _t([1.0] * D, fmt)
    out = torch.empty_like(x)
    oracle.add_rmsnorm(x, res, w, out, EPS)
    s = Decimal(a + b)
    assert (x.double() == a + b).all()
    want = nearest_bits(s / dsqrt(s * s + Decimal(EPS)), fmt)
    assert (tensor_bits(out) == want).all()


def test_rows_zero_is_noop():
    x = torch.empty(0, 16, dtype=torch.bfloat16)
    w = torch.ones(16, dtype=torch.bfloat16)
    oracle.rmsnorm(x, w, torch.empty_like(x), EPS)
