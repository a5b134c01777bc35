"""Pins for the oracle's linear layer and the norm / GLU prologue compositions.

m.lsln.cn 21-operator article section 2.2: the RMSNorm before the attention
feeds qkv_proj directly, so the norm can run as the projection's prologue
(3-5 % of the step); the same holds for the activation before the MLP's down
projection. y[b, n] = sum_k h[b, k] * W[n, k] with W in nn.Linear's [out, in]
layout, h the normed (or activated) rows rounded to the dtype as the separate
kernel would store them.

Pins: an identity W returns h bit for bit; one-hot rows of W select columns of
h; exact rational brute force (Fraction sums, nearest-value search) on small
non-square cases; doubling W doubles y exactly; the compositions equal their
two steps.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.exact import BF16, F16, F32, TORCH_DT, nearest_bits, tensor_bits

FMTS = [F32, F16, BF16]


def _lin(h, W):
    y = torch.empty(h.shape[0], W.shape[0], dtype=h.dtype)
    oracle.linear(h, W, y)
    return y


@pytest.mark.parametrize("fmt", FMTS)
def test_identity_weight_returns_h(fmt):
    h = syn.normal((5, 24), 0, 1, TORCH_DT[fmt], 60, 1)
    W = torch.eye(24, dtype=TORCH_DT[fmt])
    assert (tensor_bits(_lin(h, W)) == tensor_bits(h)).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_one_hot_rows_select_columns(fmt):
    h = syn.normal((3, 16), 0, 1, TORCH_DT[fmt], 61, 1)
    sel = [5, 0, 15, 5, 9, 2, 11]
    W = torch.zeros(len(sel), 16, dtype=TORCH_DT[fmt])
    for n, k in enumerate(sel):
        W[n, k] = 1.0
    y = _lin(h, W)
    assert (tensor_bits(y) == tensor_bits(h[:, sel].contiguous())).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_exact_rational_brute_force(fmt):
    h = syn.normal((3, 11), 0, 1, TORCH_DT[fmt], 62, 1)
    W = syn.normal((7, 11), 0, 0.5, TORCH_DT[fmt], 62, 2)
    y = _lin(h, W)
    hd, Wd = h.double().numpy(), W.double().numpy()
    for b in range(3):
        for n in range(7):
            exact = sum(Fraction(float(hd[b, k])) * Fraction(float(Wd[n, k])) for k in range(11))
            assert int(tensor_bits(y[b, n:n + 1])[0]) == nearest_bits(exact, fmt), (b, n)


@pytest.mark.parametrize("fmt", FMTS)
def test_doubling_w_doubles_y(fmt):
    h = syn.normal((4, 32), 0, 1, TORCH_DT[fmt], 63, 1)
    W = syn.normal((9, 32), 0, 0.2, TORCH_DT[fmt], 63, 2)
    assert (tensor_bits(_lin(h, W * 2)) == tensor_bits(_lin(h, W) * 2)).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_compositions_are_their_two_steps(fmt):
    dt = TORCH_DT[fmt]
    x = syn.normal((4, 64), 0, 1, dt, 64, 1)
    w = syn.normal((64,), 1, 0.1, dt, 64, 2)
    W = syn.normal((24, 64), 0, 0.1, dt, 64, 3)
    y = torch.empty(4, 24, dtype=dt)
    oracle.rmsnorm_linear(x, w, W, y, 1e-6)
    h = torch.empty_like(x)
    oracle.rmsnorm(x, w, h, 1e-6)
    assert (tensor_bits(y) == tensor_bits(_lin(h, W))).all()
    gu = syn.normal((4, 128), 0, 1, dt, 64, 4)
    for act in ("silu", "relu"):
        oracle.glu_linear(gu, W, y, act)
        a = torch.empty(4, 64, dtype=dt)
        oracle.glu(gu, a, act)
        assert (tensor_bits(y) == tensor_bits(_lin(a, W))).all()
