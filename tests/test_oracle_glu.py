"""Pins for the oracle's SwiGLU / ReGLU over a fused gate_up tensor.

silu(g) * u with silu(g) = g / (1 + e^-g) (koas-w.github.io
"preformanceimprovement" section 2, F.silu(gate) * up); relu(g) * u
(mer.dev "AsyncT vllm 适配加速笔记（一）" section 3.3, relu_and_mul); gate is the
first I columns of gate_up, up the last I (my-blog "Triton矩阵乘算子融合",
the fused gate_up_proj of width 2 * 14336).
Expected values: 80-digit Decimal exp, exact Fraction products, then the
nearest-value search of tests/exact.py.
"""
from decimal import Decimal
from fractions import Fraction

import pytest
import torch

import oracle
from swiglu_rmsnorm_add_gb300 import synthetic
from tests.exact import BF16, F16, F32, TORCH_DT, dexp, nearest_bits, tensor_bits

FMTS = [F32, F16, BF16]


def _gu(g_vals, u_vals, fmt):
    g = torch.tensor(g_vals, dtype=torch.float64).to(TORCH_DT[fmt])
    u = torch.tensor(u_vals, dtype=torch.float64).to(TORCH_DT[fmt])
    return torch.cat([g, u]).reshape(1, -1)


def _silu_exact(g: float) -> Decimal:
    return Decimal(g) / (1 + dexp(-Decimal(g)))


@pytest.mark.parametrize("fmt", FMTS)
def test_silu_known_points(fmt):
    gs = [0.0, 1.0, -1.0, 2.5, -4.0, 20.0, -20.0, 0.125]
    us = [3.0, 1.0, 1.0, -0.5, 2.0, 1.5, 1.5, -8.0]
    gu = _gu(gs, us, fmt)
    out = torch.empty(1, len(gs), dtype=TORCH_DT[fmt])
    oracle.swiglu(gu, out)
    gq = [float(v) for v in gu[0, :len(gs)].double()]
    uq = [float(v) for v in gu[0, len(gs):].double()]
    ob = tensor_bits(out)[0]
    for j, (g, u) in enumerate(zip(gq, uq)):
        want = nearest_bits(_silu_exact(g) * Decimal(u), fmt)
        assert int(ob[j]) == want or (want & 0x7FFF == 0 and int(ob[j]) & 0x7FFF == 0), (g, u)
    assert float(out[0, 0]) == 0.0            # silu(0) = 0
    # silu(1) = 1 / (1 + e^-1) = 0.7310585786300049...
    assert abs(float(out[0, 1]) - 0.7310585786300049) <= 0.7310585786300049 * 2 ** -7


@pytest.mark.parametrize("fmt", FMTS)
def test_zero_up_gives_zero(fmt):
    gu = synthetic.glu_inputs(3, 40, TORCH_DT[fmt], 4)
    gu[:, 40:] = 0
    out = torch.empty(3, 40, dtype=TORCH_DT[fmt])
    oracle.swiglu(gu, out)
    assert (out.double() == 0).all()


def test_silu_symmetry_fp32():
    # silu(g) - silu(-g) = g  (since sigma(-g) = 1 - sigma(g))
    gs = [0.3, 1.7, -2.2, 5.0, 0.01]
    gu = _gu(gs + [-g for g in gs], [1.0] * 10, F32)
    out = torch.empty(1, 10, dtype=torch.float32)
    oracle.swiglu(gu, out)
    d = (out[0, :5] - out[0, 5:]).double()
    assert torch.allclose(d, torch.tensor(gs, dtype=torch.float64), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("fmt", FMTS)
def test_brute_force_random(fmt):
    gu = synthetic.glu_inputs(4, 24, TORCH_DT[fmt], 5)
    out = torch.empty(4, 24, dtype=TORCH_DT[fmt])
    oracle.swiglu(gu, out)
    ob = tensor_bits(out)
    for t in range(4):
        for j in range(24):
            g = float(gu[t, j].double())
            u = float(gu[t, 24 + j].double())
            assert int(ob[t, j]) == nearest_bits(_silu_exact(g) * Decimal(u), fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_reglu_bit_exact(fmt):
    gu = synthetic.glu_inputs(5, 31, TORCH_DT[fmt], 6)
    out = torch.empty(5, 31, dtype=TORCH_DT[fmt])
    oracle.reglu(gu, out)
    ob = tensor_bits(out)
    for t in range(5):
        for j in range(31):
            g = Fraction(float(gu[t, j].double()))
            u = Fraction(float(gu[t, 31 + j].double()))
            want = nearest_bits(max(g, Fraction(0)) * u, fmt)
            got = int(ob[t, j])
            assert got == want or (got & 0x7FFF == 0 and want & 0x7FFF == 0) or \
                (fmt == F32 and got & 0x7FFFFFFF == 0 and want & 0x7FFFFFFF == 0)


def test_gate_is_first_half_up_is_second():
    # g = 20, u = 3 -> ~60 ; swapped (g = 3, u = 20) would give ~57.2
    gu = _gu([20.0], [3.0], F32)
    out = torch.empty(1, 1, dtype=torch.float32)
    oracle.swiglu(gu, out)
    assert abs(float(out) - 20.0 * 3.0 / (1 + 2.061153622438558e-09)) < 1e-4
    oracle.reglu(_gu([-1.0], [5.0], F32), out)
    assert float(out) == 0.0
    oracle.reglu(_gu([5.0], [-1.0], F32), out)
    assert float(out) == -5.0


def test_strided_rows():
    T, I = 3, 16
    buf = synthetic.normal((T, 2 * I + 8), 0, 1, torch.bfloat16, 7, 1)
    obuf = torch.full((T, I + 5), 9.0, dtype=torch.bfloat16)
    oracle.swiglu(buf[:, :2 * I], obuf[:, :I])
    ref = torch.empty(T, I, dtype=torch.bfloat16)
    oracle.swiglu(buf[:, :2 * I].contiguous(), ref)
    assert torch.equal(ref, obuf[:, :I]) and (obuf[:, I:].double() == 9.0).all()
