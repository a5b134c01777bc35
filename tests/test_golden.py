"""The oracle against tests/golden/: hand-derived closed forms and the
regression hashes written by tests/golden/make_golden.py."""
import json
import os
from decimal import Decimal

import pytest
import torch

import oracle
from tests.exact import BF16, F16, F32, TORCH_DT, nearest_bits, tensor_bits

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CF = json.load(open(os.path.join(GOLD, "closed_forms.json")))
FMTS = [F32, F16, BF16]


def _vec(vals, fmt):
    return torch.tensor([float(v) for v in vals], dtype=torch.float64).to(TORCH_DT[fmt])


def _check(out, want_strs, fmt):
    got = tensor_bits(out).reshape(-1)
    for g, w in zip(got, want_strs):
        wb = nearest_bits(Decimal(w), fmt)
        assert int(g) == wb or (int(g) & 0x7FFF == 0 and wb & 0x7FFF == 0), (w, hex(int(g)), hex(wb))


@pytest.mark.parametrize("fmt", FMTS)
def test_closed_form_rmsnorm(fmt):
    for case in CF["rmsnorm"]:
        x = _vec(case["x"], fmt).reshape(1, -1)
        out = torch.empty_like(x)
        oracle.rmsnorm(x, _vec(case["w"], fmt), out, case["eps"])
        _check(out, case["out"], fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("act", ["swiglu", "reglu"])
def test_closed_form_glu(fmt, act):
    for case in CF[act]:
        gu = torch.cat([_vec(case["gate"], fmt), _vec(case["up"], fmt)]).reshape(1, -1)
        out = torch.empty(1, len(case["gate"]), dtype=TORCH_DT[fmt])
        oracle.glu(gu, out, "silu" if act == "swiglu" else "relu")
        _check(out, case["out"], fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_closed_form_rope(fmt):
    for case in CF["rope"]:
        hd = case["head_dim"]
        q = _vec(case["x"], fmt).reshape(1, 1, hd)
        k = q.clone()
        v = q.clone()
        cos = torch.tensor([case["cos"]], dtype=torch.float32)
        sin = torch.tensor([case["sin"]], dtype=torch.float32)
        cache = torch.zeros(2, 1, 1, 1, hd, dtype=TORCH_DT[fmt])
        oracle.rope_kv_store(q, k, v, cos, sin, torch.zeros(1, dtype=torch.int64),
                             torch.zeros(1, dtype=torch.int64), cache)
        _check(q, case["out"], fmt)
        _check(cache[0], case["out"], fmt)


def test_regression_hashes():
    from tests.golden.make_golden import cases
    want = json.load(open(os.path.join(GOLD, "oracle_regression.json")))["cases"]
    assert cases() == want
