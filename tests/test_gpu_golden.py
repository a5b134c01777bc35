"""The CUDA path against the hand-derived worked examples in tests/golden/
(same fixtures as the oracle's own golden test)."""
import json
import os
from decimal import Decimal

import pytest
import torch

import swiglu_rmsnorm_add_gb300 as sra
from tests.exact import BF16, F16, F32, TORCH_DT, nearest_bits, tensor_bits, ulp_distance

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CF = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")))


def _vec(vals, fmt):
    return torch.tensor([float(v) for v in vals], dtype=torch.float64).to(TORCH_DT[fmt])


def _check(out, want_strs, fmt):
    vals = out.cpu().reshape(-1)
    got = tensor_bits(out.cpu()).reshape(-1)
    for i, w in enumerate(want_strs):
        if fmt == F32:
            wv = float(Decimal(w))
            assert abs(float(vals[i]) - wv) <= 1e-5 * abs(wv) + 1e-7, (w, float(vals[i]))
        else:
            wb = nearest_bits(Decimal(w), fmt)
            g = int(got[i])
            assert ulp_distance(g, wb, fmt) <= 1 or ((g | wb) & 0x7FFF) == 0, (w, hex(g))


@pytest.mark.parametrize("fmt", [F32, F16, BF16])
def test_golden_rmsnorm(fmt):
    for case in CF["rmsnorm"]:
        x = _vec(case["x"], fmt).reshape(1, -1).to(DEV)
        out = sra.rmsnorm(x, _vec(case["w"], fmt).to(DEV), eps=case["eps"])
        _check(out, case["out"], fmt)


@pytest.mark.parametrize("fmt", [F32, F16, BF16])
@pytest.mark.parametrize("act", ["swiglu", "reglu"])
def test_golden_glu(fmt, act):
    for case in CF[act]:
        gu = torch.cat([_vec(case["gate"], fmt), _vec(case["up"], fmt)]).reshape(1, -1).to(DEV)
        out = sra.glu(gu, act="silu" if act == "swiglu" else "relu")
        _check(out, case["out"], fmt)


@pytest.mark.parametrize("fmt", [F32, F16, BF16])
def test_golden_rope(fmt):
    for case in CF["rope"]:
        hd = case["head_dim"]
        q = _vec(case["x"], fmt).reshape(1, 1, hd).to(DEV)
        k, v = q.clone(), q.clone()
        cos = torch.tensor([case["cos"]], dtype=torch.float32, device=DEV)
        sin = torch.tensor([case["sin"]], dtype=torch.float32, device=DEV)
        cache = torch.zeros(2, 1, 1, 1, hd, dtype=TORCH_DT[fmt], device=DEV)
        z = torch.zeros(1, dtype=torch.int64, device=DEV)
        sra.rope_kv_store(q, k, v, cos, sin, z, z, cache)
        _check(q, case["out"], fmt)
        _check(cache[0], case["out"], fmt)
