"""Pins for the oracle's Q/K norm + RoPE + KV store composition.

mer.dev "AsyncT vllm 适配加速笔记（一）" section 3.3: the Q and K heads of the fused
QKV output go through the UClip / DyHT norm (section 0) before the rotary
embedding; koas-w.github.io "preformanceimprovement" section 1 fuses the
rotation with the paged cache store. The composition is checked through cases
that reduce it to one of its (separately pinned) parts: position 0 leaves only
the norm, unit parameters with open bounds leave only the rotation, and a
quarter turn moves normed values between the halves.
"""
import math

import pytest
import torch

import oracle
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.exact import TORCH_DT, F16, F32, BF16, tensor_bits

FMTS = [F32, F16, BF16]


def _inputs(fmt, T=6, seed=80):
    inp = syn.rope_inputs(T, seed, n_head=4, n_kv_head=2, head_dim=16, num_blocks=4, block_size=4, max_pos=64,
                          dtype=TORCH_DT[fmt], tables=syn.rope_tables(64, 16, 1e4))
    params = tuple(syn.uclip_params(16, True, True, seed + i)[i % 2] for i in range(4))
    return inp, params


def _uclip(x, a, g, lo=-1.0, hi=1.0):
    out = torch.empty_like(x)
    oracle.uclip(x, a, g, out, lo, hi)
    return out


@pytest.mark.parametrize("style", ["neox", "interleaved"])
@pytest.mark.parametrize("fmt", FMTS)
def test_position_zero_leaves_only_the_norm(fmt, style):
    inp, (qa, qg, ka, kg) = _inputs(fmt)
    inp["pos"].zero_()
    q0, k0, v0 = inp["q"].clone(), inp["k"].clone(), inp["v"].clone()
    n = oracle.qk_uclip_rope_kv_store(**inp, q_alpha=qa, q_gamma=qg, k_alpha=ka, k_gamma=kg, style=style)
    assert n == 0
    assert (tensor_bits(inp["q"]) == tensor_bits(_uclip(q0, qa, qg))).all()
    cache = inp["kv_cache"]
    for t in range(q0.shape[0]):
        s = int(inp["slot_mapping"][t])
        blk, off = divmod(s, 4)
        assert (tensor_bits(cache[0, blk, off]) == tensor_bits(_uclip(k0[t:t + 1], ka, kg)[0])).all()
        assert (tensor_bits(cache[1, blk, off]) == tensor_bits(v0[t])).all()     # V not normed
    assert torch.equal(inp["k"], k0)                                             # k itself untouched


@pytest.mark.parametrize("style", ["neox", "interleaved"])
@pytest.mark.parametrize("fmt", FMTS)
def test_unit_parameters_with_open_bounds_leave_only_the_rotation(fmt, style):
    inp, _ = _inputs(fmt, seed=81)
    ones = torch.ones(16)
    ref = {k: v.clone() for k, v in inp.items()}
    oracle.qk_uclip_rope_kv_store(**inp, q_alpha=ones, q_gamma=ones, k_alpha=ones, k_gamma=ones,
                                  clip_min=-math.inf, clip_max=math.inf, style=style)
    oracle.rope_kv_store(**ref, style=style)
    assert (tensor_bits(inp["q"]) == tensor_bits(ref["q"])).all()
    assert (tensor_bits(inp["kv_cache"]) == tensor_bits(ref["kv_cache"])).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_quarter_turn_moves_normed_halves(fmt):
    inp, (qa, qg, ka, kg) = _inputs(fmt, seed=82)
    inp["cos"], inp["sin"] = torch.zeros(64, 8), torch.ones(64, 8)
    q0 = inp["q"].clone()
    oracle.qk_uclip_rope_kv_store(**inp, q_alpha=qa, q_gamma=qg, k_alpha=ka, k_gamma=kg, clip_min=-0.5,
                                  clip_max=2.0)
    qn = _uclip(q0, qa, qg, -0.5, 2.0)
    assert torch.equal(inp["q"][..., :8], -qn[..., 8:])
    assert torch.equal(inp["q"][..., 8:], qn[..., :8])


def test_bad_positions_leave_q_raw():
    inp, (qa, qg, ka, kg) = _inputs(F32, seed=83)
    inp["pos"] = torch.tensor([3, -1, 5, 64, 7, 8], dtype=torch.int64)
    q0 = inp["q"].clone()
    n = oracle.qk_uclip_rope_kv_store(**inp, q_alpha=qa, q_gamma=qg, k_alpha=ka, k_gamma=kg)
    assert n == 2
    assert torch.equal(inp["q"][1], q0[1]) and torch.equal(inp["q"][3], q0[3])
    assert not torch.equal(inp["q"][0], q0[0])
