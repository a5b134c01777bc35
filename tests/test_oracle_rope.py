"""Pins for the oracle's fused neox RoPE + paged KV-cache store.

Semantics from koas-w.github.io "preformanceimprovement", section 1 (rotate
halves: slice, negate, concatenate; Q written back, K_rot and V scattered
through slot_mapping; kv_head = head // (n_head / n_kv_head)) and mer.dev
"AsyncT vllm 适配加速笔记（一）" section 1.1 (cache [2, num_blocks, block_size,
num_kv_heads, head_size], index 0 = K, 1 = V).

Expected values come from synthetic tables with known angles (0, 90 degrees,
an arbitrary (c, s) pair) evaluated in exact rational arithmetic, from torch
indexing of the cache tensor, and from norm preservation with real tables.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from swiglu_rmsnorm_add_gb300 import synthetic
from tests.exact import BF16, F16, F32, TORCH_DT, nearest_bits, tensor_bits


def _case(T=5, n_head=4, n_kv=2, hd=8, nb=4, bs=2, max_pos=16, fmt=BF16, seed=3):
    dt = TORCH_DT[fmt]
    q = synthetic.normal((T, n_head, hd), 0, 1, dt, seed, 1)
    k = synthetic.normal((T, n_kv, hd), 0, 1, dt, seed, 2)
    v = synthetic.normal((T, n_kv, hd), 0, 1, dt, seed, 3)
    pos = synthetic.positions(T, max_pos, seed, 4)
    slot = synthetic.slots(T, nb * bs, seed, 5)
    cache = synthetic.sentinel_cache((2, nb, bs, n_kv, hd), dt)
    return q, k, v, pos, slot, cache


def _tables(max_pos, h, c, s):
    return (torch.full((max_pos, h), c, dtype=torch.float32),
            torch.full((max_pos, h), s, dtype=torch.float32))


@pytest.mark.parametrize("fmt", [F32, F16, BF16])
def test_position_zero_is_identity(fmt):
    q, k, v, pos, slot, cache = _case(fmt=fmt)
    cos, sin = synthetic.rope_tables(16, 8, 1e6)
    pos.zero_()
    q0 = q.clone()
    n = oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    assert n == 0
    assert torch.equal(tensor_bits_t(q), tensor_bits_t(q0))
    for t in range(q.shape[0]):
        s = int(slot[t])
        assert torch.equal(cache[0, s // 2, s % 2], k[t])
        assert torch.equal(cache[1, s // 2, s % 2], v[t])


def tensor_bits_t(t):
    return torch.from_numpy(tensor_bits(t))


@pytest.mark.parametrize("fmt", [F32, F16, BF16])
def test_ninety_degrees_maps_a_b_to_minus_b_a(fmt):
    q, k, v, pos, slot, cache = _case(fmt=fmt)
    cos, sin = _tables(16, 4, 0.0, 1.0)
    q0, h = q.clone(), 4
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    assert torch.equal(q[..., :h], -q0[..., h:])
    assert torch.equal(q[..., h:], q0[..., :h])
    for t in range(q.shape[0]):
        s = int(slot[t])
        kc = cache[0, s // 2, s % 2]
        assert torch.equal(kc[:, :h], -k[t][:, h:]) and torch.equal(kc[:, h:], k[t][:, :h])


@pytest.mark.parametrize("fmt", [F32, F16, BF16])
def test_general_angle_exact(fmt):
    """cos = 0.75, sin = 0.5 (a valid table value pair for the linear formula)."""
    q, k, v, pos, slot, cache = _case(fmt=fmt, T=3)
    cos, sin = _tables(16, 4, 0.75, 0.5)
    q0 = q.clone()
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    c, s, h = Fraction(3, 4), Fraction(1, 2), 4
    qb = tensor_bits(q)
    for t in range(3):
        for hd in range(q.shape[1]):
            x = [Fraction(float(val)) for val in q0[t, hd].double()]
            for i in range(h):
                assert qb[t, hd, i] == nearest_bits(x[i] * c - x[i + h] * s, fmt)
                assert qb[t, hd, i + h] == nearest_bits(x[i + h] * c + x[i] * s, fmt)


def test_half_split_pairing_not_interleaved():
    q, k, v, pos, slot, cache = _case(T=1, n_head=1, n_kv=1, hd=8)
    q.zero_()
    q[0, 0, 0] = 1.0
    cos, sin = _tables(16, 4, 0.0, 1.0)
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    # e_0 rotates into the partner at index h = 4, not index 1
    want = torch.zeros(8, dtype=torch.bfloat16)
    want[4] = 1.0
    assert torch.equal(q[0, 0], want)


def test_each_token_uses_its_own_position_row():
    T, hd, max_pos = 6, 8, 16
    q, k, v, pos, slot, cache = _case(T=T, hd=hd, max_pos=max_pos)
    pos = torch.tensor([0, 5, 9, 5, 15, 2], dtype=torch.int64)
    cos = torch.ones(max_pos, 4, dtype=torch.float32)
    sin = torch.zeros(max_pos, 4, dtype=torch.float32)
    cos[5], sin[5] = 0.0, 1.0     # 90 degrees at position 5 only
    cos[9], sin[9] = -1.0, 0.0    # 180 degrees at position 9
    q0 = q.clone()
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    for t in range(T):
        p = int(pos[t])
        if p == 5:
            assert torch.equal(q[t, :, :4], -q0[t, :, 4:])
        elif p == 9:
            assert torch.equal(q[t], -q0[t])
        else:
            assert torch.equal(q[t], q0[t])


def test_pair_norm_preserved_fp32():
    q, k, v, pos, slot, cache = _case(fmt=F32, T=8, n_head=6, n_kv=2, hd=128, nb=8, bs=4,
                                      max_pos=32768)
    cos, sin = synthetic.rope_tables(32768, 128, 1e6)
    pos = synthetic.positions(8, 32768, 4, 9)
    q0 = q.clone().double()
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    q1 = q.double()
    n0 = q0[..., :64] ** 2 + q0[..., 64:] ** 2
    n1 = q1[..., :64] ** 2 + q1[..., 64:] ** 2
    assert torch.allclose(n1, n0, rtol=2e-6, atol=1e-12)
    assert not torch.equal(q1, q0)


def test_slot_placement_brute_force_and_sentinels():
    nb, bs, n_kv, hd, T = 4, 2, 2, 4, 5
    q, k, v, pos, slot, cache = _case(T=T, n_head=2, n_kv=n_kv, hd=hd, nb=nb, bs=bs)
    cos, sin = _tables(16, 2, 1.0, 0.0)  # identity rotation: K lands unchanged
    sentinel = cache.clone()
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    touched = torch.zeros(2, nb, bs, dtype=torch.bool)
    for t in range(T):
        s = int(slot[t])
        b, o = s // bs, s % bs
        assert torch.equal(cache[0, b, o], k[t]) and torch.equal(cache[1, b, o], v[t])
        touched[:, b, o] = True
    untouched = ~touched
    a = tensor_bits(cache).reshape(2, nb, bs, -1)
    sb = tensor_bits(sentinel).reshape(2, nb, bs, -1)
    assert (a[untouched.numpy()] == sb[untouched.numpy()]).all()
    assert (sb == 0xDEAD).all()


def test_v_is_bit_copy_and_gqa_heads():
    q, k, v, pos, slot, cache = _case(T=4, n_head=6, n_kv=2, hd=8, nb=4, bs=2)
    cos, sin = synthetic.rope_tables(16, 8, 1e4)
    pos = torch.tensor([3, 7, 11, 1], dtype=torch.int64)
    q0 = q.clone()
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    for t in range(4):
        s = int(slot[t])
        assert torch.equal(tensor_bits_t(cache[1, s // 2, s % 2]), tensor_bits_t(v[t]))
        # every Q head is rotated (GQA: 3 Q heads share each KV head, all rotate)
        assert all(not torch.equal(q[t, hh], q0[t, hh]) for hh in range(6))


def test_padding_slot_and_errors():
    T, nb, bs = 4, 4, 2
    q, k, v, pos, slot, cache = _case(T=T, nb=nb, bs=bs)
    cos, sin = synthetic.rope_tables(16, 8, 1e4)
    pos = torch.tensor([1, 2, 16, -1], dtype=torch.int64)       # tokens 2, 3: bad positions
    slot = torch.tensor([-1, 8, 3, 5], dtype=torch.int64)       # token 0 padding, token 1 out of range
    q0, c0 = q.clone(), cache.clone()
    n = oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    assert n == 3  # token 1 slot, tokens 2 and 3 positions
    assert torch.equal(tensor_bits_t(cache), tensor_bits_t(c0))  # nothing written
    assert not torch.equal(q[0], q0[0]) and not torch.equal(q[1], q0[1])  # valid positions rotate
    assert torch.equal(q[2], q0[2]) and torch.equal(q[3], q0[3])


def test_token_stride_padding_untouched():
    T, n_head, n_kv, hd = 3, 2, 1, 8
    qkv = synthetic.normal((T, (n_head + 2 * n_kv) * hd), 0, 1, torch.bfloat16, 5, 1)
    q = qkv[:, :n_head * hd].view(T, n_head, hd)
    k = qkv[:, n_head * hd:(n_head + n_kv) * hd].view(T, n_kv, hd)
    v = qkv[:, (n_head + n_kv) * hd:].view(T, n_kv, hd)
    before = qkv.clone()
    cache = synthetic.sentinel_cache((2, 2, 2, n_kv, hd))
    cos, sin = synthetic.rope_tables(16, hd, 1e4)
    pos = torch.tensor([1, 2, 3], dtype=torch.int64)
    slot = torch.tensor([0, 3, 1], dtype=torch.int64)
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)
    assert torch.equal(qkv[:, n_head * hd:], before[:, n_head * hd:])  # k, v untouched
    dense = before[:, :n_head * hd].contiguous().view(T, n_head, hd)
    cache2 = synthetic.sentinel_cache((2, 2, 2, n_kv, hd))
    oracle.rope_kv_store(dense, before[:, n_head * hd:(n_head + n_kv) * hd].contiguous().view(T, n_kv, hd),
                         before[:, (n_head + n_kv) * hd:].contiguous().view(T, n_kv, hd),
                         cos, sin, pos, slot, cache2)
    assert torch.equal(dense, q) and torch.equal(tensor_bits_t(cache2), tensor_bits_t(cache))


def test_duplicate_slots_rejected():
    q, k, v, pos, slot, cache = _case(T=3)
    cos, sin = synthetic.rope_tables(16, 8, 1e4)
    slot = torch.tensor([1, 1, 2], dtype=torch.int64)
    with pytest.raises(ValueError):
        oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache)


# ------------------------------------------------------------ interleaved (GPT-J) pairing
# m.lsln.cn "21 个算子" section 2.3 pairs each even dimension with the next odd one.

def test_interleaved_partner_is_the_next_dimension():
    q, k, v, pos, slot, cache = _case(T=1, n_head=1, n_kv=1, hd=8)
    q.zero_()
    q[0, 0, 0] = 1.0
    cos, sin = _tables(16, 4, 0.0, 1.0)
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache, style="interleaved")
    want = torch.zeros(8, dtype=torch.bfloat16)
    want[1] = 1.0   # e_0 rotates into dimension 1, not h = 4
    assert torch.equal(q[0, 0], want)


@pytest.mark.parametrize("fmt", [F32, F16, BF16])
def test_interleaved_general_angle_exact(fmt):
    q, k, v, pos, slot, cache = _case(fmt=fmt, T=3)
    # per-pair angles: pair i uses table column i
    cos = torch.tensor([[0.75, 0.5, -0.25, 1.0]] * 16, dtype=torch.float32)
    sin = torch.tensor([[0.5, -0.125, 0.875, 0.0]] * 16, dtype=torch.float32)
    q0, k0 = q.clone(), k.clone()
    oracle.rope_kv_store(q, k, v, cos, sin, pos, slot, cache, style="interleaved")
    qb, cb = tensor_bits(q), tensor_bits(cache)
    for t in range(3):
        for hd in range(q.shape[1]):
            x = [Fraction(float(val)) for val in q0[t, hd].double()]
            for i in range(4):
                c, s = Fraction(float(cos[0, i])), Fraction(float(sin[0, i]))
                assert qb[t, hd, 2 * i] == nearest_bits(x[2 * i] * c - x[2 * i + 1] * s, fmt)
                assert qb[t, hd, 2 * i + 1] == nearest_bits(x[2 * i + 1] * c + x[2 * i] * s, fmt)
        sl = int(slot[t])
        for kvh in range(k.shape[1]):
            x = [Fraction(float(val)) for val in k0[t, kvh].double()]
            for i in range(4):
                c, s = Fraction(float(cos[0, i])), Fraction(float(sin[0, i]))
                assert cb[0, sl // 2, sl % 2, kvh, 2 * i] == nearest_bits(x[2 * i] * c - x[2 * i + 1] * s, fmt)


def test_interleaved_is_a_permutation_of_neox():
    """Interleaved RoPE equals neox RoPE applied to the even/odd de-interleaved head."""
    T, nh, nkv, hd = 4, 3, 1, 16
    q, k, v, pos, slot, cache = _case(T=T, n_head=nh, n_kv=nkv, hd=hd, max_pos=64, fmt=F32)
    cos, sin = synthetic.rope_tables(64, hd, 1e4)
    perm = torch.cat([torch.arange(0, hd, 2), torch.arange(1, hd, 2)])  # [evens | odds]
    qa = q.clone()
    oracle.rope_kv_store(qa, k.clone(), v.clone(), cos, sin, pos, slot, cache.clone(), style="interleaved")
    qb = q[..., perm].contiguous()
    oracle.rope_kv_store(qb, k[..., perm].contiguous(), v[..., perm].contiguous(), cos, sin, pos, slot,
                         cache.clone())
    assert torch.equal(qa[..., perm], qb)
