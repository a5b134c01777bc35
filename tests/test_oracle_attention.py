"""Pins for the oracle's decode attention over the paged KV cache.

o[b, h] = sum_t softmax(scale * q[b, h] . K_t) V_t over request b's first
seq_lens[b] tokens, token t in block block_table[b, t // block_size] at offset
t % block_size, kv head h // (n_head / n_kv_head) (mer.dev "AsyncT vllm 适配加速笔记
（一）" sections 1.1 and 3.1; m.lsln.cn 21-operator article sections 2.1 and 5.3:
qk_score, scale + softmax and pv_agg over the cache read).

Pins: one token gives its V row; equal keys give the plain mean of V (exact
rational mean); a dominant key gives its V row exactly; 80-digit Decimal
softmax on small random cases; block-table permutation invariance with the
cache blocks moved to match; bytes beyond seq_len never read; the GQA head map;
q and scale trading a factor of two; bad entries skipped and counted.
"""
from decimal import Decimal
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.exact import BF16, F16, F32, TORCH_DT, dexp, nearest_bits, tensor_bits

FMTS = [F32, F16, BF16]


def _case(fmt, B=2, n_head=4, n_kv=2, hd=8, nb=8, bs=4, max_blocks=4, seed=90, lens=None):
    dt = TORCH_DT[fmt]
    q = syn.normal((B, n_head, hd), 0, 1, dt, seed, 1)
    cache = syn.normal((2, nb, bs, n_kv, hd), 0, 1, dt, seed, 2)
    perm = syn.rng(seed, 3).permutation(nb)[:B * max_blocks].reshape(B, max_blocks)
    table = torch.from_numpy(perm.astype(np.int32))
    if lens is None:
        lens = syn.rng(seed, 4).integers(1, max_blocks * bs + 1, size=B)
    seq = torch.tensor(lens, dtype=torch.int32)
    return q, cache, table, seq


def _run(q, cache, table, seq, scale=None):
    out = torch.empty_like(q)
    n = oracle.paged_decode_attention(q, cache, table, seq, out, scale)
    return out, n


def _rows(cache, table, seq, b, kvh, plane):
    bs = cache.shape[2]
    return [cache[plane, int(table[b, t // bs]), t % bs, kvh] for t in range(int(seq[b]))]


@pytest.mark.parametrize("fmt", FMTS)
def test_one_token_gives_its_value_row(fmt):
    q, cache, table, _ = _case(fmt)
    seq = torch.tensor([1, 1], dtype=torch.int32)
    out, n = _run(q, cache, table, seq)
    assert n == 0
    for b in range(2):
        for h in range(4):
            v0 = _rows(cache, table, seq, b, h // 2, 1)[0]
            assert (tensor_bits(out[b, h]) == tensor_bits(v0)).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_equal_keys_give_the_mean_of_values(fmt):
    q, cache, table, seq = _case(fmt, lens=[13, 7])
    cache[0] = cache[0, 0, 0]          # every key the same row
    out, _ = _run(q, cache, table, seq)
    for b in range(2):
        for h in range(4):
            vs = _rows(cache, table, seq, b, h // 2, 1)
            for d in range(8):
                mean = sum(Fraction(float(v[d])) for v in vs) / len(vs)
                assert int(tensor_bits(out[b, h, d:d + 1])[0]) == nearest_bits(mean, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_dominant_key_gives_its_value_row(fmt):
    q, cache, table, seq = _case(fmt, lens=[16, 9])
    q.zero_()
    q[:, :, 0] = 1.0
    j = 5                                # token 5 of every request dominates by > 900
    for b in range(2):
        cache[0, int(table[b, j // 4]), j % 4, :, 0] = 1000.0
    out, _ = _run(q, cache, table, seq, scale=1.0)
    for b in range(2):
        for h in range(4):
            vj = _rows(cache, table, seq, b, h // 2, 1)[j]
            assert (tensor_bits(out[b, h]) == tensor_bits(vj)).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_decimal_softmax_small_cases(fmt):
    q, cache, table, seq = _case(fmt, seed=91)
    scale = 0.3
    out, _ = _run(q, cache, table, seq, scale)
    for b in range(2):
        for h in range(4):
            ks = _rows(cache, table, seq, b, h // 2, 0)
            vs = _rows(cache, table, seq, b, h // 2, 1)
            qd = [Decimal(float(x)) for x in q[b, h]]
            s = [Decimal(scale) * sum(qd[d] * Decimal(float(k[d])) for d in range(8)) for k in ks]
            m = max(s)
            p = [dexp(x - m) for x in s]
            den = sum(p)
            for d in range(8):
                o = sum(pi * Decimal(float(v[d])) for pi, v in zip(p, vs)) / den
                assert int(tensor_bits(out[b, h, d:d + 1])[0]) == nearest_bits(o, fmt), (b, h, d)


@pytest.mark.parametrize("fmt", FMTS)
def test_block_table_permutation_and_unused_slots(fmt):
    """Moving cache blocks and the table entries that point at them changes nothing;
    neither do the slots past seq_len in the last block."""
    q, cache, table, seq = _case(fmt, lens=[14, 6], seed=92)
    out, _ = _run(q, cache, table, seq)
    perm = torch.from_numpy(syn.rng(92, 9).permutation(8))
    inv = torch.argsort(perm)
    cache2 = cache[:, perm].contiguous()          # block i of cache2 = block perm[i] of cache
    table2 = inv[table.long()].to(torch.int32)
    out2, _ = _run(q, cache2, table2, seq)
    assert (tensor_bits(out2) == tensor_bits(out)).all()
    cache3 = cache.clone()
    for b in range(2):
        L = int(seq[b])
        last = int(table[b, (L - 1) // 4])
        cache3[:, last, (L - 1) % 4 + 1:] = 1e4   # past the end of the request
        for j in range((L + 3) // 4, 4):
            cache3[:, int(table[b, j])] = 1e4     # table entries beyond the request
    out3, _ = _run(q, cache3, table, seq)
    assert (tensor_bits(out3) == tensor_bits(out)).all()


def test_gqa_head_map():
    """Heads 0, 1 read kv head 0 and heads 2, 3 kv head 1: changing kv head 1 moves only heads 2, 3."""
    q, cache, table, seq = _case(F32, seed=93)
    out, _ = _run(q, cache, table, seq)
    cache2 = cache.clone()
    cache2[:, :, :, 1] *= 2
    out2, _ = _run(q, cache2, table, seq)
    assert torch.equal(out2[:, :2], out[:, :2])
    assert not torch.equal(out2[:, 2:], out[:, 2:])
    # and each head of a group sees the same keys: equal q rows give equal outputs
    q2 = q.clone()
    q2[:, 1] = q2[:, 0]
    out4, _ = _run(q2, cache, table, seq)
    assert torch.equal(out4[:, 1], out4[:, 0])


@pytest.mark.parametrize("fmt", FMTS)
def test_q_and_scale_trade_a_factor_of_two(fmt):
    q, cache, table, seq = _case(fmt, seed=94)
    out, _ = _run(q, cache, table, seq, 0.25)
    out2, _ = _run(q * 2, cache, table, seq, 0.125)
    assert (tensor_bits(out2) == tensor_bits(out)).all()
    out3, _ = _run(q, cache, table, seq, 0.5)
    assert not (tensor_bits(out3) == tensor_bits(out)).all()


def test_bad_entries_are_skipped_and_counted():
    q, cache, table, seq = _case(F32, lens=[16, 8], seed=95)
    ref, _ = _run(q, cache, table, seq)
    bad = table.clone()
    bad[0, 1] = 99                                 # block 1 of request 0 unreadable
    out, n = _run(q, cache, bad, seq)
    assert n == 1
    assert torch.equal(out[1], ref[1])
    # the same as a request whose block 1 tokens are absent: move blocks 2, 3 forward
    q1 = q[:1].clone()
    t1 = torch.tensor([[int(table[0, 0]), int(table[0, 2]), int(table[0, 3]), 0]], dtype=torch.int32)
    o1, _ = _run(q1, cache, t1, torch.tensor([12], dtype=torch.int32))
    assert torch.equal(out[0], o1[0])
    over = torch.tensor([17, 0], dtype=torch.int32)   # past 4 blocks of 4, and an empty request
    out, n = _run(q, cache, table, over)
    assert n == 1
    assert torch.equal(out[0], _run(q, cache, table, torch.tensor([16, 0], dtype=torch.int32))[0][0])
    assert (out[1] == 0).all()
