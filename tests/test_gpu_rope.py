"""GPU parity: fused RoPE + paged KV-cache store vs the oracle, in both
pairings: neox halves (i, i + head_dim/2) and interleaved GPT-J pairs
(2i, 2i + 1) (m.lsln.cn 21-operator article, section 2.3).

Workload: Qwen2.5-1.5B GQA (12 Q / 2 KV heads, head_dim 128, bf16), T in
{1, 64, 2048}, positions uniform in [0, 32768), theta 1e6 tables, a
[2, 4096, 16, 2, 128] cache prefilled with the 0xDEAD sentinel and distinct
slots (koas-w.github.io "preformanceimprovement" section 1; cache layout of
mer.dev "AsyncT vllm 适配加速笔记（一）" section 1.1).
Q and K within 1 ulp; V copies, slot placement and every untouched cache byte
bit-exact; error counts exact.
"""
import pytest
import torch

import oracle
import swiglu_rmsnorm_add_gb300 as sra
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.parity import assert_bits_equal, assert_close, assert_values_equal

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


STYLES = ["neox", "interleaved"]


def run_both(inp, max_pos=None, expect_err=None, style="neox"):
    d = {k: v.to(DEV) for k, v in inp.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sra.rope_kv_store(d["q"], d["k"], d["v"], d["cos"], d["sin"], d["pos"], d["slot_mapping"], d["kv_cache"],
                      err_count=err, max_pos=max_pos, style=style)
    torch.cuda.synchronize()
    n = oracle.rope_kv_store(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], inp["pos"],
                             inp["slot_mapping"], inp["kv_cache"], max_pos=max_pos, style=style)
    assert int(err.item()) == n
    if expect_err is not None:
        assert n == expect_err
    return d


def check(d, inp, what):
    cache_g, cache_o = d["kv_cache"].cpu(), inp["kv_cache"]
    assert_close(d["q"], inp["q"], f"{what}: q")
    assert_close(cache_g[0], cache_o[0], f"{what}: K plane")
    assert_bits_equal(cache_g[1], cache_o[1], f"{what}: V plane")
    # placement: the set of slots whose K-plane bytes changed is the same on both
    sent = syn.sentinel_cache(cache_o.shape[1:], cache_o.dtype)
    iv = torch.int32 if cache_o.element_size() == 4 else torch.int16
    touched_g = (cache_g[0].view(iv) != sent.view(iv)).flatten(2).any(-1)
    touched_o = (cache_o[0].view(iv) != sent.view(iv)).flatten(2).any(-1)
    assert torch.equal(touched_g, touched_o), f"{what}: slot placement"


@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("T", syn.ROPE_T)
def test_config_qwen25(T, style):
    tables = syn.rope_tables(32768, 128, 1e6)
    inp = syn.rope_inputs(T, 1002, tables=tables)
    d = run_both(inp, expect_err=0, style=style)
    check(d, inp, f"T={T} {style}")


@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("n_head,n_kv,hd", [(12, 2, 128), (8, 8, 64), (16, 1, 256), (4, 2, 32), (6, 3, 10),
                                            (4, 4, 8), (2, 1, 2)])
def test_head_layouts_and_dtypes(dtype, n_head, n_kv, hd, style):
    tables = syn.rope_tables(4096, hd, 1e4)
    inp = syn.rope_inputs(37, 20, n_head=n_head, n_kv_head=n_kv, head_dim=hd, num_blocks=8, block_size=16,
                          max_pos=4096, dtype=dtype, tables=tables)
    d = run_both(inp, style=style)
    check(d, inp, f"{n_head}/{n_kv}/{hd} {dtype} {style}")


def test_interleaved_ninety_degrees_and_identity():
    """cos 0, sin 1 turns each pair (x[2i], x[2i+1]) into (-x[2i+1], x[2i]);
    position 0 is the identity."""
    inp = syn.rope_inputs(16, 27, num_blocks=4)
    inp["cos"], inp["sin"] = torch.zeros(32768, 64), torch.ones(32768, 64)
    q0 = inp["q"].clone()
    d = run_both(inp, style="interleaved")
    assert_values_equal(d["q"][..., 0::2], -q0[..., 1::2], "90 degrees, even dims")
    assert_values_equal(d["q"][..., 1::2], q0[..., 0::2], "90 degrees, odd dims")
    inp = syn.rope_inputs(16, 28, num_blocks=4)
    inp["pos"].zero_()
    q0 = inp["q"].clone()
    d = run_both(inp, style="interleaved")
    assert_values_equal(d["q"], q0, "pos 0 is the identity")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_interleaved_is_neox_on_permuted_dims(dtype):
    """Interleaved RoPE of x equals neox RoPE of x with its dimensions permuted
    (evens first, then odds), permuted back: both kernels, bit for bit."""
    inp = syn.rope_inputs(64, 29, num_blocks=8, dtype=dtype)
    perm = torch.cat([torch.arange(0, 128, 2), torch.arange(1, 128, 2)])
    inv = torch.argsort(perm)
    a = {k: v.to(DEV) for k, v in inp.items()}
    b = {k: v.to(DEV) for k, v in inp.items()}
    for key in ("q", "k", "v"):
        b[key] = b[key][..., perm].contiguous()
    sra.rope_kv_store(a["q"], a["k"], a["v"], a["cos"], a["sin"], a["pos"], a["slot_mapping"], a["kv_cache"],
                      style="interleaved")
    sra.rope_kv_store(b["q"], b["k"], b["v"], b["cos"], b["sin"], b["pos"], b["slot_mapping"], b["kv_cache"])
    torch.cuda.synchronize()
    assert_bits_equal(a["q"], b["q"][..., inv], "q")
    # untouched slots hold the sentinel in both, so the whole cache compares
    assert_bits_equal(a["kv_cache"], b["kv_cache"][..., inv], "cache")


def test_position_zero_identity_and_ninety_degrees():
    inp = syn.rope_inputs(16, 21, num_blocks=4)
    inp["pos"].zero_()
    q0 = inp["q"].clone()
    d = run_both(inp)
    assert_values_equal(d["q"], q0, "pos 0 is the identity")
    inp = syn.rope_inputs(16, 22, num_blocks=4)
    cos = torch.zeros(32768, 64)
    sin = torch.ones(32768, 64)
    inp["cos"], inp["sin"] = cos, sin
    q0 = inp["q"].clone()
    d = run_both(inp)
    assert_values_equal(d["q"][..., :64], -q0[..., 64:], "90 degrees, first half")
    assert_values_equal(d["q"][..., 64:], q0[..., :64], "90 degrees, second half")


@pytest.mark.parametrize("style", STYLES)
def test_padding_bad_slots_and_positions(style):
    inp = syn.rope_inputs(8, 23, num_blocks=4)   # 64 slots
    inp["slot_mapping"] = torch.tensor([-1, 3, 64, 5, 1000, 7, -1, 9], dtype=torch.int64)
    inp["pos"] = torch.tensor([1, 2, 3, -4, 5, 32768, 7, 8], dtype=torch.int64)
    # errors: slot 64 and 1000 out of range (2), positions -4 and 32768 (2)
    d = run_both(inp, expect_err=4, style=style)
    check(d, inp, f"padding / errors {style}")


@pytest.mark.parametrize("style", STYLES)
def test_fused_qkv_views_and_misaligned_scalar_path(style):
    T, nh, nkv, hd = 40, 12, 2, 128
    W = (nh + 2 * nkv) * hd
    qkv = syn.normal((T, W + 8), 0, 1, torch.bfloat16, 24, 1)   # padded rows
    tables = syn.rope_tables(32768, hd, 1e6)
    pos = syn.positions(T, 32768, 24, 2)
    slot = syn.slots(T, 64 * 16, 24, 3)
    for off in (0, 1):   # off = 1: every row 2-byte aligned -> scalar path
        base = syn.normal((T * (W + 8) + 1,), 0, 1, torch.bfloat16, 24, 4)
        buf = base[off:off + T * (W + 8)].view(T, W + 8)
        q = buf[:, :nh * hd].view(T, nh, hd)
        k = buf[:, nh * hd:(nh + nkv) * hd].view(T, nkv, hd)
        v = buf[:, (nh + nkv) * hd:W].view(T, nkv, hd)
        cache = syn.sentinel_cache((2, 64, 16, nkv, hd))
        inp = dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(), cos=tables[0], sin=tables[1], pos=pos,
                   slot_mapping=slot, kv_cache=cache)
        bd = base.to(DEV)
        bufd = bd[off:off + T * (W + 8)].view(T, W + 8)
        dq = bufd[:, :nh * hd].view(T, nh, hd)
        dk = bufd[:, nh * hd:(nh + nkv) * hd].view(T, nkv, hd)
        dv = bufd[:, (nh + nkv) * hd:W].view(T, nkv, hd)
        dc = cache.to(DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        sra.rope_kv_store(dq, dk, dv, tables[0].to(DEV), tables[1].to(DEV), pos.to(DEV), slot.to(DEV), dc,
                          err_count=err, style=style)
        oracle.rope_kv_store(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], pos, slot, cache, style=style)
        assert_close(dq, inp["q"], f"fused view q off={off}")
        assert_close(dc.cpu()[0], cache[0], "K")
        assert_bits_equal(dc.cpu()[1], cache[1], "V")
        # k, v and the row padding are untouched
        after = bufd.cpu()
        assert_bits_equal(after[:, nh * hd:], buf[:, nh * hd:], "k, v, padding untouched")


@pytest.mark.parametrize("style", STYLES)
def test_duplicate_free_large_T_cache_untouched_elsewhere(style):
    inp = syn.rope_inputs(2048, 25)
    d = run_both(inp, expect_err=0, style=style)
    check(d, inp, f"T=2048 full cache {style}")


def test_zero_tokens():
    inp = syn.rope_inputs(0, 26, num_blocks=2)
    d = {k: v.to(DEV) for k, v in inp.items()}
    sra.rope_kv_store(d["q"], d["k"], d["v"], d["cos"], d["sin"], d["pos"], d["slot_mapping"], d["kv_cache"])
    assert_bits_equal(d["kv_cache"], inp["kv_cache"], "no-op")


# ------------------------------------------------ Q/K UClip fused into the load
def _qk_params(hd, seed):
    return tuple(syn.uclip_params(hd, True, True, seed + i)[i % 2] for i in range(4))


@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,n_head,n_kv,hd", [(64, 12, 2, 128), (2048, 12, 2, 128), (37, 8, 8, 64), (29, 6, 3, 10),
                                              (5, 16, 1, 256)])
def test_qk_uclip_fused_vs_oracle(style, dtype, T, n_head, n_kv, hd):
    """Fused Q/K norm + RoPE + store vs the oracle's uclip-then-rope composition."""
    max_pos = 32768 if hd == 128 else 4096
    tables = syn.rope_tables(max_pos, hd, 1e6 if hd == 128 else 1e4)
    inp = syn.rope_inputs(T, 30, n_head=n_head, n_kv_head=n_kv, head_dim=hd,
                          num_blocks=max(8, (T + 15) // 16), max_pos=max_pos, dtype=dtype, tables=tables)
    params = _qk_params(hd, 30)
    d = {k: v.to(DEV) for k, v in inp.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sra.rope_kv_store(d["q"], d["k"], d["v"], d["cos"], d["sin"], d["pos"], d["slot_mapping"], d["kv_cache"],
                      err_count=err, style=style, qk_uclip=tuple(p.to(DEV) for p in params), clip=(-0.9, 1.1))
    torch.cuda.synchronize()
    n = oracle.qk_uclip_rope_kv_store(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], inp["pos"],
                                      inp["slot_mapping"], inp["kv_cache"], *params, clip_min=-0.9, clip_max=1.1,
                                      style=style)
    assert int(err.item()) == n == 0
    check(d, inp, f"qk_uclip {style} {dtype} {n_head}/{n_kv}/{hd}")


@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_qk_uclip_fused_equals_separate_kernels(style, dtype):
    """The fused kernel is bit-identical to sra.uclip on the Q and K heads followed by
    the plain rope_kv_store on the fused QKV views (same fp32 steps, same roundings)."""
    T, nh, nkv, hd = 512, 12, 2, 128
    qkv = syn.qkv_inputs(T, nh, nkv, hd, dtype, 31).to(DEV)
    tables = [t.to(DEV) for t in syn.rope_tables(32768, hd, 1e6)]
    pos = syn.positions(T, 32768, 31, 2).to(DEV)
    slot = syn.slots(T, 64 * 16, 31, 3).to(DEV)
    qa, qg, ka, kg = (p.to(DEV) for p in _qk_params(hd, 31))
    a, b = qkv.clone(), qkv.clone()
    ca = syn.sentinel_cache((2, 64, 16, nkv, hd), dtype).to(DEV)
    cb = ca.clone()
    sra.rope_kv_store(a[:, :nh], a[:, nh:nh + nkv], a[:, nh + nkv:], *tables, pos, slot, ca, style=style,
                      qk_uclip=(qa, qg, ka, kg))
    kn = torch.empty(T, nkv, hd, dtype=dtype, device=DEV)
    sra.dyht(b[:, :nh], qa, qg, b[:, :nh])
    sra.dyht(b[:, nh:nh + nkv], ka, kg, kn)
    sra.rope_kv_store(b[:, :nh], kn, b[:, nh + nkv:], *tables, pos, slot, cb, style=style)
    torch.cuda.synchronize()
    assert_bits_equal(a[:, :nh], b[:, :nh], "q")
    assert_bits_equal(a[:, nh:], qkv[:, nh:], "k and v inputs untouched")
    assert_bits_equal(ca, cb, "cache")


def test_qk_uclip_bad_positions_and_scalar_path():
    """Bad positions leave q raw and count; a 2-byte-misaligned fused view takes the scalar path."""
    T, nh, nkv, hd = 24, 4, 2, 64
    inp = syn.rope_inputs(T, 32, n_head=nh, n_kv_head=nkv, head_dim=hd, num_blocks=4, max_pos=4096,
                          tables=syn.rope_tables(4096, hd, 1e4))
    inp["pos"][3] = -2
    inp["pos"][9] = 4096
    params = _qk_params(hd, 32)
    W = (nh + 2 * nkv) * hd
    base = syn.normal((T * W + 1,), 0, 1, torch.bfloat16, 32, 9)
    buf = base[1:].view(T, W)
    q = buf[:, :nh * hd].view(T, nh, hd)
    k = buf[:, nh * hd:(nh + nkv) * hd].view(T, nkv, hd)
    v = buf[:, (nh + nkv) * hd:].view(T, nkv, hd)
    bd = base.to(DEV)
    bufd = bd[1:].view(T, W)
    dq = bufd[:, :nh * hd].view(T, nh, hd)
    dk = bufd[:, nh * hd:(nh + nkv) * hd].view(T, nkv, hd)
    dv = bufd[:, (nh + nkv) * hd:].view(T, nkv, hd)
    dc = inp["kv_cache"].to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sra.rope_kv_store(dq, dk, dv, inp["cos"].to(DEV), inp["sin"].to(DEV), inp["pos"].to(DEV),
                      inp["slot_mapping"].to(DEV), dc, err_count=err, qk_uclip=tuple(p.to(DEV) for p in params))
    qo = q.contiguous()
    n = oracle.qk_uclip_rope_kv_store(qo, k.contiguous(), v.contiguous(), inp["cos"], inp["sin"], inp["pos"],
                                      inp["slot_mapping"], inp["kv_cache"], *params)
    assert int(err.item()) == n == 2
    assert_close(dq, qo, "q")
    assert_close(dc.cpu()[0], inp["kv_cache"][0], "K")
    assert_bits_equal(dc.cpu()[1], inp["kv_cache"][1], "V")
    assert_bits_equal(dq[3], q[3], "bad position: q raw")


# ------------------------------------------------ forced kernel variants
@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,n_head,n_kv,hd", [(2048, 12, 2, 128), (1, 12, 2, 128), (37, 8, 8, 64), (29, 16, 1, 256),
                                              (37, 6, 3, 10), (5, 2, 1, 2), (7, 3, 1, 64)])
def test_forced_variants(variant, style, dtype, T, n_head, n_kv, hd):
    """One task per thread (0) and two tasks per thread sharing a cos / sin load (1); the
    second needs an even number of head units and refuses the rest."""
    max_pos = 32768 if hd == 128 else 4096
    tables = syn.rope_tables(max_pos, hd, 1e6 if hd == 128 else 1e4)
    inp = syn.rope_inputs(T, 31, n_head=n_head, n_kv_head=n_kv, head_dim=hd,
                          num_blocks=max(8, (T + 15) // 16), max_pos=max_pos, dtype=dtype, tables=tables)
    sra.force_variant("rope_kv_store", variant)
    try:
        try:
            d = run_both(inp, expect_err=0, style=style)
        except sra.SRAError as e:
            assert variant == 1 and (n_head + 2 * n_kv) % 2 == 1 and e.status == -7
            return
        assert variant == 0 or (n_head + 2 * n_kv) % 2 == 0
        check(d, inp, f"variant {variant} {style} {dtype} T={T} {n_head}/{n_kv}/{hd}")
    finally:
        sra.force_variant("rope_kv_store", -1)


@pytest.mark.parametrize("style", STYLES)
def test_two_tasks_per_thread_padding_bad_slots_and_uclip(style):
    sra.force_variant("rope_kv_store", 1)
    try:
        inp = syn.rope_inputs(8, 23, num_blocks=4)   # 64 slots
        inp["slot_mapping"] = torch.tensor([-1, 3, 64, 5, 1000, 7, -1, 9], dtype=torch.int64)
        inp["pos"] = torch.tensor([1, 2, 3, -4, 5, 32768, 7, 8], dtype=torch.int64)
        d = run_both(inp, expect_err=4, style=style)
        check(d, inp, f"two tasks per thread, padding / errors {style}")

        tables = syn.rope_tables(32768, 128, 1e6)
        inp = syn.rope_inputs(2048, 32, tables=tables)
        params = _qk_params(128, 32)
        d = {k: v.to(DEV) for k, v in inp.items()}
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        sra.rope_kv_store(d["q"], d["k"], d["v"], d["cos"], d["sin"], d["pos"], d["slot_mapping"], d["kv_cache"],
                          err_count=err, style=style, qk_uclip=tuple(p.to(DEV) for p in params), clip=(-0.9, 1.1))
        torch.cuda.synchronize()
        n = oracle.qk_uclip_rope_kv_store(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], inp["pos"],
                                          inp["slot_mapping"], inp["kv_cache"], *params, clip_min=-0.9,
                                          clip_max=1.1, style=style)
        assert int(err.item()) == n == 0
        check(d, inp, f"two tasks per thread, qk_uclip {style}")
    finally:
        sra.force_variant("rope_kv_store", -1)
