"""GPU parity of the 28-layer decode chain at batch 1 and 64 (Qwen2.5-1.5B shapes).

Each kernel is checked against the oracle applied to that kernel's actual
inputs, snapshotted just before the call, so drift cannot compound. The
residual stream x is updated by correctly rounded additions of seeded
activations only, so the end-to-end x after 56 updates is also compared
bit-exactly with an oracle-only run of the whole chain. The chain is then
captured in a CUDA graph and one replay is checked to equal an eager step.
"""
import pytest
import torch

import oracle
from swiglu_rmsnorm_add_gb300.chain import DecodeChain
from tests.parity import assert_bits_equal, assert_close

pytestmark = pytest.mark.gpu


def _cpu(t):
    return t.detach().cpu().clone()


@pytest.mark.parametrize("B", [1, 64])
def test_chain_per_kernel_and_end_to_end(B):
    ch = DecodeChain(B, num_blocks=256)  # 4096 slots per layer cache, enough for B <= 64
    x_oracle = _cpu(ch.x)
    for l in range(ch.L):
        L = ch.layers[l]
        for i, (name, call) in enumerate(ch.layer_calls(l)):
            if name == "add_rmsnorm":
                res = L["attn_res"] if i == 0 else L["mlp_res"]
                w = L["w_ln1"] if i == 0 else L["w_ln2"]
                out = L["h1"] if i == 0 else L["h2"]
                x_in = _cpu(ch.x)
                call()
                ref = torch.empty(B, ch.H, dtype=ch.dtype)
                x_ref = x_in.clone()
                oracle.add_rmsnorm(x_ref, _cpu(res), _cpu(w), ref, ch.eps)
                assert_bits_equal(ch.x, x_ref, f"layer {l} residual {i}")
                assert_close(out, ref, f"layer {l} norm {i}")
                # oracle-only chain
                oracle.add_rmsnorm(x_oracle, _cpu(res), _cpu(w), torch.empty_like(ref), ch.eps)
            elif name == "rope_kv_store":
                q, k, v, cache = _cpu(L["q"]), _cpu(L["k"]), _cpu(L["v"]), _cpu(L["kv_cache"])
                call()
                n = oracle.rope_kv_store(q, k, v, _cpu(ch.cos), _cpu(ch.sin), _cpu(ch.pos), _cpu(L["slots"]),
                                         cache)
                assert n == 0
                assert_close(L["q"], q, f"layer {l} q")
                kc = L["kv_cache"].cpu()
                assert_close(kc[0], cache[0], f"layer {l} K")
                assert_bits_equal(kc[1], cache[1], f"layer {l} V")
            else:
                gu = _cpu(L["gate_up"])
                call()
                ref = torch.empty(B, ch.I, dtype=ch.dtype)
                oracle.swiglu(gu, ref)
                assert_close(L["act"], ref, f"layer {l} swiglu")
    assert_bits_equal(ch.x, x_oracle, "end-to-end residual stream after 56 updates")


@pytest.mark.parametrize("pdl", [False, True])
def test_graph_replay_equals_eager(pdl):
    a = DecodeChain(4, layers=3, num_blocks=16)
    b = DecodeChain(4, layers=3, num_blocks=16)
    a.step()
    b.capture(pdl=pdl)   # capture warms up with one eager step, so both have run one step
    for _ in range(3):
        a.step()
        b.replay()
    torch.cuda.synchronize()
    assert_bits_equal(a.x, b.x, "x")
    for la, lb in zip(a.layers, b.layers):
        for key in ("h1", "h2", "act", "q", "kv_cache"):
            assert_bits_equal(la[key], lb[key], key)


def test_eager_pdl_calls_match():
    """Back-to-back eager launches with programmatic dependent launch on."""
    import swiglu_rmsnorm_add_gb300 as sra

    a = DecodeChain(64, layers=4, num_blocks=256)
    b = DecodeChain(64, layers=4, num_blocks=256)
    prev = sra.set_pdl(True)
    try:
        for _ in range(2):
            b.step()
    finally:
        sra.set_pdl(prev)
    for _ in range(2):
        a.step()
    torch.cuda.synchronize()
    assert_bits_equal(a.x, b.x, "x")
    for la, lb in zip(a.layers, b.layers):
        for key in ("h1", "h2", "act", "q", "kv_cache"):
            assert_bits_equal(la[key], lb[key], key)
