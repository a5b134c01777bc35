"""GPU: decode attention through the entry point that allocates nothing.

Some callers cannot allocate device memory: a serving stack whose allocator owns
the whole GPU and hands out only KV-cache blocks, or a plugin living in another
framework's process that must not call cudaMalloc behind that framework's back.
For them sra_paged_decode_attention_noalloc keeps the long-context split's
partial results in one device array the library holds. It must give what the
entry points with a caller-owned workspace (or none) give, call after call: the
array keeps the previous call's contents, so each test makes two calls in a row
on different inputs of one shape and compares both with the existing entry
point, within the attention tests' tolerance (the same kernel runs on both
sides, so the results are expected to agree exactly), and with the CPU oracle
at that tolerance, so a defect the two entry points share cannot pass.

This file is collected last, so a run that stops at its first failure has
already run every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

import oracle
import swiglu_rmsnorm_add_gb300 as sra
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.test_gpu_attention import assert_attention_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(B, ctx, n_head, n_kv, hd, dtype, seed):
    nb = B * ((ctx + 15) // 16) + 8
    q, cache, table, seq = syn.attention_inputs(B, ctx, n_head, n_kv, hd, 16, nb, dtype, seed)
    if B > 1:
        seq[0] = ctx - 7  # one ragged request
    return q, cache, table, seq


@pytest.mark.parametrize("B,ctx,n_head,n_kv,hd,dtype", [
    (1, 32768, 12, 2, 128, torch.bfloat16),   # one request, a long context: the split uses the array
    (2, 16384, 8, 1, 64, torch.float16),
    (32, 1024, 12, 2, 128, torch.bfloat16),   # many requests: the cluster kernel, no scratch
])
def test_noalloc_matches_existing_entry_twice(B, ctx, n_head, n_kv, hd, dtype):
    ws = None
    for call, seed in enumerate((1040, 1041)):
        q, cache, table, seq = _inputs(B, ctx, n_head, n_kv, hd, dtype, seed)
        dq, dc, dt, ds = q.to(DEV), cache.to(DEV), table.to(DEV), seq.to(DEV)
        if call == 0:
            ws = sra.decode_attention_workspace(B, n_head, n_kv, hd, table.shape[1], 16, dtype, DEV)
            assert (ws is None) == (B == 32)
        err_a = torch.zeros(1, dtype=torch.int32, device=DEV)
        err_b = torch.zeros(1, dtype=torch.int32, device=DEV)
        want = sra.paged_decode_attention(dq, dc, dt, ds, workspace=ws, err_count=err_a)
        got = torch.full_like(dq, float("nan"))
        sra.paged_decode_attention_noalloc(dq, dc, dt, ds, got, err_count=err_b)
        torch.cuda.synchronize()
        assert int(err_a.item()) == int(err_b.item()) == 0
        assert_attention_close(got, want, cache, table, seq, f"no-alloc call {call + 1} B={B} ctx={ctx}")
        ref = torch.empty_like(q)
        assert oracle.paged_decode_attention(q, cache, table, seq, ref) == 0
        assert_attention_close(got, ref, cache, table, seq, f"no-alloc vs oracle, call {call + 1} B={B} ctx={ctx}")


def test_noalloc_requires_out():
    q, cache, table, seq = _inputs(1, 256, 12, 2, 128, torch.bfloat16, 1042)
    with pytest.raises(ValueError):
        sra.paged_decode_attention_noalloc(q.to(DEV), cache.to(DEV), table.to(DEV), seq.to(DEV), None)
