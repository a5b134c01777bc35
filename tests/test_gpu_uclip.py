"""GPU parity: UClip / DyHT clamp(alpha * x, lo, hi) * gamma vs the oracle.

Workloads (mer.dev "AsyncT vllm 适配加速笔记（一）": section 0 puts DyHT in place
of every RMSNorm; section 3.3 runs it as one kernel, also on the Q/K heads of a
fused QKV projection): DyHT over Qwen2.5-1.5B-shaped hidden rows [T, 1536] for
the residual-norm token counts T in {1, 16, 256, 4096}, and the Q/K norm on
narrow views of a fused QKV output [T, 12 + 2 + 2, 128] for T in {1, 64, 2048},
in place. x ~ N(0, 1), alpha ~ U(0.25, 1), gamma ~ N(1, 0.1), fp32 parameters.
The page's kernel fixes the arithmetic (fp32 a * x, the clamp against fp32
bounds, fp32 * g, one rounding to the dtype) and the oracle follows it, so the
outputs are compared bit for bit (+0 and -0 equal); every byte outside the
written view is bit-exact too.
"""
import math

import pytest
import torch

import oracle
import swiglu_rmsnorm_add_gb300 as sra
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.parity import assert_bits_equal, assert_values_equal

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DTYPES = [torch.float32, torch.float16, torch.bfloat16]


def both(x, alpha, gamma, lo=-1.0, hi=1.0):
    """(gpu, oracle) outputs for a CPU input view x, computed out of place."""
    ref = torch.empty(x.shape, dtype=x.dtype)
    oracle.uclip(x, alpha, gamma, ref, lo, hi)
    got = sra.uclip(x.to(DEV), alpha.to(DEV), gamma.to(DEV), None, lo, hi)
    torch.cuda.synchronize()
    return got.cpu(), ref


@pytest.mark.parametrize("T", syn.ADD_RMS_T)
def test_config_dyht_hidden_rows(T):
    x = syn.normal((T, 1536), 0.0, 1.0, torch.bfloat16, 1005, 1)
    alpha, gamma = syn.uclip_params(1536, False, True, 1005)
    ref = torch.empty_like(x)
    oracle.dyht(x, alpha, gamma, ref)
    got = sra.dyht(x.to(DEV), alpha.to(DEV), gamma.to(DEV))
    assert_values_equal(got, ref, f"DyHT T={T}")


@pytest.mark.parametrize("T", syn.ROPE_T)
def test_config_qk_norm_in_place_on_fused_qkv(T):
    nh, nkv, hd = 12, 2, 128
    qkv = syn.qkv_inputs(T, nh, nkv, hd, torch.bfloat16, 1006)
    aq, gq = syn.uclip_params(hd, True, True, 1006)
    ak, gk = syn.uclip_params(hd, True, True, 1007)
    ref = qkv.clone()
    oracle.dyht(ref[:, :nh], aq, gq, ref[:, :nh])
    oracle.dyht(ref[:, nh:nh + nkv], ak, gk, ref[:, nh:nh + nkv])
    d = qkv.to(DEV)
    q, k = d[:, :nh], d[:, nh:nh + nkv]
    sra.dyht(q, aq.to(DEV), gq.to(DEV), q)
    sra.dyht(k, ak.to(DEV), gk.to(DEV), k)
    got = d.cpu()
    assert_values_equal(got[:, :nh + nkv], ref[:, :nh + nkv], f"Q/K T={T}")
    assert_bits_equal(got[:, nh + nkv:], qkv[:, nh + nkv:], "V untouched")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("a_pc,g_pc", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("N,H,D", [(1, 1, 1), (3, 1, 7), (5, 3, 64), (17, 2, 100), (9, 1, 1000), (4, 4, 4095),
                                   (2, 1, 8192), (700, 1, 24), (33, 5, 8)])
def test_shapes_dtypes_parameters(dtype, a_pc, g_pc, N, H, D):
    x = syn.normal((N, H, D), 0.0, 1.5, dtype, 1008, N * 31 + D)
    alpha, gamma = syn.uclip_params(D, a_pc, g_pc, 1008 + D)
    got, ref = both(x, alpha, gamma, -0.8, 1.25)
    assert_values_equal(got, ref, f"{N}x{H}x{D} {dtype} apc={a_pc} gpc={g_pc}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_strided_views_and_guard_bands(dtype):
    """Heads-outer (permuted) input, padded rows, misaligned base (scalar path),
    a separate strided output: values as on contiguous data, every other byte of
    the output buffer untouched."""
    N, H, D = 37, 6, 96
    alpha, gamma = syn.uclip_params(D, True, True, 1009)
    # name -> (base buffer, view of it)
    views = {
        "padded": (syn.normal((N, H, D + 8), 0, 1, dtype, 1009, 1), lambda b: b[:, :, :D]),
        "heads outer": (syn.normal((H, N, D), 0, 1, dtype, 1009, 2), lambda b: b.permute(1, 0, 2)),
        "misaligned": (syn.normal((N * H * D + 1,), 0, 1, dtype, 1009, 3), lambda b: b[1:].view(N, H, D)),
    }
    for name, (base, view) in views.items():
        ref = torch.empty(N, H, D, dtype=dtype)
        oracle.uclip(view(base).contiguous(), alpha, gamma, ref, -1.0, 1.0)
        xd = view(base.to(DEV))
        # a 16-byte aligned strided output with a guard band of 8 columns each side and one extra head
        obuf = torch.full((N, H + 1, D + 16), 7.0, dtype=dtype, device=DEV)
        out = obuf[:, :H, 8:8 + D]
        sra.uclip(xd, alpha.to(DEV), gamma.to(DEV), out, -1.0, 1.0)
        torch.cuda.synchronize()
        assert_values_equal(out, ref, name)
        ob = obuf.cpu()
        mask = torch.ones(N, H + 1, D + 16, dtype=torch.bool)
        mask[:, :H, 8:8 + D] = False
        assert bool((ob[mask] == 7.0).all()), f"{name}: guard band overwritten"


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place_matches_out_of_place(dtype):
    x = syn.normal((300, 4, 128), 0, 1, dtype, 1010, 1)
    alpha, gamma = syn.uclip_params(128, True, False, 1010)
    got, ref = both(x, alpha, gamma)
    d = x.to(DEV)
    sra.uclip(d, alpha.to(DEV), gamma.to(DEV), d)
    assert_bits_equal(d, got, "in place == out of place")
    assert_values_equal(d, ref, "in place")


@pytest.mark.parametrize("dtype", DTYPES)
def test_special_values_and_bounds(dtype):
    vals = [math.nan, math.inf, -math.inf, 0.0, -0.0, 1e-30, -3.0, 3.0, 0.5, -0.5]
    x = torch.tensor(vals, dtype=torch.float64).to(dtype).reshape(1, -1)
    for (lo, hi) in [(-1.0, 1.0), (0.0, 0.0), (-math.inf, math.inf), (-2.0, -1.0)]:
        got, ref = both(x, torch.tensor([1.5]), torch.tensor([-2.0]), lo, hi)
        assert float(ref[0, 0]) == float(torch.tensor(lo, dtype=torch.float32) * -2.0)  # NaN -> lo, times g
        assert_values_equal(got, ref, f"bounds ({lo}, {hi})")


def test_large_rows_sampled():
    """A 65 536 x 1536 bf16 DyHT (the bandwidth-bound shape): sampled rows vs the oracle."""
    x = syn.normal((65536, 1536), 0, 1, torch.bfloat16, 1011, 1)
    alpha, gamma = syn.uclip_params(1536, False, True, 1011)
    got = sra.dyht(x.to(DEV), alpha.to(DEV), gamma.to(DEV)).cpu()
    rows = torch.from_numpy(syn.rng(1011, 2).choice(65536, size=64, replace=False))
    ref = torch.empty(64, 1536, dtype=torch.bfloat16)
    oracle.dyht(x[rows], alpha, gamma, ref)
    assert_values_equal(got[rows], ref, "sampled rows")
    assert bool(torch.isfinite(got).all())


def test_zero_rows_and_errors():
    x = torch.empty(0, 3, 64, dtype=torch.bfloat16, device=DEV)
    a, g = torch.ones(64, device=DEV), torch.ones(1, device=DEV)
    sra.uclip(x, a, g)
    y = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    for lo, hi in ((1.0, -1.0), (math.nan, 1.0)):
        with pytest.raises(sra.SRAError):
            sra.uclip(y, a, g, None, lo, hi)
    with pytest.raises(sra.SRAError):   # out overlapping x, not in place
        sra.uclip(y[:, :32], a[:32], g, y[:, 16:48])
