"""GPU parity: SwiGLU and ReGLU over a fused gate_up tensor vs the oracle.

Workload: the Llama-3-8B MLP gate_up [T, 2 x 14336] bf16 ~N(0,1), T in
{1, 64, 512, 4096} (my-blog "Triton矩阵乘算子融合": the gate_up shape with
N = 28672), silu(gate) * up (koas-w.github.io "preformanceimprovement"
section 2) and relu(gate) * up (mer.dev "AsyncT vllm 适配加速笔记（一）" section
3.3). SwiGLU within 1 ulp; ReGLU bit-exact (the fp32 product of two 16-bit
values is exact, so one rounding gives the correctly rounded result).
T <= 512 is compared in full; T = 4096 on sampled rows plus the whole output's
finite-ness.
"""
import pytest
import torch

import oracle
import swiglu_rmsnorm_add_gb300 as sra
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.parity import assert_close, assert_values_equal

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
I8B = syn.LLAMA3_8B_MLP["intermediate"]


def gpu_glu(gu, act, out=None):
    out = sra.glu(gu.to(DEV), out, act)
    torch.cuda.synchronize()
    return out


def oracle_glu(gu, act):
    T, W = gu.shape
    ref = torch.empty(T, W // 2, dtype=gu.dtype)
    oracle.glu(gu, ref, act)
    return ref


@pytest.mark.parametrize("act", ["silu", "relu"])
@pytest.mark.parametrize("T", [1, 64, 512])
def test_config_llama3_full(T, act):
    gu = syn.glu_inputs(T, I8B, torch.bfloat16, 1003)
    got = gpu_glu(gu, act).cpu()
    ref = oracle_glu(gu, act)
    if act == "relu":
        assert_values_equal(got, ref, f"reglu T={T}")
    else:
        assert_close(got, ref, f"swiglu T={T}")


@pytest.mark.parametrize("act", ["silu", "relu"])
def test_config_llama3_t4096_sampled(act):
    T = 4096
    gu = syn.glu_inputs(T, I8B, torch.bfloat16, 1003)
    got = gpu_glu(gu, act).cpu()
    assert torch.isfinite(got.float()).all()
    g = torch.Generator().manual_seed(5)
    idx = torch.cat([torch.tensor([0, 1, T - 1]), torch.randint(0, T, (61,), generator=g)])
    ref = oracle_glu(gu[idx].contiguous(), act)
    if act == "relu":
        assert_values_equal(got[idx], ref, "reglu sampled")
    else:
        assert_close(got[idx], ref, "swiglu sampled")


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("act", ["silu", "relu"])
@pytest.mark.parametrize("T,I", [(1, 1), (3, 5), (7, 6), (33, 4), (17, 1000), (65, 8960), (9, 4099)])
def test_odd_shapes_and_dtypes(dtype, act, T, I):
    gu = syn.glu_inputs(T, I, dtype, 30)
    buf = torch.full((T * I + 128,), 7.0, dtype=dtype, device=DEV)
    out = buf[64:64 + T * I].view(T, I)
    gpu_glu(gu, act, out)
    b = buf.cpu()
    assert (b[:64].double() == 7).all() and (b[-64:].double() == 7).all()
    ref = oracle_glu(gu, act)
    if act == "relu":
        assert_values_equal(out, ref, f"reglu {T}x{I} {dtype}")
    else:
        assert_close(out, ref, f"swiglu {T}x{I} {dtype}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_extreme_gates(dtype):
    vals = [0.0, -0.0, 1.0, -1.0, 8.0, -8.0, 20.0, -20.0, 40.0, -40.0, 80.0, -80.0, 1e-3, -1e-3, 3.5, -3.5]
    I = len(vals)
    g = torch.tensor(vals, dtype=torch.float32)
    u = torch.linspace(-3, 3, I)
    gu = torch.cat([g, u]).reshape(1, 2 * I).to(dtype)
    for act in ("silu", "relu"):
        got = gpu_glu(gu, act).cpu()
        ref = oracle_glu(gu, act)
        assert_close(got, ref, f"{act} extreme gates {dtype}")


def test_strided_rows_and_misaligned():
    T, I = 19, 8960
    for off in (0, 1, 2):
        base = syn.normal((T * (2 * I + 16) + 8,), 0, 1, torch.bfloat16, 31, off)
        gu = base[off:off + T * (2 * I + 16)].view(T, 2 * I + 16)[:, :2 * I]
        bd = base.to(DEV)
        gud = bd[off:off + T * (2 * I + 16)].view(T, 2 * I + 16)[:, :2 * I]
        ob = torch.full((T, I + 24), 3.0, dtype=torch.bfloat16, device=DEV)
        out = ob[:, off:off + I]
        sra.swiglu(gud, out)
        ref = oracle_glu(gu.contiguous(), "silu")
        assert_close(out, ref, f"strided off={off}")
        o = ob.cpu()
        assert (o[:, :off].double() == 3).all() and (o[:, off + I:].double() == 3).all()


def test_zero_rows():
    gu = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    out = sra.swiglu(gu)
    assert out.shape == (0, 32)
