"""GPU parity: SwiGLU and ReGLU over a fused gate_up tensor vs the oracle.

Workload: the Llama-3-8B MLP gate_up [T, 2 x 14336] bf16 ~N(0,1), T in
{1, 64, 512, 4096} (my-blog "Triton矩阵乘算子融合": the gate_up shape with
N = 28672), silu(gate) * up (koas-w.github.io "preformanceimprovement"
section 2) and relu(gate) * up (mer.dev "AsyncT vllm 适配加速笔记（一）" section
3.3). SwiGLU within 1 ulp; ReGLU bit-exact (the fp32 product of two 16-bit
values is exact, so one rounding gives the correctly rounded result).
Every configured T is compared in full, and every 16-bit gate pattern (with up
values that keep the far-negative SiLU outputs normal) is compared too.
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
def test_config_llama3_t4096_full(act):
    """The dominant workload, every one of its 4096 x 14336 outputs against the oracle."""
    T = 4096
    gu = syn.glu_inputs(T, I8B, torch.bfloat16, 1003)
    got = gpu_glu(gu, act).cpu()
    ref = oracle_glu(gu, act)
    if act == "relu":
        assert_values_equal(got, ref, "reglu T=4096")
    else:
        assert_close(got, ref, "swiglu T=4096")


def _every_gate(dtype, ups):
    """gate_up [len(ups), 2 * 65536]: row k holds every 16-bit gate pattern of the
    format, with the up half set to ups[k]."""
    pats = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(dtype)
    g = pats.reshape(1, -1).expand(len(ups), -1)
    u = torch.tensor(ups, dtype=torch.float64).to(dtype).reshape(-1, 1).expand(-1, pats.numel())
    return torch.cat([g, u], dim=1).contiguous()


# Up values: the ones of the method's far-negative edge (1, -3, 0.5), plus the
# largest and smallest scales each format holds, which keep silu(g) * u a normal
# number for gates far below -87 (where e^-g leaves fp32's range).
_UPS = {torch.bfloat16: [1.0, -3.0, 0.5, 2.0 ** 100, -(2.0 ** 120), 2.0 ** -100],
        torch.float16: [1.0, -3.0, 0.5, 65504.0, -(2.0 ** -24), 2.0 ** 10]}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("act", ["silu", "relu"])
def test_every_gate_pattern(dtype, act):
    """All 65 536 gate bit patterns (NaN, infinities, subnormals, both zeros and the
    whole negative range down to the format's largest magnitude), each with every
    up value: SwiGLU within 1 ulp, ReGLU bit-exact."""
    gu = _every_gate(dtype, _UPS[dtype])
    got = gpu_glu(gu, act).cpu()
    ref = oracle_glu(gu, act)
    if act == "relu":
        assert_values_equal(got, ref, f"reglu every gate {dtype}")
    else:
        assert_close(got, ref, f"swiglu every gate {dtype}")


def test_fp32_gate_range():
    """fp32 gates: every bf16 pattern widened (exact), 262 144 random fp32 patterns
    and a dense sweep of [-200, -60], against the oracle at 1e-5 relative."""
    g16 = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    rnd = torch.randint(-(2 ** 31), 2 ** 31 - 1, (262144,), generator=torch.Generator().manual_seed(7),
                        dtype=torch.int64).to(torch.int32).view(torch.float32)
    sweep = torch.linspace(-200.0, -60.0, 65536, dtype=torch.float64).float()
    gates = torch.cat([g16, rnd, sweep])
    for u in (1.0, -3.0, 0.5, 2.0 ** 100, 2.0 ** -100):
        gu = torch.cat([gates, torch.full_like(gates, u)]).reshape(1, -1)
        got = gpu_glu(gu, "silu").cpu()
        ref = oracle_glu(gu, "silu")
        assert_close(got, ref, f"swiglu fp32 gates, u={u}")


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


@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("act", ["silu", "relu"])
def test_every_variant(variant, dtype, act):
    """Both register settings of the GLU kernel (48 registers; the compiler's choice)
    on a ragged shape and on every 16-bit gate pattern."""
    sra.force_variant("glu", variant)
    try:
        gu = syn.glu_inputs(37, 1000, dtype, 32)
        got = gpu_glu(gu, act).cpu()
        ref = oracle_glu(gu, act)
        (assert_values_equal if act == "relu" else assert_close)(got, ref, f"glu variant {variant} {dtype} {act}")
        if dtype != torch.float32:
            gu = _every_gate(dtype, _UPS[dtype])
            got = gpu_glu(gu, act).cpu()
            ref = oracle_glu(gu, act)
            (assert_values_equal if act == "relu" else assert_close)(got, ref, f"every gate, variant {variant}")
    finally:
        sra.force_variant("glu", -1)
