"""GPU parity: RMSNorm and residual-add + RMSNorm through the C ABI vs the oracle.

Workloads: the Qwen2.5-1.5B hidden row (4 x 1536 bf16); the 2 x 256-row sweep
over D in {128 ... 8192} in fp32 / fp16 / bf16 (agent.csdn.net
"使用Triton实现RMSNorm算子", performance section); add_rmsnorm at T in
{1, 16, 256, 4096} x 1536 bf16; plus ragged / odd widths (the D = 2176 case the
same page discusses), misaligned and strided rows, in-place use, every kernel
variant forced, and guard bands around every output.
"""
import pytest
import torch

import oracle
import swiglu_rmsnorm_add_gb300 as sra
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.parity import assert_bits_equal, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DTYPES = [torch.float32, torch.float16, torch.bfloat16]
GUARD = 64


def guarded(shape, dtype, fill=-3.0):
    """A CUDA tensor of `shape` inside a buffer with GUARD sentinel elements on each side."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device=DEV)
    return buf, buf[GUARD:GUARD + n].view(*shape)


def check_guards(buf, fill=-3.0):
    b = buf.cpu()
    assert (b[:GUARD].double() == fill).all() and (b[-GUARD:].double() == fill).all(), "guard band overwritten"


def run_rms(x, w, eps=syn.EPS):
    buf, out = guarded(x.shape, x.dtype)
    sra.rmsnorm(x.to(DEV), w.to(DEV), out, eps)
    torch.cuda.synchronize()
    check_guards(buf)
    ref = torch.empty_like(x)
    oracle.rmsnorm(x, w, ref, eps)
    return out.cpu(), ref


def test_config_decode_rows():
    x, w = syn.rms_inputs(4, 1536, torch.bfloat16, 1000)
    got, ref = run_rms(x, w)
    assert_close(got, ref, "rmsnorm [4,1536] bf16")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", syn.RMS_SWEEP_D)
def test_config_sweep(dtype, D):
    x, w = syn.rms_inputs(syn.RMS_SWEEP_ROWS, D, dtype, 1001)
    got, ref = run_rms(x, w)
    assert_close(got, ref, f"rmsnorm [512,{D}] {dtype}")


@pytest.mark.parametrize("T", syn.ADD_RMS_T)
def test_config_add_rmsnorm(T):
    x, r, w = syn.add_rms_inputs(T, 1536, torch.bfloat16, 1001)
    xd = x.to(DEV)
    buf, out = guarded(x.shape, x.dtype)
    sra.add_rmsnorm(xd, r.to(DEV), w.to(DEV), out, syn.EPS)
    torch.cuda.synchronize()
    check_guards(buf)
    ref = torch.empty_like(x)
    oracle.add_rmsnorm(x, r, w, ref, syn.EPS)
    assert_bits_equal(xd, x, f"add_rmsnorm residual T={T}")
    assert_close(out, ref, f"add_rmsnorm out T={T}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [1, 2, 3, 7, 8, 9, 15, 17, 127, 129, 1000, 2176, 3001])
@pytest.mark.parametrize("rows", [1, 5, 300])
def test_ragged_widths(dtype, D, rows):
    x, w = syn.rms_inputs(rows, D, dtype, 7)
    got, ref = run_rms(x, w)
    assert_close(got, ref, f"rmsnorm [{rows},{D}] {dtype}")
    xa, ra, wa = syn.add_rms_inputs(rows, D, dtype, 8)
    xd = xa.to(DEV)
    out = sra.add_rmsnorm(xd, ra.to(DEV), wa.to(DEV), eps=syn.EPS)
    ref = torch.empty_like(xa)
    oracle.add_rmsnorm(xa, ra, wa, ref, syn.EPS)
    assert_bits_equal(xd, xa, "residual")
    assert_close(out, ref, f"add_rmsnorm [{rows},{D}] {dtype}")


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,D", [(3, 1536), (700, 1536), (64, 2176), (40, 8192), (5, 333), (1, 1),
                                    (333, 4095), (512, 8192)])
def test_every_variant(variant, dtype, rows, D):
    sra.force_variant("rmsnorm", variant)
    try:
        x, w = syn.rms_inputs(rows, D, dtype, 9)
        try:
            got, ref = run_rms(x, w)
        except sra.SRAError as e:
            assert e.status == -7  # this variant cannot hold the row in registers
            return
        assert_close(got, ref, f"variant {variant} [{rows},{D}] {dtype}")
        xa, ra, wa = syn.add_rms_inputs(rows, D, dtype, 10)
        xd = xa.to(DEV)
        out = sra.add_rmsnorm(xd, ra.to(DEV), wa.to(DEV), eps=syn.EPS)
        ref = torch.empty_like(xa)
        oracle.add_rmsnorm(xa, ra, wa, ref, syn.EPS)
        assert_bits_equal(xd, xa, "residual")
        assert_close(out, ref, f"add variant {variant}")
    finally:
        sra.force_variant("rmsnorm", -1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [40000, 70000])
def test_wide_rows_smem_and_two_pass(dtype, D):
    x, w = syn.rms_inputs(6, D, dtype, 11)
    got, ref = run_rms(x, w)
    assert_close(got, ref, f"wide [{6},{D}]")


def test_misaligned_and_strided():
    dtype = torch.bfloat16
    rows, D, stride = 33, 1536, 1600
    base = syn.normal((rows * stride + 1,), 0, 1, dtype, 12, 1)
    x = base[1:1 + rows * stride].view(rows, stride)[:, :D]   # 2-byte aligned rows
    w = syn.normal((D,), 1, 0.1, dtype, 12, 2)
    xd_base = base.to(DEV)
    xd = xd_base[1:1 + rows * stride].view(rows, stride)[:, :D]
    obuf = torch.full((rows, D + 8), 5.0, dtype=dtype, device=DEV)
    out = obuf[:, 3:3 + D]
    sra.rmsnorm(xd, w.to(DEV), out, syn.EPS)
    ref = torch.empty(rows, D, dtype=dtype)
    oracle.rmsnorm(x.contiguous(), w, ref, syn.EPS)
    assert_close(out, ref, "misaligned strided")
    ob = obuf.cpu()
    assert (ob[:, :3].double() == 5).all() and (ob[:, 3 + D:].double() == 5).all()


def test_in_place():
    x, w = syn.rms_inputs(64, 1536, torch.bfloat16, 13)
    xd = x.to(DEV)
    sra.rmsnorm(xd, w.to(DEV), xd, syn.EPS)
    ref = torch.empty_like(x)
    oracle.rmsnorm(x, w, ref, syn.EPS)
    assert_close(xd, ref, "in-place")


def test_zero_rows_and_zero_row_values():
    x = torch.zeros(0, 1536, dtype=torch.bfloat16, device=DEV)
    w = torch.ones(1536, dtype=torch.bfloat16, device=DEV)
    sra.rmsnorm(x, w, torch.empty_like(x), syn.EPS)
    z = torch.zeros(3, 1536, dtype=torch.bfloat16, device=DEV)
    out = sra.rmsnorm(z, w, eps=syn.EPS)
    assert (out.double() == 0).all()


def test_res_equal_x_doubles():
    x, _, w = syn.add_rms_inputs(16, 1536, torch.bfloat16, 14)
    xd = x.to(DEV)
    out = sra.add_rmsnorm(xd, xd, w.to(DEV), eps=syn.EPS)
    x2 = x.clone()
    ref = torch.empty_like(x)
    oracle.add_rmsnorm(x2, x.clone(), w, ref, syn.EPS)
    assert_bits_equal(xd, x2, "x + x")
    assert_close(out, ref, "res == x")


def test_non_default_stream():
    s = torch.cuda.Stream()
    x, w = syn.rms_inputs(256, 1536, torch.bfloat16, 15)
    with torch.cuda.stream(s):
        xd, wd = x.to(DEV), w.to(DEV)
        out = sra.rmsnorm(xd, wd, eps=syn.EPS)
    s.synchronize()
    ref = torch.empty_like(x)
    oracle.rmsnorm(x, w, ref, syn.EPS)
    assert_close(out, ref, "side stream")


def test_companion_large_rows_sampled():
    """The bench's row-scaled shape (65536 x 1536 bf16), compared on sampled rows."""
    rows, D = 65536, 1536
    x, w = syn.rms_inputs(rows, D, torch.bfloat16, 16)
    out = sra.rmsnorm(x.to(DEV), w.to(DEV), eps=syn.EPS).cpu()
    idx = torch.tensor([0, 1, 777, 31337, rows - 1])
    ref = torch.empty(len(idx), D, dtype=torch.bfloat16)
    oracle.rmsnorm(x[idx].contiguous(), w, ref, syn.EPS)
    assert_close(out[idx], ref, "sampled rows")


def _range_rows(D, dtype, seed):
    """Rows whose fp32 sum of squares overflows or underflows, beside ordinary rows.

    The pages accumulate in fp32 to keep bf16 from overflowing
    (koas-w.github.io "preformanceimprovement", section 3); the result asked for
    is still the exact formula, so these rows are compared with the fp64 oracle
    like any other: elements of 2^100 (the sum of squares passes fp32's range),
    one element of 2^120 in an ordinary row, rows of 2^-60 and 2^-130 (bf16 /
    fp32 subnormals), an ordinary row, a zero row, and a row holding one
    infinity. fp16 cannot reach the first four, so its rows stay in range.
    """
    g = syn.normal((8, D), 0, 1, torch.float32, seed, 1).double()
    big, one, tiny, sub = (2.0 ** 100, 2.0 ** 120, 2.0 ** -60, 2.0 ** -130)
    if dtype == torch.float16:
        big, one, tiny, sub = (2.0 ** 12, 2.0 ** 15, 2.0 ** -10, 2.0 ** -20)
    rows = [g[0] * big, g[1].clone(), g[2] * tiny, g[3] * sub, g[4], torch.zeros(D, dtype=torch.float64),
            g[6].clone(), -g[7] * big]
    rows[1][D // 3] = one
    rows[6][D // 2] = float("inf")
    return torch.stack(rows).to(dtype)


@pytest.mark.parametrize("variant", [-1, 0, 1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [1536, 333, 8192])
@pytest.mark.parametrize("eps", [0.0, syn.EPS])
def test_rows_beyond_the_fp32_sum_range(variant, dtype, D, eps):
    """Every variant (and the planner's choice) on rows whose squares overflow or
    underflow fp32: within 1 ulp of the oracle, NaN where the formula gives
    0 * inf (a zero row with eps = 0, an infinite element)."""
    sra.force_variant("rmsnorm", variant)
    try:
        x = _range_rows(D, dtype, 17)
        w = syn.normal((D,), 1, 0.1, dtype, 17, 2)
        try:
            got, ref = run_rms(x, w, eps)
        except sra.SRAError as e:
            assert e.status == -7 and variant >= 0  # this variant cannot hold the row in registers
            return
        assert_close(got, ref, f"rmsnorm variant {variant} [{8},{D}] {dtype} eps={eps}")
        # the fused add: the stored sum is the same big / tiny row
        res = (x.double() * 2.0 ** -8).to(dtype)
        xd = x.to(DEV)
        out = sra.add_rmsnorm(xd, res.to(DEV), w.to(DEV), eps=eps)
        xr, ref = x.clone(), torch.empty_like(x)
        oracle.add_rmsnorm(xr, res, w, ref, eps)
        assert_bits_equal(xd, xr, "residual")
        assert_close(out, ref, f"add_rmsnorm variant {variant} [{8},{D}] {dtype} eps={eps}")
    finally:
        sra.force_variant("rmsnorm", -1)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("g,nv", [(2, 8), (2, 16), (4, 8), (4, 16), (8, 8), (8, 16)])
@pytest.mark.parametrize("rows,D", [(512, 4096), (512, 8192), (300, 6000), (1, 8192), (777, 2056), (9, 5000)])
def test_warps_row_every_group(dtype, g, nv, rows, D):
    """warps_row forced to each (warps per row, accesses per lane) that can hold the row:
    rows of several groups per CTA, fewer rows than groups; rmsnorm and add_rmsnorm
    against the oracle."""
    sra.force_variant("rmsnorm", 8 | (nv << 8) | (g << 16))
    try:
        x, w = syn.rms_inputs(rows, D, dtype, 18)
        try:
            got, ref = run_rms(x, w)
        except sra.SRAError as e:
            assert e.status == -7 and 32 * g * nv < -(-D // (16 // x.element_size()))
            return
        assert_close(got, ref, f"warps_row g{g} nv{nv} [{rows},{D}] {dtype}")
        xa, ra, wa = syn.add_rms_inputs(rows, D, dtype, 19)
        xd = xa.to(DEV)
        buf, out = guarded(xa.shape, dtype)
        sra.add_rmsnorm(xd, ra.to(DEV), wa.to(DEV), out, syn.EPS)
        torch.cuda.synchronize()
        check_guards(buf)
        ref = torch.empty_like(xa)
        oracle.add_rmsnorm(xa, ra, wa, ref, syn.EPS)
        assert_bits_equal(xd, xa, "residual")
        assert_close(out, ref, f"add warps_row g{g} nv{nv} [{rows},{D}] {dtype}")
    finally:
        sra.force_variant("rmsnorm", -1)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [4100, 8190, 2053])
def test_warps_row_ragged_tail(dtype, D):
    """Rows padded to a 16-byte stride with D % (16 / element size) != 0: the scalar
    tail of warps_row (the first threads of the group own one element each)."""
    stride = -(-D // 8) * 8
    rows = 300
    base = syn.normal((rows, stride), 0, 1, dtype, 20, 1)
    x = base[:, :D]
    w = syn.normal((D,), 1, 0.1, dtype, 20, 2)
    sra.force_variant("rmsnorm", 8)
    try:
        xd = base.to(DEV)[:, :D]
        obuf = torch.full((rows, stride), 9.0, dtype=dtype, device=DEV)
        sra.rmsnorm(xd, w.to(DEV), obuf[:, :D], syn.EPS)
        ref = torch.empty(rows, D, dtype=dtype)
        oracle.rmsnorm(x.contiguous(), w, ref, syn.EPS)
        assert_close(obuf[:, :D], ref, f"warps_row tail [{rows},{D}] {dtype}")
        assert bool((obuf[:, D:].cpu().double() == 9).all())
    finally:
        sra.force_variant("rmsnorm", -1)
