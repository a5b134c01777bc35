"""GPU parity: RMSNorm / GLU fused as the prologue of the projection they feed.

m.lsln.cn 21-operator article section 2.2 (ln1 fused into qkv_proj); the same
fusion of the MLP's activation into its down projection. Workloads: the
Qwen2.5-1.5B projections at decode batch sizes 1, 16 and 64: ln1 + qkv_proj
(K = 1536, N = 2048) and silu(gate) * up + down_proj (I = 8960, N = 1536);
x ~ N(0, 1), RMSNorm weight ~ N(1, 0.1), W ~ N(0, 0.02).

Tolerance. The kernels accumulate in fp32 and round the normed (or activated)
rows to the dtype before the product, as the oracle does; an h element whose
fp32 value lands on the other side of a rounding midpoint than the oracle's
moves y by one ulp of h times |W_nk|, and the fp32 sums add about
sqrt(K) * 2^-24 of S[b, n] = sum_k |h[b, k]| |W[n, k]|. The bound: within 1 ulp
of the oracle (bf16 / fp16), or within 1e-5 * S + 4u * max_k |h_k W_nk| (two
such h elements, u the dtype's unit roundoff); fp32: 1e-5 relative + 1e-6 * S.
"""
import pytest
import torch

import oracle
import swiglu_rmsnorm_add_gb300 as sra
from swiglu_rmsnorm_add_gb300 import synthetic as syn
from tests.parity import ulp_distance

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


UNIT = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11, torch.float32: 2.0 ** -24}


def assert_linear_close(got, want, h, W, what):
    got, want = got.cpu(), want.cpu()
    Ha, Wa = h.double().abs(), W.double().abs()
    S = Ha @ Wa.T
    M = (Ha[:, None, :] * Wa[None, :, :]).amax(-1) if h.shape[1] * W.shape[0] * h.shape[0] <= 2 ** 26 else S
    # two h elements on the other side of a rounding midpoint: 2 * 2u * max_k |h_k W_nk|
    atol = 1e-5 * S + 4 * UNIT[want.dtype] * M
    err = (got.double() - want.double()).abs()
    if want.dtype == torch.float32:
        bad = err > 1e-5 * want.double().abs() + 1e-6 * S
    else:
        bad = (ulp_distance(got, want) > 1) & (err > atol)
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} of {bad.numel()} outputs off (max err {float(err.max()):.3g})"


def norm_case(B, K, N, dtype, seed, rows=None, ws=False):
    x = syn.normal((B, K), 0, 1, dtype, seed, 1)
    w = syn.normal((K,), 1, 0.1, dtype, seed, 2)
    W = syn.linear_weight(N, K, dtype, seed)
    wsp = sra.linear_workspace(B, K, dtype, DEV) if ws else None
    got = sra.rmsnorm_linear(x.to(DEV), w.to(DEV), W.to(DEV), workspace=wsp).cpu()
    sel = torch.arange(B) if rows is None else rows
    h = torch.empty(len(sel), K, dtype=dtype)
    oracle.rmsnorm(x[sel].contiguous(), w, h, 1e-6)
    want = torch.empty(len(sel), N, dtype=dtype)
    oracle.linear(h, W, want)
    return got[sel], want, h, W


def glu_case(B, I, N, dtype, seed, act="silu", rows=None, ws=False):
    gu = syn.normal((B, 2 * I), 0, 1, dtype, seed, 3)
    W = syn.linear_weight(N, I, dtype, seed)
    wsp = sra.linear_workspace(B, I, dtype, DEV) if ws else None
    got = sra.glu_linear(gu.to(DEV), W.to(DEV), act=act, workspace=wsp).cpu()
    sel = torch.arange(B) if rows is None else rows
    h = torch.empty(len(sel), I, dtype=dtype)
    oracle.glu(gu[sel].contiguous(), h, act)
    want = torch.empty(len(sel), N, dtype=dtype)
    oracle.linear(h, W, want)
    return got[sel], want, h, W


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("act", ["silu", "relu"])
@pytest.mark.parametrize("B,I,N", [(1, 64, 128), (17, 640, 384), (40, 4160, 640), (64, 8960, 1536), (33, 1024, 256)])
def test_glu_fused_into_the_tcgen05_projection(dtype, act, B, I, N):
    """The GLU computed inside the tcgen05 projection (gate and up tiles by TMA, h's tile made in
    place by eight warps), forced from 1 row: against the oracle's glu then linear."""
    sra.force_variant("linear", 1)
    try:
        before = sra.wait_timeouts()
        got, want, h, W = glu_case(B, I, N, dtype, 1090 + B, act=act)
        torch.cuda.synchronize()
        assert sra.wait_timeouts() == before
    finally:
        sra.force_variant("linear", -1)
    assert_linear_close(got, want, h, W, f"fused glu tcgen05 {act} {dtype} B={B} I={I} N={N}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("B,K,N", [(1, 64, 128), (17, 640, 384), (40, 4160, 640), (64, 1536, 2048), (33, 1024, 256),
                                   (64, 8192, 256)])
def test_rmsnorm_fused_into_the_tcgen05_projection(dtype, B, K, N):
    """The RMSNorm computed inside the tcgen05 projection (the CTA's x tiles by TMA, the
    cluster's partial sums of squares exchanged, h's tiles normed in place), forced from 1 row:
    against the oracle's rmsnorm then linear; no bounded wait runs out."""
    before = sra.wait_timeouts()
    sra.force_variant("linear", 1)
    try:
        got, want, h, W = norm_case(B, K, N, dtype, 1090 + K + B)
    finally:
        sra.force_variant("linear", -1)
    torch.cuda.synchronize()
    assert sra.wait_timeouts() == before
    assert_linear_close(got, want, h, W, f"fused rmsnorm tcgen05 {dtype} B={B} K={K} N={N}")


@pytest.mark.parametrize("splits", [1, 3, 5, 12, 16])
def test_rmsnorm_fused_tcgen05_splits(splits):
    """The fused RMSNorm with its K split forced over clusters of 1-16 CTAs (16 tiles of K,
    ragged ranges at 3, 5 and 12): against the oracle."""
    try:
        sra.force_variant("linear", 1 | (splits << 8))
        try:
            got, want, h, W = norm_case(33, 1024, 256, torch.bfloat16, 1095 + splits)
        finally:
            sra.force_variant("linear", -1)
    except sra.SRAError:
        if splits <= 8:
            raise
        pytest.skip(f"the device cannot place a {splits}-CTA cluster")
    assert_linear_close(got, want, h, W, f"fused rmsnorm tcgen05 splits={splits}")


def test_glu_fused_into_the_tcgen05_projection_far_negative_gates():
    """Gates below -64 in some 8-element chunks take the careful SiLU inside the fused kernel."""
    B, I, N = 24, 1024, 256
    gu = syn.normal((B, 2 * I), 0, 1, torch.bfloat16, 1095, 3)
    gu[:, 5] = -90.0
    gu[3, 17:25] = -200.0
    gu[7, 512] = -70.0
    W = syn.linear_weight(N, I, torch.bfloat16, 1095)
    got = sra.glu_linear(gu.to(DEV), W.to(DEV)).cpu()   # 24 rows: the fused tcgen05 kernel
    h = torch.empty(B, I, dtype=torch.bfloat16)
    oracle.glu(gu, h, "silu")
    want = torch.empty(B, N, dtype=torch.bfloat16)
    oracle.linear(h, W, want)
    assert_linear_close(got, want, h, W, "fused glu far-negative gates")


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("case", ["norm", "silu", "relu"])
@pytest.mark.parametrize("B", [1, 5, 16])
def test_decode_batch_kernel_k_split(case, B, splits):
    """The decode-batch projection kernel with its K split over clusters of 1-8 CTAs forced
    (K = 1664: 26 tiles, so 3, 5 and 8 leave ragged slices; the RMSNorm rows still take their
    norm over the whole row): against the oracle, and the same bytes for every split count up to
    the fp32 sum's order."""
    sra.force_variant("linear_narrow", splits << 8)
    try:
        if case == "norm":
            got, want, h, W = norm_case(B, 1664, 384, torch.bfloat16, 1080 + B)
        else:
            got, want, h, W = glu_case(B, 1664, 384, torch.bfloat16, 1080 + B, act=case)
    finally:
        sra.force_variant("linear_narrow", -1)
    assert_linear_close(got, want, h, W, f"narrow {case} B={B} splits={splits}")


@pytest.mark.parametrize("B", syn.LINEAR_B)
def test_config_qwen25_ln1_qkv(B):
    got, want, h, W = norm_case(B, syn.QWEN25_QKV["K"], syn.QWEN25_QKV["N"], torch.bfloat16, 1030)
    assert_linear_close(got, want, h, W, f"ln1+qkv B={B}")


@pytest.mark.parametrize("B", syn.LINEAR_B)
def test_config_qwen25_swiglu_down(B):
    rows = None if B <= 16 else torch.arange(0, B, 7)
    got, want, h, W = glu_case(B, syn.QWEN25_DOWN["I"], syn.QWEN25_DOWN["N"], torch.bfloat16, 1031, rows=rows)
    assert_linear_close(got, want, h, W, f"swiglu+down B={B}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("B", [1, 5, 16, 17, 33, 64, 100])
@pytest.mark.parametrize("K,N", [(64, 64), (640, 192), (128, 1024), (100, 40), (1536, 2048)])
def test_norm_shapes_dtypes(dtype, B, K, N):
    got, want, h, W = norm_case(B, K, N, dtype, 1032 + K + B)
    assert_linear_close(got, want, h, W, f"norm {dtype} B={B} K={K} N={N}")


@pytest.mark.parametrize("act", ["silu", "relu"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("B,I,N", [(1, 64, 64), (7, 960, 128), (64, 512, 256), (3, 72, 40)])
def test_glu_shapes_dtypes(act, dtype, B, I, N):
    got, want, h, W = glu_case(B, I, N, dtype, 1033 + I + B, act)
    assert_linear_close(got, want, h, W, f"{act} {dtype} B={B} I={I} N={N}")


def test_strided_rows_and_outputs():
    """x rows padded (row stride K + 64), y written into a wider buffer: guard columns untouched."""
    B, K, N = 20, 512, 256
    base = syn.normal((B, K + 64), 0, 1, torch.bfloat16, 1034, 1)
    x = base[:, :K]
    w = syn.normal((K,), 1, 0.1, torch.bfloat16, 1034, 2)
    W = syn.linear_weight(N, K, torch.bfloat16, 1034)
    ybuf = torch.full((B, N + 8), 3.0, dtype=torch.bfloat16, device=DEV)
    sra.rmsnorm_linear(base.to(DEV)[:, :K], w.to(DEV), W.to(DEV), ybuf[:, :N])
    h = torch.empty(B, K, dtype=torch.bfloat16)
    oracle.rmsnorm(x.contiguous(), w, h, 1e-6)
    want = torch.empty(B, N, dtype=torch.bfloat16)
    oracle.linear(h, W, want)
    assert_linear_close(ybuf[:, :N], want, h, W, "strided")
    assert bool((ybuf[:, N:].cpu() == 3.0).all())


@pytest.mark.parametrize("prologue", ["rmsnorm", "silu"])
def test_strided_rows_and_outputs_fused_tcgen05(prologue):
    """The one-launch tcgen05 kernels (forced) on padded input rows (row stride K + 64, or 2K + 64
    for gate_up) writing into a wider y: matches the oracle, guard columns untouched."""
    B, K, N = 20, 512, 256
    W = syn.linear_weight(N, K, torch.bfloat16, 1097)
    ybuf = torch.full((B, N + 8), 3.0, dtype=torch.bfloat16, device=DEV)
    h = torch.empty(B, K, dtype=torch.bfloat16)
    sra.force_variant("linear", 1)
    try:
        if prologue == "rmsnorm":
            base = syn.normal((B, K + 64), 0, 1, torch.bfloat16, 1097, 1)
            w = syn.normal((K,), 1, 0.1, torch.bfloat16, 1097, 2)
            sra.rmsnorm_linear(base.to(DEV)[:, :K], w.to(DEV), W.to(DEV), ybuf[:, :N])
            oracle.rmsnorm(base[:, :K].contiguous(), w, h, 1e-6)
        else:
            base = syn.normal((B, 2 * K + 64), 0, 1, torch.bfloat16, 1097, 3)
            sra.glu_linear(base.to(DEV)[:, :2 * K], W.to(DEV), ybuf[:, :N])
            oracle.glu(base[:, :2 * K].contiguous(), h, "silu")
    finally:
        sra.force_variant("linear", -1)
    want = torch.empty(B, N, dtype=torch.bfloat16)
    oracle.linear(h, W, want)
    assert_linear_close(ybuf[:, :N], want, h, W, f"strided, fused tcgen05 {prologue}")
    assert bool((ybuf[:, N:].cpu() == 3.0).all())


def test_llama3_8b_down_sampled():
    """The Llama-3-8B down projection (I = 14336, N = 4096) at batch 64, sampled rows."""
    rows = torch.tensor([0, 13, 40, 63])
    got, want, h, W = glu_case(64, 14336, 4096, torch.bfloat16, 1035, rows=rows)
    assert_linear_close(got, want, h, W, "llama3 down")


@pytest.mark.parametrize("B", [1, 17, 32, 33, 64, 100])
def test_workspace_config_qwen25(B):
    """The workspace entry points (norm / activation in their own kernel from 32 rows, the
    projection over h) on the Qwen2.5-1.5B projections."""
    got, want, h, W = norm_case(B, syn.QWEN25_QKV["K"], syn.QWEN25_QKV["N"], torch.bfloat16, 1036, ws=True)
    assert_linear_close(got, want, h, W, f"ws ln1+qkv B={B}")
    rows = None if B <= 17 else torch.arange(0, B, 7)
    got, want, h, W = glu_case(B, syn.QWEN25_DOWN["I"], syn.QWEN25_DOWN["N"], torch.bfloat16, 1037, rows=rows,
                               ws=True)
    assert_linear_close(got, want, h, W, f"ws swiglu+down B={B}")


@pytest.mark.parametrize("act", ["silu", "relu"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("B,K,N", [(32, 64, 64), (50, 640, 192), (64, 512, 256), (96, 100, 40)])
def test_workspace_shapes_dtypes(act, dtype, B, K, N):
    got, want, h, W = norm_case(B, K, N, dtype, 1038 + K + B, ws=True)
    assert_linear_close(got, want, h, W, f"ws norm {dtype} B={B} K={K} N={N}")
    got, want, h, W = glu_case(B, K, N, dtype, 1039 + K + B, act, ws=True)
    assert_linear_close(got, want, h, W, f"ws {act} {dtype} B={B} I={K} N={N}")


def test_workspace_equals_its_two_steps():
    """From 32 rows the workspace path is the RMSNorm kernel writing h into the workspace,
    then the projection of h: the workspace ends up holding exactly sra.rmsnorm's output,
    and y matches the oracle's projection of that h."""
    B, K, N = 64, 1536, 2048
    x = syn.normal((B, K), 0, 1, torch.bfloat16, 1040, 1).to(DEV)
    w = syn.normal((K,), 1, 0.1, torch.bfloat16, 1040, 2).to(DEV)
    W = syn.linear_weight(N, K, torch.bfloat16, 1040).to(DEV)
    ws = sra.linear_workspace(B, K, torch.bfloat16, DEV)
    y = sra.rmsnorm_linear(x, w, W, workspace=ws)
    h = sra.rmsnorm(x, w, eps=1e-6)
    assert torch.equal(ws.view(B, K).view(torch.int16), h.view(torch.int16))  # the workspace holds h
    want = torch.empty(B, N, dtype=torch.bfloat16)
    oracle.linear(h.cpu(), W.cpu(), want)
    assert_linear_close(y, want, h.cpu(), W.cpu(), "ws two steps")


_SELFTEST_TIMEOUTS = [0]  # timeouts the self-test below causes on purpose


def test_no_wait_ran_out():
    """The tile copies of every call above landed within their bounded waits."""
    x = syn.normal((64, 1536), 0.0, 1.0, torch.bfloat16, 77, 1).to(DEV)
    w = syn.normal((1536,), 1.0, 0.1, torch.bfloat16, 77, 2).to(DEV)
    W = syn.linear_weight(2048, 1536, torch.bfloat16, 77).to(DEV)
    sra.rmsnorm_linear(x, w, W, eps=syn.EPS)
    torch.cuda.synchronize()
    assert sra.wait_timeouts() == _SELFTEST_TIMEOUTS[0]


def test_bounded_wait_gives_up():
    """A wait on a barrier that nothing completes gives up after its bound, is counted, and
    leaves the GPU usable (the calls after it run and match the oracle)."""
    before = sra.wait_timeouts()
    assert sra.wait_selftest(DEV) == 0
    torch.cuda.synchronize()
    _SELFTEST_TIMEOUTS[0] += 1
    assert sra.wait_timeouts() == before + 1
    got, want, h, W = norm_case(64, 1536, 2048, torch.bfloat16, 1041)
    assert_linear_close(got, want, h, W, "after the self-test")


@pytest.mark.parametrize("eps", [0.0, 1e-6])
@pytest.mark.parametrize("dtype,B,K,N,ws", [
    (torch.bfloat16, 1, 1536, 2048, False),     # decode-batch kernel
    (torch.bfloat16, 16, 1536, 2048, False),
    (torch.bfloat16, 64, 1536, 2048, False),    # the RMSNorm fused into the tcgen05 projection
    (torch.bfloat16, 64, 1536, 2048, True),     # prologue kernel into a workspace
    (torch.float16, 33, 640, 192, False),
    (torch.float16, 33, 640, 256, False),       # the RMSNorm fused into the tcgen05 projection
    (torch.float32, 5, 640, 192, False),        # CUDA-core kernel
    (torch.bfloat16, 3, 100, 40, False),
])
def test_norm_rows_beyond_the_fp32_sum_range(eps, dtype, B, K, N, ws):
    """RMSNorm prologue rows whose fp32 sum of squares overflows (elements of 2^100)
    or loses its digits (2^-60 and 2^-130 with eps = 0) beside ordinary rows: the
    fused projection equals the oracle's rmsnorm then linear, as on any row."""
    x = syn.normal((B, K), 0, 1, torch.float32, 1035, 1).double()
    scales = [2.0 ** 100, 2.0 ** -130, 1.0, 2.0 ** -60] if dtype != torch.float16 else [2.0 ** 12, 2.0 ** -10, 1.0]
    for b in range(B):
        x[b] *= scales[b % len(scales)]
    x = x.to(dtype)
    w = syn.normal((K,), 1, 0.1, dtype, 1035, 2)
    W = syn.linear_weight(N, K, dtype, 1035)
    wsp = sra.linear_workspace(B, K, dtype, DEV) if ws else None
    got = sra.rmsnorm_linear(x.to(DEV), w.to(DEV), W.to(DEV), eps=eps, workspace=wsp).cpu()
    h = torch.empty(B, K, dtype=dtype)
    oracle.rmsnorm(x, w, h, eps)
    assert bool(torch.isfinite(h.float()).all())
    want = torch.empty(B, N, dtype=dtype)
    oracle.linear(h, W, want)
    assert_linear_close(got, want, h, W, f"norm range {dtype} B={B} K={K} eps={eps} ws={ws}")


def _tc_case(prologue, dtype, B, K, N, seed, force=1, l2=False):
    """The workspace path with its projection forced onto the tcgen05 kernel (`force`: the
    variant word, K splits and ring depth included); with `l2`, a workspace large enough for
    the K split's partials, which are then summed through L2."""
    W = syn.linear_weight(N, K, dtype, seed)
    wsp = sra.linear_workspace(B, K, dtype, DEV, N if l2 else None)
    sra.force_variant("linear", force)
    try:
        if prologue == "rmsnorm":
            x = syn.normal((B, K), 0, 1, dtype, seed, 1)
            w = syn.normal((K,), 1, 0.1, dtype, seed, 2)
            got = sra.rmsnorm_linear(x.to(DEV), w.to(DEV), W.to(DEV), workspace=wsp).cpu()
            h = torch.empty(B, K, dtype=dtype)
            oracle.rmsnorm(x, w, h, 1e-6)
        else:
            gu = syn.normal((B, 2 * K), 0, 1, dtype, seed, 3)
            got = sra.glu_linear(gu.to(DEV), W.to(DEV), act=prologue, workspace=wsp).cpu()
            h = torch.empty(B, K, dtype=dtype)
            oracle.glu(gu, h, prologue)
    finally:
        sra.force_variant("linear", -1)
    want = torch.empty(B, N, dtype=dtype)
    oracle.linear(h, W, want)
    return got, want, h, W


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("prologue,B,K,N", [
    ("rmsnorm", 32, 64, 128),       # one tile of K, one slice
    ("rmsnorm", 33, 640, 256),      # ragged rows, K split
    ("rmsnorm", 64, 1536, 2048),    # Qwen2.5-1.5B ln1 + qkv_proj, batch 64
    ("silu", 64, 8960, 1536),       # Qwen2.5-1.5B SwiGLU + down_proj, batch 64
    ("relu", 48, 1024, 384),
    ("silu", 40, 4160, 640),        # K tiles not a multiple of the cluster's splits
])
def test_tcgen05_projection(dtype, prologue, B, K, N):
    """The projection of h on the fifth-generation tensor cores (W tile as the MMA's A
    operand, h as B, fp32 accumulator in tensor memory) against the oracle's rmsnorm /
    glu then linear, at the fused projections' tolerance; no bounded wait runs out."""
    before = sra.wait_timeouts()
    got, want, h, W = _tc_case(prologue, dtype, B, K, N, 1050 + K + B)
    torch.cuda.synchronize()
    assert sra.wait_timeouts() == before
    assert_linear_close(got, want, h, W, f"tcgen05 {prologue} {dtype} B={B} K={K} N={N}")


@pytest.mark.parametrize("l2", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("prologue,B,K,N", [
    ("rmsnorm", 32, 64, 128),
    ("rmsnorm", 33, 640, 256),
    ("silu", 64, 8960, 1536),
    ("relu", 48, 1024, 384),
    ("silu", 40, 4160, 640),
])
def test_tcgen05_projection_partials_through_l2(dtype, prologue, B, K, N, l2):
    """The K split summed through the cluster's shared memory (a workspace of B * K elements)
    and through L2 (the size sra_linear_workspace_size gives): both against the oracle."""
    before = sra.wait_timeouts()
    got, want, h, W = _tc_case(prologue, dtype, B, K, N, 1070 + K + B, l2=l2)
    torch.cuda.synchronize()
    assert sra.wait_timeouts() == before
    assert_linear_close(got, want, h, W, f"tcgen05 l2={l2} {prologue} {dtype} B={B} K={K} N={N}")


@pytest.mark.parametrize("stages", [4, 8])
@pytest.mark.parametrize("splits", [1, 3, 5, 12, 16])
@pytest.mark.parametrize("prologue,B,K,N", [("silu", 64, 8960, 1536), ("rmsnorm", 33, 1280, 256)])
def test_tcgen05_ring_depth_and_splits(prologue, B, K, N, splits, stages):
    """Both ring depths of the tcgen05 projection and K splits that are not powers of two
    (clusters of 3, 5 and 12 CTAs; 16 is a non-portable size) against the oracle."""
    before = sra.wait_timeouts()
    try:
        got, want, h, W = _tc_case(prologue, torch.bfloat16, B, K, N, 1062 + splits,
                                   force=1 | (splits << 8) | (stages << 16), l2=splits % 2 == 1)
    except sra.SRAError:
        if splits <= 8:
            raise
        pytest.skip(f"the device cannot place a {splits}-CTA cluster with a {stages}-stage ring")
    torch.cuda.synchronize()
    assert sra.wait_timeouts() == before
    assert_linear_close(got, want, h, W, f"tcgen05 {prologue} splits={splits} stages={stages}")


def test_tcgen05_forced_where_it_cannot_serve():
    """Forced onto the tcgen05 kernel, a call it cannot serve (more than 64 rows, or N not a
    multiple of 128) fails before anything is enqueued; smaller batches, which take the fused
    kernel without a workspace split, still run."""
    W = syn.linear_weight(192, 256, torch.bfloat16, 1060).to(DEV)
    x = syn.normal((80, 256), 0, 1, torch.bfloat16, 1060, 1).to(DEV)
    w = syn.normal((256,), 1, 0.1, torch.bfloat16, 1060, 2).to(DEV)
    sra.force_variant("linear", 1)
    try:
        with pytest.raises(sra.SRAError):
            sra.rmsnorm_linear(x, w, W, workspace=sra.linear_workspace(80, 256, torch.bfloat16, DEV))
        with pytest.raises(sra.SRAError):
            sra.rmsnorm_linear(x[:40], w, W, workspace=sra.linear_workspace(40, 256, torch.bfloat16, DEV))
        y = sra.rmsnorm_linear(x[:8], w, W, workspace=sra.linear_workspace(8, 256, torch.bfloat16, DEV))
        torch.cuda.synchronize()
        assert bool(torch.isfinite(y.float()).all())
    finally:
        sra.force_variant("linear", -1)


@pytest.mark.parametrize("variant", [0, 1])
def test_workspace_projection_both_kernels(variant):
    """SwiGLU + down_proj at batch 64 over a workspace with the projection forced onto the
    mma.sync kernel (0) and onto the tcgen05 kernel (1): both match the oracle."""
    B, I, N = 64, 8960, 1536
    gu = syn.normal((B, 2 * I), 0, 1, torch.bfloat16, 1061, 3)
    W = syn.linear_weight(N, I, torch.bfloat16, 1061)
    sra.force_variant("linear", variant)
    try:
        got = sra.glu_linear(gu.to(DEV), W.to(DEV), workspace=sra.linear_workspace(B, I, torch.bfloat16, DEV)).cpu()
    finally:
        sra.force_variant("linear", -1)
    rows = torch.arange(0, B, 5)
    h = torch.empty(len(rows), I, dtype=torch.bfloat16)
    oracle.glu(gu[rows].contiguous(), h, "silu")
    want = torch.empty(len(rows), N, dtype=torch.bfloat16)
    oracle.linear(h, W, want)
    assert_linear_close(got[rows], want, h, W, f"down_proj over a workspace, linear variant {variant}")
