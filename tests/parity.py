"""Parity comparison between the CUDA path and the oracle (test helper).

Tolerance (stated once, used by every GPU test):
  * bf16 / fp16 outputs: |gpu - oracle| <= 1 ulp, measured as the distance
    between the two bit patterns in the format's ordered encoding (so the ulp is
    the one at the oracle's rounded value; +0 and -0 are 0 apart);
  * fp32 outputs: |gpu - oracle| <= 1e-5 * |oracle| + 2^-140 (relative 1e-5;
    the floor only covers outputs in fp32's subnormal range, whose spacing is
    2^-149, so an output near zero is still held to 1e-5 of its own size);
  * in every format NaN must meet NaN and an infinity the same infinity;
  * bit-exact where the method fixes the bits (cache placement, untouched
    bytes, the residual update, V copies, ReGLU).
"""
from __future__ import annotations

import torch

FP32_REL = 1e-5
FP32_ABS = 2.0 ** -140


def _ordered16(t: torch.Tensor) -> torch.Tensor:
    a = t.contiguous().view(torch.int16).to(torch.int32)
    return torch.where(a < 0, -(a & 0x7FFF), a)


def ulp_distance(got: torch.Tensor, want: torch.Tensor) -> torch.Tensor:
    assert got.dtype == want.dtype and got.dtype in (torch.bfloat16, torch.float16)
    return (_ordered16(got.cpu()) - _ordered16(want.cpu())).abs()


def _specials_match(got: torch.Tensor, want: torch.Tensor, what: str) -> torch.Tensor:
    """Checks NaN and infinity placement; returns the mask of finite oracle values."""
    g, w = got.float(), want.float()
    nan = torch.isnan(w)
    assert torch.equal(torch.isnan(g), nan), f"{what}: NaN mismatch ({int((torch.isnan(g) != nan).sum())})"
    inf = torch.isinf(w)
    bad = inf & (g != w)
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} infinities not matched"
    gi = torch.isinf(g) & ~inf
    assert not bool(gi.any()), f"{what}: {int(gi.sum())} finite oracle values came out infinite"
    return ~(nan | inf)


def assert_close(got: torch.Tensor, want: torch.Tensor, what: str = "") -> None:
    got, want = got.cpu(), want.cpu()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    fin = _specials_match(got, want, what)
    if got.dtype == torch.float32:
        g, w = got.double()[fin], want.double()[fin]
        if w.numel() == 0:
            return
        err = (g - w).abs()
        bound = FP32_REL * w.abs() + FP32_ABS
        bad = err > bound
        assert not bool(bad.any()), (
            f"{what}: {int(bad.sum())} fp32 values off; max rel {float((err / w.abs().clamp_min(1e-30)).max()):.3g}")
        return
    d = ulp_distance(got, want)
    bad = (d > 1) & fin
    assert not bool(bad.any()), (
        f"{what}: {int(bad.sum())} of {d.numel()} outputs beyond 1 ulp (max {int(d[fin].max())}); "
        f"first at {tuple(int(i) for i in bad.nonzero()[0])}")


def assert_bits_equal(got: torch.Tensor, want: torch.Tensor, what: str = "") -> None:
    got, want = got.cpu().contiguous(), want.cpu().contiguous()
    assert got.shape == want.shape, what
    iv = torch.int32 if got.element_size() == 4 else torch.int16
    a, b = got.view(iv), want.view(iv)
    bad = a != b
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} elements differ bitwise"


def assert_values_equal(got: torch.Tensor, want: torch.Tensor, what: str = "") -> None:
    """Bit-exact except that +0 and -0 count as equal."""
    got, want = got.cpu(), want.cpu()
    if got.dtype == torch.float32:
        g, w = got.view(torch.int32), want.view(torch.int32)
        zero = ((g & 0x7FFFFFFF) == 0) & ((w & 0x7FFFFFFF) == 0)
    else:
        g, w = got.view(torch.int16), want.view(torch.int16)
        zero = ((g & 0x7FFF) == 0) & ((w & 0x7FFF) == 0)
    bad = (g != w) & ~zero
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} elements differ"
