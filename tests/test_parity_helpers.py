"""The tolerance helpers the GPU parity tests use, checked on hand-made cases (CPU).

A helper that accepted too much would let every GPU test pass, so each rule is
tried on both sides of its bound: 1 ulp passes and 2 do not (across zero and
at the largest finite value too), NaN and infinity must match exactly, and the
fp32 bound is relative even for outputs near zero.
"""
import math

import pytest
import torch

from tests.parity import assert_bits_equal, assert_close, assert_values_equal, ulp_distance


def _bits16(vals, dtype):
    return torch.tensor(vals, dtype=torch.int32).to(torch.int16).view(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_ulp_distance_crosses_zero_and_signs(dtype):
    # +0 and -0 are 0 apart; the smallest positive and negative subnormals are 2 apart
    a = _bits16([0x0000, 0x0001, 0x0001, 0x3C00], dtype)
    b = _bits16([-0x8000, -0x7FFF, 0x0002, 0x3C02], dtype)
    assert ulp_distance(a, b).tolist() == [0, 2, 1, 2]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_one_ulp_passes_two_fail(dtype):
    want = torch.tensor([1.0, -3.0, 1e-3], dtype=dtype)
    one = (want.view(torch.int16) + 1).view(dtype)
    assert_close(one, want)
    two = (want.view(torch.int16) + 2).view(dtype)
    with pytest.raises(AssertionError):
        assert_close(two, want)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_specials_must_match(dtype):
    want = torch.tensor([math.nan, math.inf, -math.inf, 1.0], dtype=dtype)
    assert_close(want.clone(), want)
    for bad in ([1.0, math.inf, -math.inf, 1.0],          # NaN lost
                [math.nan, -math.inf, -math.inf, 1.0],    # wrong infinity
                [math.nan, math.inf, -math.inf, math.nan]):  # NaN invented
        with pytest.raises(AssertionError):
            assert_close(torch.tensor(bad, dtype=dtype), want)
    # the largest finite value is 1 ulp from infinity in the bit order; that is not a pass
    big = torch.tensor([torch.finfo(dtype).max], dtype=dtype)
    with pytest.raises(AssertionError):
        assert_close(big, torch.tensor([math.inf], dtype=dtype))


def test_fp32_relative_bound_holds_near_zero():
    want = torch.tensor([1.0, 1e-20, -3e-30], dtype=torch.float32)
    assert_close(want * (1 + 0.9e-5), want)
    with pytest.raises(AssertionError):
        assert_close(want * torch.tensor([1.0, 1 + 2e-5, 1.0]), want)   # a small output held to 1e-5 too
    sub = torch.tensor([2.0 ** -149 * 7], dtype=torch.float32)
    assert_close(sub + 2.0 ** -149, sub)   # subnormal spacing is covered by the 2^-140 floor


def test_bit_and_value_equality():
    a = torch.tensor([0.0, 1.0], dtype=torch.bfloat16)
    b = torch.tensor([-0.0, 1.0], dtype=torch.bfloat16)
    assert_values_equal(a, b)
    with pytest.raises(AssertionError):
        assert_bits_equal(a, b)
