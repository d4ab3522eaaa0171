"""Pins for the oracle's quantiser (step a1)."""

import numpy as np
import pytest
import torch

from oracle import e4m3, quant
from fp8_block_sparse_gb300 import workloads as wl


def _bf16(x):
    return wl.to_bf16_bits(np.asarray(x, np.float32))


@pytest.mark.parametrize("scale", [None, 1.0, 0.0123, 0.25, 3.7, 1.0 / 448])
def test_matches_torch_scale_then_cast(scale):
    g = np.random.default_rng(7)
    x = _bf16(g.standard_normal((257, 96)).astype(np.float32) * 2.0)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    amax = float(xf.abs().max())
    if scale is not None and amax / scale > 464:   # keep inside torch's non-NaN range
        scale = amax / 448
    s_inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(1.0 if scale is None else scale,
                                                                  dtype=torch.float32)
    ref = (xf * s_inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(quant.quantize(x, scale), ref)


def test_fp16_input_matches_torch():
    g = np.random.default_rng(8)
    x = (g.standard_normal((64, 128)) * 10).astype(np.float16)
    ref = (torch.from_numpy(x).float() * (1.0 / 0.5)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(quant.quantize(x.view(np.uint16), 0.5, dtype="fp16"), ref)


def test_unit_scale_is_identity_on_e4m3_exact_inputs():
    # strictly monotone e4m3-exact integers, the style of test input the
    # vLLM PR 45892 page uses so fp8 and bf16 paths agree exactly
    exact = [*range(1, 17), *range(18, 33, 2), *range(36, 65, 4), *range(72, 129, 8),
             *range(144, 257, 16), *range(288, 449, 32)]
    v = np.array(exact + [-e for e in exact] + [0.0, 2.0 ** -9, 0.375], np.float32)
    codes = quant.quantize(_bf16(v), None)
    np.testing.assert_array_equal(e4m3.decode(codes), v.astype(np.float64))


def test_absent_scale_equals_unit_scale():
    g = np.random.default_rng(9)
    x = _bf16(g.standard_normal(5000).astype(np.float32) * 50)
    np.testing.assert_array_equal(quant.quantize(x, None), quant.quantize(x, 1.0))


def test_scale_is_applied_as_fp32_inverse_then_one_multiply():
    # the inverse is the IEEE single quotient 1.0f/scale
    assert quant.scale_inverse(3.0) == np.float32(1.0) / np.float32(3.0)
    x = _bf16([3.0, 6.0, 1.5])
    np.testing.assert_array_equal(quant.quantize(x, 3.0),
                                  e4m3.encode(np.array([1.0, 2.0, 0.5], np.float32)))
    # 2.125 * (1/2) = 1.0625 lies exactly halfway between e4m3 1.0 and 1.125
    # and rounds to the even code 0x38 (1.0)
    assert quant.quantize(_bf16([2.125]), 2.0)[0] == 0x38
    assert quant.quantize(_bf16([2.375]), 2.0)[0] == 0x3A   # 1.1875 -> 1.25 (even)


def test_scale_inverse_is_the_fp32_reciprocal_of_the_fp32_scale():
    # reading 1 (sglang PR 25460 page, fp8_quantize excerpt: a host-side
    # scale_inv): one IEEE single division of 1 by the scale rounded to fp32,
    # checked against torch's fp32 division
    g = np.random.default_rng(9)
    scales = np.concatenate([g.uniform(1e-4, 10.0, 4000), [0.0123, 3.7, 1.0 / 448, 0.1, 1.0 / 3]])
    want = (torch.ones(len(scales), dtype=torch.float32) /
            torch.from_numpy(scales).to(torch.float32)).numpy()
    got = np.array([quant.scale_inverse(float(s)) for s in scales], dtype=np.float32)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    # the check is sensitive: dividing in float64 first rounds differently for some scales
    f64_first = np.array([np.float32(1.0 / s) for s in scales], dtype=np.float32)
    assert np.any(f64_first.view(np.uint32) != want.view(np.uint32))
    assert quant.scale_inverse(None) == np.float32(1.0)
