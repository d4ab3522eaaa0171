"""GPU parity of msa_quant_fp8 (step a1) against the oracle: bit-exact codes."""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq

pytestmark = pytest.mark.gpu


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("cfg", ["tiny", "prefill8k"])
def test_config_tensors_bit_exact(msa, cfg):
    w = wl.make_gqa(wl.CONFIGS[cfg])
    for name, arr in (("q", w.q), ("idx_q", w.idx_q)):
        got = msa.quant_fp8(_dev_bf16(arr), w.scales[name]).cpu().numpy()
        np.testing.assert_array_equal(got, oq.quantize(arr, w.scales[name]))


def test_prefill32k_sampled_rows_bit_exact(msa):
    # full-size tensors in the launch the benchmark times; oracle on sampled rows
    cfg = wl.CONFIGS["prefill32k"]
    w = wl.make_gqa(cfg)
    g = np.random.default_rng(0)
    for name, arr in (("q", w.q), ("idx_q", w.idx_q)):
        got = msa.quant_fp8(_dev_bf16(arr), w.scales[name]).cpu().numpy()
        rows = g.choice(arr.shape[0], size=512, replace=False)
        np.testing.assert_array_equal(got[rows], oq.quantize(arr[rows], w.scales[name]))


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 7), (5, 48), (257, 128), (1000, 576), (31, 1)])
def test_shapes_and_tails(msa, rows, cols):
    g = np.random.default_rng(rows * 1000 + cols)
    bits = wl.to_bf16_bits(g.standard_normal((rows, cols)).astype(np.float32) * 40)
    got = msa.quant_fp8(_dev_bf16(bits), 0.37).cpu().numpy()
    np.testing.assert_array_equal(got, oq.quantize(bits, 0.37))


def test_strided_and_misaligned_views(msa):
    g = np.random.default_rng(3)
    big = wl.to_bf16_bits(g.standard_normal((64, 160)).astype(np.float32) * 3)
    x = _dev_bf16(big)
    view = x[:, :128]                                   # row stride 160, vector path
    got = msa.quant_fp8(view, 0.01).cpu().numpy()
    np.testing.assert_array_equal(got, oq.quantize(big[:, :128], 0.01))
    view = x[:, 1:129]                                  # 2-byte offset: scalar path
    got = msa.quant_fp8(view, 0.01).cpu().numpy()
    np.testing.assert_array_equal(got, oq.quantize(big[:, 1:129], 0.01))


def test_special_values(msa):
    v = np.array([0.0, -0.0, 448.0, 460.0, 464.0, 500.0, 1e30, -1e30, np.inf, -np.inf, np.nan,
                  2.0 ** -10, 3 * 2.0 ** -10, -(2.0 ** -12), 1.0625, 2.0 ** -9, 240.0, 232.0] * 2,
                 np.float32)
    bits = wl.to_bf16_bits(v)
    got = msa.quant_fp8(_dev_bf16(bits), None).cpu().numpy()
    np.testing.assert_array_equal(got, oq.quantize(bits, None))


def test_fp16_input(msa):
    g = np.random.default_rng(4)
    x = (g.standard_normal((333, 96)) * 20).astype(np.float16)
    got = msa.quant_fp8(torch.from_numpy(x).cuda(), 0.2).cpu().numpy()
    np.testing.assert_array_equal(got, oq.quantize(x.view(np.uint16), 0.2, dtype="fp16"))


def test_empty_and_e5m2(msa):
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    assert msa.quant_fp8(x, 1.0).shape == (0, 128)
    lib = msa.load()
    y = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((4, 16), dtype=torch.uint8, device="cuda")
    import ctypes
    assert lib.msa_quant_fp8(ctypes.c_void_p(y.data_ptr()), 0, 4, 16, 16, ctypes.c_void_p(o.data_ptr()),
                             3, 16, None, None) == 2


def test_multi_launch_equals_separate_calls(msa):
    # Q and idx_q of the 8k workload plus a strided slice (handled by its own
    # launch after the shared one): every output byte-identical to quant_fp8's
    w = wl.make_gqa(wl.CONFIGS["prefill8k"])
    q, iq = _dev_bf16(w.q), _dev_bf16(w.idx_q)
    sl = q[:1000, :, :64]                                   # rows of 64 with stride 128
    outs = msa.quant_fp8_multi([(q, w.scales["q"]), (iq, w.scales["idx_q"]), (sl, 0.75)])
    for got, (x, sc) in zip(outs, [(q, w.scales["q"]), (iq, w.scales["idx_q"]), (sl, 0.75)]):
        assert torch.equal(got, msa.quant_fp8(x, sc))
    assert np.array_equal(outs[1].cpu().numpy(), oq.quantize(w.idx_q, w.scales["idx_q"]))
    # one tensor, and a scale-free entry
    one = msa.quant_fp8_multi([(iq, None)])[0]
    assert np.array_equal(one.cpu().numpy(), oq.quantize(w.idx_q, None))
