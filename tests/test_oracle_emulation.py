"""The oracle's emulation of the kernels' intended numerics (diagnostic).

With P kept in fp32 and no output rounding, the emulation's blockwise lazy
softmax is algebraically the float64 oracle, so the two agree to fp32
rounding: that pins the emulation. The other cases predict what each
precision choice of the kernels costs against the float64 oracle: the
designs built (f16 P in prefill, two e4m3 terms in decode) sit inside the
parity bars, and a single e4m3 P term does not (which is why neither kernel
uses it)."""

import numpy as np
import pytest

from fp8_block_sparse_gb300 import workloads as wl
from oracle import attention as oa, emulate as em, index_topk as oi, mla as om, quant as oq

BAR_ABS, BAR_REL, BAR_LSE = 4e-2, 1e-2, 2e-3


def _args(w):
    q8 = oq.quantize(w.q, w.scales["q"])
    k8 = oq.quantize(w.k_pool, w.scales["k"])
    v8 = oq.quantize(w.v_pool, w.scales["v"])
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    ids, _ = oi.index_topk(iq, ik, w.page_table, w.seq_lens, w.cu_q, w.cfg.topk)
    return (q8, k8, v8, w.page_table, w.seq_lens, w.cu_q, ids, w.sink, w.sm_scale,
            w.scales["q"], w.scales["k"], w.scales["v"])


def _errors(args, **kw):
    ref = oa.sparse_attention(*args)
    o, ml, lse = em.emulate_attention(*args, **kw)
    return (np.abs(o - ref[0]).max(), np.linalg.norm(o - ref[0]) / np.linalg.norm(ref[0]),
            np.abs(lse - ref[2]).max(), np.abs(ml - ref[1]).max())


@pytest.fixture(scope="module")
def tiny():
    return _args(wl.make_gqa(wl.CONFIGS["tiny"], T_override=300))


@pytest.fixture(scope="module")
def decode():
    cfg = wl.GQAConfig("emu_dec", 24, (), 1, 16, 2, 4, 128, 128, 16, "channel",
                       len_range=(100, 9000), max_pages=80, pool_factor=1.2, seed=52)
    return _args(wl.make_gqa(cfg))


@pytest.mark.parametrize("head", [0.0, 4.0])
def test_fp32_p_without_output_rounding_is_the_oracle(tiny, decode, head):
    for args in (tiny, decode):
        err, rel, lerr, merr = _errors(args, p_format="fp32", head=head, round_out=False)
        assert rel < 1e-6 and lerr < 1e-5 and merr < 1e-5, (err, rel, lerr, merr)


def test_bf16_rounding_helper():
    import torch
    x = np.array([1.0, 1.00390625, 1.01171875, -3.0e-3, 65504.0], np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: to even (1); 1 + 3*2^-8 is a
    # tie between 1 + 2^-7 and 1 + 2^-6: to even (1 + 2^-6)
    np.testing.assert_array_equal(em.bf16_round(x)[:3], [1.0, 1.0, 1.015625])
    g = np.random.default_rng(0)
    y = (g.standard_normal(100000) * np.exp(g.uniform(-20, 20, 100000))).astype(np.float32)
    y = np.concatenate([x, y])
    want = torch.from_numpy(y).to(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(em.bf16_round(y), want)


def test_prefill_design_f16_p_is_inside_the_bars(tiny):
    err, rel, lerr, _ = _errors(tiny, **em.PREFILL)
    assert err <= BAR_ABS and rel <= BAR_REL and lerr <= BAR_LSE


def test_decode_design_two_e4m3_terms_is_inside_the_bars(decode):
    err, rel, lerr, _ = _errors(decode, **em.DECODE)
    assert err <= BAR_ABS and rel <= BAR_REL and lerr <= BAR_LSE


@pytest.mark.parametrize("which", ["tiny", "decode"])
def test_single_e4m3_p_fails_the_relative_bar(tiny, decode, which):
    args = tiny if which == "tiny" else decode
    _, rel, _, _ = _errors(args, p_format="e4m3")
    assert rel > BAR_REL


@pytest.fixture(scope="module")
def mla():
    w = wl.make_mla(wl.CONFIGS["mla"], T_override=6, S_override=3000, topk_override=512, len_range=(200, 512))
    return (oq.quantize(w.q, w.scales["q"]), oq.quantize(w.kv, w.scales["kv"]), w.indices, w.topk_length,
            w.sink, w.sm_scale, w.scales["q"], w.scales["kv"])


def _mla_errors(args, **kw):
    ref = om.sparse_mla(*args)
    o, ml, lse = em.emulate_mla(*args, **kw)
    return (np.abs(o - ref[0]).max(), np.linalg.norm(o - ref[0]) / np.linalg.norm(ref[0]),
            np.abs(lse - ref[2]).max(), np.abs(ml - ref[1]).max())


def test_mla_emulation_fp32_is_the_oracle_and_f16_is_inside_the_bars(mla):
    err, rel, lerr, merr = _mla_errors(mla, p_format="fp32", round_out=False)
    assert rel < 1e-6 and lerr < 1e-5 and merr < 1e-5, (err, rel, lerr, merr)
    err, rel, lerr, _ = _mla_errors(mla)
    assert err <= BAR_ABS and rel <= BAR_REL and lerr <= BAR_LSE
