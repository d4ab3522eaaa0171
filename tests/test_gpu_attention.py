"""GPU parity of msa_sparse_attn_fwd (steps a4/a5) against the oracle.

Bar (stated for this path): O within max-abs 4e-2 and relative Frobenius
1e-2 of the float64 oracle, lse within 2e-3 absolute; max_logit is an fp32
dot times the folded scale and is held to 1e-4 relative.
"""

import numpy as np
import pytest

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, attention as oa
from gpu_helpers import dev, sample_tokens, sample_extremes

pytestmark = pytest.mark.gpu


def _codes(w):
    return (oq.quantize(w.q, w.scales["q"]), oq.quantize(w.k_pool, w.scales["k"]),
            oq.quantize(w.v_pool, w.scales["v"]))


def _check(got, ref, tol_abs=4e-2, tol_rel=1e-2, tol_lse=2e-3, bf16_term=False):
    """bf16_term adds the output's own rounding (half a bf16 ulp, 2**-9 |O|,
    doubled for margin) to the absolute bar: only for cases whose |O| runs far
    beyond the configs' range, where bf16 storage alone exceeds 4e-2."""
    o, ml, lse = got
    o_ref, ml_ref, lse_ref = ref
    allowed = tol_abs + (2.0 ** -8 * np.abs(o_ref) if bf16_term else 0.0)
    err = np.abs(o - o_ref)
    rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    assert np.all(err <= allowed) and rel <= tol_rel, (err.max(), rel)
    assert np.abs(lse - lse_ref).max() <= tol_lse * (max(1.0, np.abs(lse_ref).max() * 2.0 ** -12) if bf16_term else 1.0)
    fin = np.isfinite(ml_ref)
    assert np.array_equal(fin, np.isfinite(ml))
    np.testing.assert_allclose(ml[fin], ml_ref[fin], rtol=1e-4, atol=1e-5)
    return err.max(), rel


def run_attention(msa, w, ids, tokens=None, sink=True, scales=True):
    q8, k8, v8 = _codes(w)
    sc = w.scales if scales else {"q": None, "k": None, "v": None}
    s = w.sink if sink else None
    o, ml, lse = msa.sparse_attn_fwd(dev(q8), dev(k8), dev(v8), dev(w.page_table), dev(w.seq_lens),
                                     dev(w.cu_q), dev(ids), None if s is None else dev(s), w.sm_scale,
                                     sc["q"], sc["k"], sc["v"], w.max_q_len)
    msa.check_errors()
    tok = np.arange(w.T) if tokens is None else np.asarray(tokens)
    got = (o.float().cpu().numpy()[tok].astype(np.float64), ml.cpu().numpy()[tok],
           lse.cpu().numpy()[tok])
    ref = oa.sparse_attention(q8, k8, v8, w.page_table, w.seq_lens, w.cu_q, ids, s, w.sm_scale,
                              sc["q"], sc["k"], sc["v"], tokens=tok)
    return _check(got, ref, bf16_term=not scales)


def test_tiny_all_rows(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"])
    ids = wl.random_topk(0, w.seq_lens, w.cu_q, w.cfg.Hidx, w.cfg.topk)
    run_attention(msa, w, ids)


@pytest.mark.parametrize("T", [1, 17, 129, 1000])
def test_ragged(msa, T):
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=T)
    ids = wl.random_topk(T, w.seq_lens, w.cu_q, w.cfg.Hidx, w.cfg.topk)
    run_attention(msa, w, ids)


@pytest.mark.parametrize("topk", [1, 2, 5])
def test_topk_sizes(msa, topk):
    w = wl.make_gqa(wl.CONFIGS["prefill8k"], T_override=1500)
    ids = wl.random_topk(topk, w.seq_lens, w.cu_q, w.cfg.Hidx, topk)
    run_attention(msa, w, ids)


@pytest.mark.parametrize("hq,hkv,hidx", [(16, 1, 4), (2, 2, 1), (8, 2, 8), (4, 1, 2)])
def test_head_layouts(msa, hq, hkv, hidx):
    cfg = wl.GQAConfig("heads", 1, (700,), 0, hq, hkv, hidx, 128, 64, 3, "channel", seed=hq + hkv)
    w = wl.make_gqa(cfg)
    ids = wl.random_topk(5, w.seq_lens, w.cu_q, hidx, 3)
    run_attention(msa, w, ids)


def test_no_sink_and_unit_scales(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=600)
    ids = wl.random_topk(3, w.seq_lens, w.cu_q, 1, 8)
    run_attention(msa, w, ids, sink=False)
    run_attention(msa, w, ids, scales=False)


def test_varlen_prefill_with_prefix(msa):
    cfg = wl.GQAConfig("varlen", 3, (700, 1500, 2100), 0, 16, 2, 4, 128, 128, 8, "channel",
                       pool_factor=1.2, seed=11)
    w = wl.make_gqa(cfg)
    q_lens = np.array([700, 300, 257], np.int32)
    w.cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(w.cu_q[-1])
    w.q, w.idx_q = w.q[:T], w.idx_q[:T]
    ids = wl.random_topk(9, w.seq_lens, w.cu_q, 4, 8)
    run_attention(msa, w, ids)


def test_prefill8k_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["prefill8k"])
    ids = wl.random_topk(1, w.seq_lens, w.cu_q, 4, 16)
    tok = np.sort(np.random.default_rng(0).choice(w.T, size=200, replace=False))
    run_attention(msa, w, ids, tokens=tok)


def test_prefill32k_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["prefill32k"])
    ids = wl.random_topk(2, w.seq_lens, w.cu_q, 4, 64)
    run_attention(msa, w, np.ascontiguousarray(ids), tokens=sample_tokens(w.T, 256, 1))


def test_decode_small_contexts(msa):
    cfg = wl.GQAConfig("dec", 40, (), 1, 16, 2, 4, 128, 128, 8, "channel",
                       len_range=(1, 3000), max_pages=24, pool_factor=1.3, seed=12)
    w = wl.make_gqa(cfg)
    ids = wl.random_topk(4, w.seq_lens, w.cu_q, 4, 8)
    run_attention(msa, w, ids)


@pytest.mark.parametrize("hq,hkv,hidx,topk", [(8, 1, 1, 64), (16, 1, 2, 16), (4, 4, 4, 5)])
def test_decode_head_layouts(msa, hq, hkv, hidx, topk):
    cfg = wl.GQAConfig("dec2", 9, (), 1, hq, hkv, hidx, 128, 64, topk, "normal",
                       len_range=(100, 9000), max_pages=80, pool_factor=1.1, seed=hq * 7 + topk)
    w = wl.make_gqa(cfg)
    ids = wl.random_topk(6, w.seq_lens, w.cu_q, hidx, topk)
    run_attention(msa, w, ids)


def test_decode_config_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["decode"])
    ids = wl.random_topk(3, w.seq_lens, w.cu_q, 4, 64)
    from gpu_helpers import dev_bf16
    k8 = msa.quant_fp8(dev_bf16(w.k_pool), w.scales["k"])
    v8 = msa.quant_fp8(dev_bf16(w.v_pool), w.scales["v"])
    q8 = oq.quantize(w.q, w.scales["q"])
    o, ml, lse = msa.sparse_attn_fwd(dev(q8), k8, v8, dev(w.page_table), dev(w.seq_lens),
                                     dev(w.cu_q), dev(ids), dev(w.sink), w.sm_scale, w.scales["q"],
                                     w.scales["k"], w.scales["v"], 1)
    msa.check_errors()
    seqs = sample_extremes(w.seq_lens, 32, 5)
    pages = np.unique(w.page_table[seqs][w.page_table[seqs] >= 0])
    k_ref = np.zeros((w.num_pages,) + w.k_pool.shape[1:], np.uint8)
    v_ref = np.zeros_like(k_ref)
    k_ref[pages] = oq.quantize(w.k_pool[pages], w.scales["k"])
    v_ref[pages] = oq.quantize(w.v_pool[pages], w.scales["v"])
    assert np.array_equal(k_ref[pages], k8.cpu().numpy()[pages])
    ref = oa.sparse_attention(q8, k_ref, v_ref, w.page_table, w.seq_lens, w.cu_q, ids, w.sink,
                              w.sm_scale, w.scales["q"], w.scales["k"], w.scales["v"], tokens=seqs)
    got = (o.float().cpu().numpy()[seqs].astype(np.float64), ml.cpu().numpy()[seqs],
           lse.cpu().numpy()[seqs])
    _check(got, ref)


def _poison_tails(w, k8, v8):
    """Copies of the K/V pools whose rows past each sequence's length, in its
    last page, are e4m3 NaN (0x7F): positions >= seq_len are not part of the
    sequence, so the result must not depend on them."""
    kp, vp = k8.copy(), v8.copy()
    for b in range(w.cfg.B):
        L = int(w.seq_lens[b])
        if L % 128:
            page = w.page_table[b, (L - 1) // 128]
            kp[page, :, L % 128:, :] = 0x7F
            vp[page, :, L % 128:, :] = 0x7F
    return kp, vp


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_nan_past_seq_len_is_ignored(msa, kind):
    if kind == "decode":
        cfg = wl.GQAConfig("decnan", 12, (), 1, 16, 2, 4, 128, 128, 8, "channel",
                           len_range=(1, 2000), max_pages=16, pool_factor=1.2, seed=31)
    else:
        cfg = wl.GQAConfig("prenan", 3, (200, 77, 301), 0, 8, 2, 2, 128, 64, 4, "normal",
                           max_pages=8, pool_factor=1.0, seed=32)
    w = wl.make_gqa(cfg)
    assert np.any(w.seq_lens % 128)
    ids = wl.random_topk(8, w.seq_lens, w.cu_q, w.cfg.Hidx, w.cfg.topk)
    q8, k8, v8 = _codes(w)
    kp, vp = _poison_tails(w, k8, v8)
    o, ml, lse = msa.sparse_attn_fwd(dev(q8), dev(kp), dev(vp), dev(w.page_table), dev(w.seq_lens),
                                     dev(w.cu_q), dev(ids), dev(w.sink), w.sm_scale, w.scales["q"],
                                     w.scales["k"], w.scales["v"], w.max_q_len)
    msa.check_errors()
    got = (o.float().cpu().numpy().astype(np.float64), ml.cpu().numpy(), lse.cpu().numpy())
    assert np.all(np.isfinite(got[0]))
    ref = oa.sparse_attention(q8, k8, v8, w.page_table, w.seq_lens, w.cu_q, ids, w.sink, w.sm_scale,
                              w.scales["q"], w.scales["k"], w.scales["v"])
    _check(got, ref)
