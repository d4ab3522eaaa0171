"""GPU parity of msa_sparse_mla_fwd (step a6) against the oracle.

Bar as for the GQA path: O within max-abs 4e-2 and relative Frobenius 1e-2,
lse within 2e-3 absolute, max_logits to 1e-4 relative.
"""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, mla as om
from gpu_helpers import dev, dev_bf16, sample_extremes

pytestmark = pytest.mark.gpu


def _check(got, ref):
    o, ml, lse = got
    o_ref, ml_ref, lse_ref = ref
    err = np.abs(o - o_ref).max()
    rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    assert err <= 4e-2 and rel <= 1e-2, (err, rel)
    assert np.abs(lse - lse_ref).max() <= 2e-3
    fin = np.isfinite(ml_ref)
    assert np.array_equal(fin, np.isfinite(ml))
    np.testing.assert_allclose(ml[fin], ml_ref[fin], rtol=1e-4, atol=1e-5)


def _run(msa, w, tokens=None, use_len=True, sink=True, q8=None):
    q8 = oq.quantize(w.q, w.scales["q"]) if q8 is None else q8
    kv8 = oq.quantize(w.kv, w.scales["kv"])
    tl = w.topk_length if use_len else None
    s = w.sink if sink else None
    o, ml, lse = msa.sparse_mla_fwd(dev(q8), dev(kv8), dev(w.indices), None if tl is None else dev(tl),
                                    None if s is None else dev(s), w.sm_scale, w.scales["q"],
                                    w.scales["kv"])
    msa.check_errors()
    tok = np.arange(w.q.shape[0]) if tokens is None else np.asarray(tokens)
    got = (o.float().cpu().numpy()[tok].astype(np.float64), ml.cpu().numpy()[tok], lse.cpu().numpy()[tok])
    ref = om.sparse_mla(q8, kv8, w.indices, tl, s, w.sm_scale, w.scales["q"], w.scales["kv"], tokens=tok)
    _check(got, ref)


@pytest.mark.parametrize("T,S,topk,lr", [(8, 600, 128, (1, 128)), (5, 3000, 256, (60, 256)),
                                         (3, 200, 64, (64, 64)), (4, 5000, 512, (300, 512))])
def test_small_cases(msa, T, S, topk, lr):
    w = wl.make_mla(wl.CONFIGS["mla"], T_override=T, S_override=S, topk_override=topk, len_range=lr)
    _run(msa, w)


def test_without_topk_length_and_sink(msa):
    w = wl.make_mla(wl.CONFIGS["mla"], T_override=6, S_override=900, topk_override=192, len_range=(192, 192))
    _run(msa, w, use_len=False, sink=False)


def test_negative_entries_inside_length_are_skipped(msa):
    w = wl.make_mla(wl.CONFIGS["mla"], T_override=6, S_override=1000, topk_override=128, len_range=(100, 128))
    w.indices = w.indices.copy()
    w.indices[:, 5:9] = -1
    _run(msa, w)


def test_mla_config_sampled(msa):
    w = wl.make_mla(wl.CONFIGS["mla"])
    q8 = msa.quant_fp8(dev_bf16(w.q), w.scales["q"])
    kv8 = oq.quantize(w.kv, w.scales["kv"])
    o, ml, lse = msa.sparse_mla_fwd(q8, dev(kv8), dev(w.indices), dev(w.topk_length), dev(w.sink),
                                    w.sm_scale, w.scales["q"], w.scales["kv"])
    msa.check_errors()
    tok = sample_extremes(w.topk_length, 64, 0)        # incl. the shortest and longest lists
    q8_ref = np.zeros((w.q.shape[0],) + w.q.shape[1:], np.uint8)
    q8_ref[tok] = oq.quantize(w.q[tok], w.scales["q"])
    assert np.array_equal(q8_ref[tok], q8.cpu().numpy()[tok])
    ref = om.sparse_mla(q8_ref, kv8, w.indices, w.topk_length, w.sink, w.sm_scale, w.scales["q"],
                        w.scales["kv"], tokens=tok)
    got = (o.float().cpu().numpy()[tok].astype(np.float64), ml.cpu().numpy()[tok], lse.cpu().numpy()[tok])
    _check(got, ref)
