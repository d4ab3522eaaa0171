"""GPU parity of msa_index_topk (steps a2+a3) against the oracle.

Block ids must match bit for bit on every row whose exact decision gap (the
score difference between the last selected and the first unselected block)
exceeds the fp32 accumulation bound; rows inside the bound are near-ties where
either choice is a correct top-k, and are checked for a valid layout and
counted.
"""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, index_topk as oi
from gpu_helpers import dev, dev_bf16, topk_decision_bound, check_topk_rows

pytestmark = pytest.mark.gpu


def _run(msa, w, topk=None, tokens=None, iq=None, ik=None):
    topk = w.cfg.topk if topk is None else topk
    iq = oq.quantize(w.idx_q, w.scales["idx_q"]) if iq is None else iq
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"]) if ik is None else ik
    ids = msa.index_topk(dev(iq), dev(ik), dev(w.page_table), dev(w.seq_lens), dev(w.cu_q), topk,
                         w.max_q_len)
    msa.check_errors()
    got = ids.cpu().numpy()
    tok = np.arange(w.T) if tokens is None else np.asarray(tokens)
    ref, gaps = oi.index_topk(iq, ik, w.page_table, w.seq_lens, w.cu_q, topk, tokens=tok)
    seq, pos = oi.query_positions(w.seq_lens, w.cu_q)
    bound = _bounds(iq, ik, w.page_table, seq, pos, tok)
    def exact(i, n):
        t = tok[n]
        return oi.block_scores(iq[t], ik, w.page_table[seq[t], :pos[t] // 128])[i]
    near = check_topk_rows(got[:, tok], ref, gaps, bound, pos[tok] // 128, topk, exact)
    assert near <= max(2, 0.05 * gaps.size), near
    return got, near


def _bounds(iq, ik, page_table, seq, pos, tok):
    """[Hidx, n] accumulation bounds over the keys of each row's scored blocks."""
    hidx, D = iq.shape[1], iq.shape[2]
    out = np.empty((hidx, len(tok)))
    for n, t in enumerate(tok):
        own = int(pos[t]) // 128
        keys = ik[page_table[seq[t], :own]].reshape(-1, D) if own else ik[:0, 0]
        out[:, n] = topk_decision_bound(iq[t], lambda _: keys, D)
    return out


def test_tiny_all_rows(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"])
    _run(msa, w)


@pytest.mark.parametrize("T", [1000, 129, 1])
def test_ragged_lengths(msa, T):
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=T)
    _run(msa, w)


@pytest.mark.parametrize("topk", [1, 2, 3, 33])
def test_topk_values(msa, topk):
    w = wl.make_gqa(wl.CONFIGS["prefill8k"], T_override=2500)
    _run(msa, w, topk=topk)


def test_prefill8k_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["prefill8k"])
    tok = np.random.default_rng(0).choice(w.T, size=600, replace=False)
    _run(msa, w, tokens=np.sort(tok))


def test_prefill32k_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["prefill32k"])
    tok = np.random.default_rng(1).choice(w.T, size=160, replace=False)
    tok = np.concatenate([np.sort(tok), [w.T - 1]])
    _run(msa, w, tokens=tok)


def test_varlen_prefill_with_prefix(msa):
    # three sequences, the last two continue an existing prefix (q_len < seq_len)
    cfg = wl.GQAConfig("varlen", 3, (700, 1500, 2100), 0, 16, 2, 4, 128, 128, 8, "channel",
                       pool_factor=1.2, seed=11)
    w = wl.make_gqa(cfg)
    q_lens = np.array([700, 300, 257], np.int32)
    w.cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(w.cu_q[-1])
    w.q, w.idx_q = w.q[:T], w.idx_q[:T]
    _run(msa, w)


def test_decode_small_contexts(msa):
    cfg = wl.GQAConfig("dec", 40, (), 1, 16, 2, 4, 128, 128, 8, "channel",
                       len_range=(1, 3000), max_pages=24, pool_factor=1.3, seed=12)
    _run(msa, wl.make_gqa(cfg))


def test_decode_config_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["decode"])
    ik = msa.quant_fp8(dev_bf16(w.idx_k_pool), w.scales["idx_k"]).cpu().numpy()   # full pool
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    ids = msa.index_topk(dev(iq), dev(ik), dev(w.page_table), dev(w.seq_lens), dev(w.cu_q),
                         w.cfg.topk, 1)
    msa.check_errors()
    got = ids.cpu().numpy()
    seqs = np.random.default_rng(2).choice(w.cfg.B, size=12, replace=False)
    # the oracle reads only the sampled sequences' pages, quantised by its own codec
    pages = np.unique(w.page_table[seqs][w.page_table[seqs] >= 0])
    ik_ref = np.zeros_like(ik)
    ik_ref[pages] = oq.quantize(w.idx_k_pool[pages], w.scales["idx_k"])
    assert np.array_equal(ik_ref[pages], ik[pages])
    ref, gaps = oi.index_topk(iq, ik_ref, w.page_table, w.seq_lens, w.cu_q, w.cfg.topk, tokens=seqs)
    seq, pos = oi.query_positions(w.seq_lens, w.cu_q)
    bound = _bounds(iq, ik_ref, w.page_table, seq, pos, seqs)
    own = (w.seq_lens[seqs] - 1) // 128
    check_topk_rows(got[:, seqs], ref, gaps, bound, own, w.cfg.topk)


def test_bad_page_id_is_reported_not_trapped(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=600)
    w.page_table = w.page_table.copy()
    w.page_table[0, 1] = 10 ** 6
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    msa.index_topk(dev(iq), dev(ik), dev(w.page_table), dev(w.seq_lens), dev(w.cu_q), 8, w.max_q_len)
    with pytest.raises(msa.MsaError) as e:
        msa.check_errors()
    assert e.value.status == 6
    msa.check_errors()      # the word was cleared
