"""GPU parity of msa_index_topk (steps a2+a3) against the oracle.

Block ids must match the exact selection bit for bit on every checked row.
Inputs follow the no-tie rule (oracle/no_tie.py): a token whose exact
decision gap (the score difference between its last selected and first
unselected block) is within the fp32 accumulation bound of some row is
redrawn before the run, so every checked row has one correct answer. The
number of redrawn tokens is printed with each case.
"""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, index_topk as oi, no_tie
from gpu_helpers import dev, dev_bf16, check_topk_rows, sample_tokens, sample_extremes

pytestmark = pytest.mark.gpu


def apply_no_tie(w, ik, topk, tokens=None):
    """Redraws the near-tie tokens among `tokens` (all by default) in place;
    returns the redrawn tokens."""
    bits, red = no_tie.redraw_near_ties(w.idx_q, w.scales["idx_q"], ik, w.page_table, w.seq_lens,
                                        w.cu_q, topk, wl.idx_q_redraw(w), tokens=tokens)
    w.idx_q = bits
    return red


def _run(msa, w, topk=None, tokens=None):
    topk = w.cfg.topk if topk is None else topk
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    tok = np.arange(w.T) if tokens is None else np.asarray(tokens)
    red = apply_no_tie(w, ik, topk, tok)
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    ids = msa.index_topk(dev(iq), dev(ik), dev(w.page_table), dev(w.seq_lens), dev(w.cu_q), topk,
                         w.max_q_len)
    msa.check_errors()
    got = ids.cpu().numpy()
    ref, gaps = oi.index_topk(iq, ik, w.page_table, w.seq_lens, w.cu_q, topk, tokens=tok)
    bound = no_tie.row_bounds(iq, ik, w.page_table, w.seq_lens, w.cu_q, tok)
    _, pos = oi.query_positions(w.seq_lens, w.cu_q)
    near = check_topk_rows(got[:, tok], ref, gaps, bound, pos[tok] // 128, topk)
    assert near == 0, near
    print(f"{w.cfg.name}: {gaps.size} rows exact, {len(red)} of {len(tok)} tokens redrawn")
    return got


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
    _run(msa, w, tokens=sample_tokens(w.T, 600, 0))


def test_prefill32k_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["prefill32k"])
    _run(msa, w, tokens=sample_tokens(w.T, 256, 1))


@pytest.mark.parametrize("Hidx,max_pages", [(4, 0), (4, 20), (8, 24), (2, 32), (16, 24), (1, 28)])
def test_varlen_prefill_with_prefix(msa, Hidx, max_pages):
    # three sequences, the last two continue an existing prefix (q_len < seq_len);
    # with a page-table width that is a multiple of 4 the full query tiles write
    # their scores by TMA and the ragged ones (each sequence's last) by threads,
    # next to the rows of the following sequence's tokens
    cfg = wl.GQAConfig("varlen", 3, (700, 1500, 2100), 0, 16, 2, Hidx, 128, 128, 8, "channel",
                       max_pages=max_pages, pool_factor=1.2, seed=11)
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


@pytest.mark.parametrize("Hidx,d_idx", [(1, 128), (2, 64), (16, 128)])
def test_decode_index_head_counts(msa, Hidx, d_idx):
    # the decode scorer puts a token's Hidx query rows in the N = 16 columns
    # of one MMA: one column, two, and all sixteen; d_idx 64 takes the 64-byte
    # swizzle
    cfg = wl.GQAConfig("dech", 24, (), 1, 16, 1, Hidx, 128, d_idx, 8, "channel",
                       len_range=(1000, 5000), max_pages=40, pool_factor=1.3, seed=30 + Hidx)
    _run(msa, wl.make_gqa(cfg))


def test_decode_config_sampled(msa):
    w = wl.make_gqa(wl.CONFIGS["decode"])
    ik = msa.quant_fp8(dev_bf16(w.idx_k_pool), w.scales["idx_k"]).cpu().numpy()   # full pool
    seqs = sample_extremes(w.seq_lens, 32, 2)
    # the oracle reads only the sampled sequences' pages, quantised by its own codec
    pages = np.unique(w.page_table[seqs][w.page_table[seqs] >= 0])
    ik_ref = np.zeros_like(ik)
    ik_ref[pages] = oq.quantize(w.idx_k_pool[pages], w.scales["idx_k"])
    assert np.array_equal(ik_ref[pages], ik[pages])
    red = apply_no_tie(w, ik_ref, w.cfg.topk, seqs)
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    ids = msa.index_topk(dev(iq), dev(ik), dev(w.page_table), dev(w.seq_lens), dev(w.cu_q),
                         w.cfg.topk, 1)
    msa.check_errors()
    got = ids.cpu().numpy()
    ref, gaps = oi.index_topk(iq, ik_ref, w.page_table, w.seq_lens, w.cu_q, w.cfg.topk, tokens=seqs)
    bound = no_tie.row_bounds(iq, ik_ref, w.page_table, w.seq_lens, w.cu_q, seqs)
    own = (w.seq_lens[seqs] - 1) // 128
    assert check_topk_rows(got[:, seqs], ref, gaps, bound, own, w.cfg.topk) == 0
    print(f"decode: {gaps.size} rows exact, {len(red)} of {len(seqs)} sequences redrawn")


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_exact_ties_go_to_the_lower_block_id(msa, kind):
    """Logical blocks that share a physical index-K page score exactly alike
    on both sides (the same fp32 MMA of the same operands on the GPU, the same
    exact dot in the oracle), so the selection's tie rule decides: equal
    scores go to the lower block id (oracle/index_topk.py, reading: ties by
    the lower id). Every sequence's blocks cycle through three pages; rows
    whose boundary falls inside a group of equal scores take the tie pass,
    the others the exact-threshold path. The three pages' exact scores are
    checked to lie further apart than the fp32 bound of each row, so every
    row has exactly one correct answer."""
    if kind == "prefill":
        w = wl.make_gqa(wl.CONFIGS["tiny"])
    else:
        cfg = wl.GQAConfig("dec", 24, (), 1, 16, 2, 4, 128, 128, 8, "channel",
                           len_range=(1200, 3000), max_pages=24, pool_factor=1.3, seed=21)
        w = wl.make_gqa(cfg)
    pt = w.page_table.copy()
    cols = np.broadcast_to(np.arange(pt.shape[1], dtype=np.int32), pt.shape)
    pt[pt >= 0] = cols[pt >= 0] % 3
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    topk = w.cfg.topk
    ids = msa.index_topk(dev(iq), dev(ik), dev(pt), dev(w.seq_lens), dev(w.cu_q), topk,
                         w.max_q_len)
    msa.check_errors()
    ref, _ = oi.index_topk(iq, ik, pt, w.seq_lens, w.cu_q, topk)
    _, pos = oi.query_positions(w.seq_lens, w.cu_q)
    chooses = np.nonzero(pos // 128 + 1 > topk)[0]             # rows with a choice to make
    assert chooses.size > 0
    bound = no_tie.row_bounds(iq, ik, pt, w.seq_lens, w.cu_q, chooses)
    ties = 0
    for n, t in enumerate(chooses):
        sc = oi.block_scores(iq[t], ik, np.arange(3))              # [Hidx, 3]
        srt = np.sort(sc, axis=1)
        assert np.all(np.diff(srt, axis=1) > bound[:, n:n + 1]), t
        own = int(pos[t]) // 128
        for i in range(sc.shape[0]):
            per_block = sc[i, np.arange(own) % 3]
            kth = np.sort(per_block)[::-1][topk - 2:topk]       # the (topk-1)-th and next score
            ties += int(kth[0] == kth[1])
    assert ties > 0                                            # the tie pass did run
    assert np.array_equal(ids.cpu().numpy(), ref)
    print(f"{kind}: {chooses.size} tokens with a choice, {ties} rows tied at the boundary")


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


def test_rows_of_a_rejected_sequence_are_minus_one(msa):
    # the middle sequence claims more tokens than its page-table row holds:
    # its rows are -1, the error is reported, the other sequences are exact
    cfg = wl.GQAConfig("varlen", 3, (700, 1500, 2100), 0, 16, 2, 4, 128, 128, 8, "channel",
                       pool_factor=1.2, seed=11)
    w = wl.make_gqa(cfg)
    q_lens = np.array([700, 300, 257], np.int32)
    w.cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(w.cu_q[-1])
    w.q, w.idx_q = w.q[:T], w.idx_q[:T]
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    good = np.r_[np.arange(0, 700), np.arange(1000, T)]
    apply_no_tie(w, ik, cfg.topk, good)
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    bad = w.seq_lens.copy()
    bad[1] = w.page_table.shape[1] * 128 + 1
    ids = msa.index_topk(dev(iq), dev(ik), dev(w.page_table), dev(bad), dev(w.cu_q), cfg.topk,
                         w.max_q_len)
    with pytest.raises(msa.MsaError) as e:
        msa.check_errors()
    assert e.value.status == 6
    got = ids.cpu().numpy()
    assert (got[:, 700:1000] == -1).all()
    ref, gaps = oi.index_topk(iq, ik, w.page_table, w.seq_lens, w.cu_q, cfg.topk, tokens=good)
    bound = no_tie.row_bounds(iq, ik, w.page_table, w.seq_lens, w.cu_q, good)
    _, pos = oi.query_positions(w.seq_lens, w.cu_q)
    assert check_topk_rows(got[:, good], ref, gaps, bound, pos[good] // 128, cfg.topk) == 0
