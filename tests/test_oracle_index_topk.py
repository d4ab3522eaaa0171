"""Pins for the oracle's block scores and ascending top-k (steps a2+a3)."""

import itertools

import numpy as np
import pytest

from oracle import e4m3, index_topk as ot


def _int_value_512(codes):
    """Exact integer value*512 of e4m3 codes, from the bit fields (independent decode)."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c >> 7, -1, 1)
    E = (c >> 3) & 0xF
    M = c & 7
    mag = np.where(E == 0, M, (8 + M) << np.maximum(E - 1, 0))
    return s * mag


def _finite_codes(g, shape, max_code=0x70):
    c = g.integers(0, max_code, size=shape).astype(np.uint8)
    sign = g.integers(0, 2, size=shape).astype(np.uint8) << 7
    return c | sign


def test_block_scores_equal_exact_integer_arithmetic():
    g = np.random.default_rng(1)
    D, n_pages = 128, 9
    q = _finite_codes(g, (3, D), 0x7F)            # full finite range incl. 448
    pool = _finite_codes(g, (n_pages, 128, D), 0x7F)
    pages = g.permutation(n_pages)[:6]
    got = ot.block_scores(q, pool, pages)
    qi = _int_value_512(q)
    ki = _int_value_512(pool[pages])              # [6, 128, D]
    dots = np.einsum("hd,nkd->hnk", qi, ki)       # exact int64
    ref = dots.max(axis=2).astype(np.float64) / 2.0 ** 18
    np.testing.assert_array_equal(got, ref)


def test_planted_block_maxima_decide_the_selection():
    # one index head, q = e_0 (code 0x38 = 1.0): a key's score is its channel 0
    g = np.random.default_rng(2)
    D, own, topk = 64, 9, 4
    q = np.zeros((1, 1, D), np.uint8)
    q[0, 0, 0] = 0x38
    pool = _finite_codes(g, (own + 1, 128, D), 0x30)     # other channels: any finite
    pool[:, :, 0] = 0x20                                   # low channel-0 everywhere
    hot = {2: 0x60, 5: 0x58, 7: 0x50}                       # 2 > 5 > 7 by value
    for blk, code in hot.items():
        pool[blk, g.integers(0, 128), 0] = code            # one planted max per hot block
    pool[4, 17, 0] = 0x48                                   # runner-up, must be dropped
    page_table = np.arange(own + 1, dtype=np.int32)[None, :]
    seq_lens = np.array([own * 128 + 5], np.int32)
    cu_q = np.array([0, 1], np.int32)
    ids, gaps = ot.index_topk(q, pool, page_table, seq_lens, cu_q, topk)
    np.testing.assert_array_equal(ids[0, 0], [2, 5, 7, own])
    assert gaps[0, 0] == e4m3.decode(np.uint8(0x50)) - e4m3.decode(np.uint8(0x48))


def _brute_force(scores, k_minus_1):
    n = len(scores)
    winners = []
    for sub in itertools.combinations(range(n), k_minus_1):
        rest = [j for j in range(n) if j not in sub]
        if all((scores[a], -a) > (scores[b], -b) for a in sub for b in rest):
            winners.append(sub)
    assert len(winners) == 1
    return list(winners[0])


@pytest.mark.parametrize("seed", range(40))
def test_selection_matches_brute_force_over_all_subsets(seed):
    g = np.random.default_rng(100 + seed)
    own = int(g.integers(1, 10))                     # candidates 0..own-1
    topk = int(g.integers(2, own + 2))               # forces a choice when topk < own + 1
    scores = g.integers(-3, 4, size=own).astype(np.float64)   # many ties
    ids, gap = ot.select_blocks(scores, own, topk)
    if own + 1 <= topk:
        expect = list(range(own + 1)) + [-1] * (topk - own - 1)
        assert gap == float("inf")
    else:
        expect = _brute_force(scores, topk - 1) + [own]
    np.testing.assert_array_equal(ids, expect)


@pytest.mark.parametrize("topk", [16, 32, 33, 48, 64])
def test_selection_matches_cpu_sort_reference(topk):
    # the topk matrix the sglang PR 30971 page checks its warp sort against
    g = np.random.default_rng(topk)
    for own in (topk - 1, topk, topk + 1, 3 * topk, 255):
        scores = g.standard_normal(own)
        ids, _ = ot.select_blocks(scores, own, topk)
        if own + 1 <= topk:
            ref = list(range(own + 1)) + [-1] * (topk - own - 1)
        else:
            ref = sorted(sorted(range(own), key=lambda j: (-scores[j], j))[: topk - 1]) + [own]
        np.testing.assert_array_equal(ids, ref)


def _random_case(seed, T, hidx, d, topk, pool_extra=3):
    g = np.random.default_rng(seed)
    nblk = (T + 127) // 128
    n_pages = nblk + pool_extra
    pool = _finite_codes(g, (n_pages, 128, d), 0x58)
    q = _finite_codes(g, (T, hidx, d), 0x58)
    pt = g.permutation(n_pages)[:nblk].astype(np.int32)[None, :]
    return q, pool, pt, np.array([T], np.int32), np.array([0, T], np.int32)


def test_output_invariants():
    T, topk = 1100, 4
    q, pool, pt, sl, cu = _random_case(5, T, 2, 64, topk)
    ids, _ = ot.index_topk(q, pool, pt, sl, cu, topk)
    for i in range(2):
        for t in range(T):
            row = ids[i, t]
            own = t // 128
            valid = row[row >= 0]
            assert len(valid) == min(topk, own + 1)
            assert np.all(row[len(valid):] == -1)            # -1 only as a suffix
            assert np.all(np.diff(valid) > 0)                # strictly ascending
            assert valid[-1] == own                          # own block forced, largest
            if own + 1 <= topk:
                np.testing.assert_array_equal(valid, np.arange(own + 1))


def test_page_table_indirection():
    T, topk = 700, 3
    q, pool, pt, sl, cu = _random_case(6, T, 1, 128, topk)
    ids_a, _ = ot.index_topk(q, pool, pt, sl, cu, topk)
    # move every page to a new physical slot; the logical result must not change
    perm = np.random.default_rng(0).permutation(pool.shape[0])
    pool_b = np.empty_like(pool)
    pool_b[perm] = pool
    ids_b, _ = ot.index_topk(q, pool_b, perm[pt].astype(np.int32), sl, cu, topk)
    np.testing.assert_array_equal(ids_a, ids_b)


def test_decode_rows_use_their_own_sequence():
    # two sequences with q_len 1 equal two single-sequence calls
    g = np.random.default_rng(11)
    d, topk = 64, 3
    pool = _finite_codes(g, (12, 128, d), 0x58)
    q = _finite_codes(g, (2, 1, d), 0x58)
    pt = np.array([[3, 7, 1, 0, -1, -1], [2, 4, 5, 6, 8, 9]], np.int32)
    sl = np.array([4 * 128 - 3, 6 * 128], np.int32)
    ids, _ = ot.index_topk(q, pool, pt, sl, np.array([0, 1, 2], np.int32), topk)
    for b in range(2):
        one, _ = ot.index_topk(q[b:b + 1], pool, pt[b:b + 1], sl[b:b + 1],
                               np.array([0, 1], np.int32), topk)
        np.testing.assert_array_equal(ids[:, b], one[:, 0])
        assert ids[0, b, -1] == (sl[b] - 1) // 128
