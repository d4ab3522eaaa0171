"""Pins of the no-tie input rule (oracle/no_tie.py): the accumulation bound
by hand-worked values and against fp32 sums in several orders, the keys a
row's bound runs over by brute force, and the redraw's contract (planted
ties are redrawn, other rows untouched, deterministic, never above the first
draw's amax)."""

import numpy as np
import pytest

from fp8_block_sparse_gb300 import workloads as wl
import oracle.no_tie as nt
from oracle import e4m3, quant as oq

ONE, TWO, HALF = 0x38, 0x40, 0x30          # e4m3 codes of 1.0, 2.0, 0.5


def test_codes_used_here():
    assert list(e4m3.decode(np.array([ONE, TWO, HALF], np.uint8))) == [1.0, 2.0, 0.5]


def test_bound_hand_worked():
    # one head of 64 ones against two keys (64 twos, 64 halves): the larger
    # key sum is 128, so the bound is 2 * 64 * 2**-23 * 128 = 2**-9
    q = np.full((1, 64), ONE, np.uint8)
    k = np.stack([np.full(64, TWO, np.uint8), np.full(64, HALF, np.uint8)])
    assert nt.accumulation_bound(q, k)[0] == 2.0 ** -9
    # negative codes count by magnitude; D = 128 doubles the factor
    q2 = np.full((2, 128), ONE | 0x80, np.uint8)
    q2[1] = HALF
    b = nt.accumulation_bound(q2, np.full((1, 128), TWO, np.uint8))
    assert b[0] == 2.0 * 128 * 2.0 ** -23 * 256 and b[1] == 2.0 * 128 * 2.0 ** -23 * 128
    assert nt.accumulation_bound(q, k[:0]).tolist() == [0.0]


def _fp32_sums(prod: np.ndarray, rng) -> list:
    p = prod.astype(np.float32)
    out = [np.float32(0)] * 4
    acc = np.float32(0)
    for x in p:
        acc = np.float32(acc + x)
    out[0] = acc
    acc = np.float32(0)
    for x in p[::-1]:
        acc = np.float32(acc + x)
    out[1] = acc
    v = p.copy()
    while len(v) > 1:                         # pairwise tree
        v = (v[0::2] + v[1::2]).astype(np.float32)
    out[2] = v[0]
    acc = np.float32(0)
    for x in p[rng.permutation(len(p))]:
        acc = np.float32(acc + x)
    out[3] = acc
    return out


@pytest.mark.parametrize("D", [64, 128])
def test_bound_covers_fp32_accumulation(D):
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, size=(200, D)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F                   # no NaN codes
    q, keys = codes[:1], codes[1:]
    half_bound = nt.accumulation_bound(q, keys)[0] / 2
    qv, kv = e4m3.decode(q[0]), e4m3.decode(keys)
    for row in kv:
        prod = qv * row                                    # exact in fp32 and fp64
        exact = float(prod.sum())
        for s in _fp32_sums(prod, rng):
            assert abs(float(s) - exact) <= half_bound


def test_row_bound_runs_over_every_scored_key():
    w = wl.make_gqa(wl.CONFIGS["prefill8k"], T_override=700)
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    tok = [0, 127, 128, 300, 699]
    got = nt.row_bounds(iq, ik, w.page_table, w.seq_lens, w.cu_q, tok)
    for n, t in enumerate(tok):
        own = t // 128
        for h in range(w.cfg.Hidx):
            best = 0.0
            for j in range(own):                            # brute force over blocks and keys
                page = w.page_table[0, j]
                for key in range(128):
                    s = np.abs(e4m3.decode(ik[page, key])) @ np.abs(e4m3.decode(iq[t, h]))
                    best = max(best, float(s))
            assert got[h, n] == 2.0 * w.cfg.d_idx * 2.0 ** -23 * best


def test_planted_ties_are_redrawn_and_nothing_else():
    # tiny selects 8 blocks, so only tokens whose own block is >= 8 choose
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=1500)
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    bits = w.idx_q.copy()
    planted = [1100, 1300, 1499]
    bits[planted] = 0                          # every score 0: gap 0, bound 0 -> a tie
    early = 500                                # own block < topk: no choice, never a tie
    bits[early] = 0
    out, red = nt.redraw_near_ties(bits, w.scales["idx_q"], ik, w.page_table, w.seq_lens, w.cu_q,
                                   w.cfg.topk, wl.idx_q_redraw(w))
    assert set(planted) <= set(red) and early not in red
    keep = np.setdiff1d(np.arange(w.T), red)
    assert np.array_equal(out[keep], bits[keep])
    codes = oq.quantize(out, w.scales["idx_q"])
    near, gaps, bounds = nt.near_tie_tokens(codes, ik, w.page_table, w.seq_lens, w.cu_q,
                                            w.cfg.topk, range(w.T))
    assert len(near) == 0 and np.all(gaps > bounds)
    again, red2 = nt.redraw_near_ties(bits, w.scales["idx_q"], ik, w.page_table, w.seq_lens,
                                      w.cu_q, w.cfg.topk, wl.idx_q_redraw(w))
    assert red2 == red and np.array_equal(again, out)


def test_redraw_above_first_amax_is_refused():
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=1200)
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    bits = w.idx_q.copy()
    bits[1150] = 0
    base = wl.idx_q_redraw(w)
    big = wl.to_bf16_bits(np.full(bits.shape[1:], 1e4, np.float32))
    seen = []

    def redraw(t, a):
        seen.append(a)
        return big if a == 0 else base(t, a)

    out, red = nt.redraw_near_ties(bits, w.scales["idx_q"], ik, w.page_table, w.seq_lens, w.cu_q,
                                   w.cfg.topk, redraw, tokens=[1150])
    assert red == [1150] and seen[:2] == [0, 1]
    assert np.array_equal(out[1150], base(1150, 1))


def test_redraw_restricted_to_listed_tokens():
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=1500)
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    bits = w.idx_q.copy()
    bits[[1100, 1300]] = 0
    out, red = nt.redraw_near_ties(bits, w.scales["idx_q"], ik, w.page_table, w.seq_lens, w.cu_q,
                                   w.cfg.topk, wl.idx_q_redraw(w), tokens=[1300, 1400])
    assert red == [1300] and np.array_equal(out[1100], bits[1100])


def test_a_redraw_that_ties_again_is_redrawn_again():
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=1200)
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    bits = w.idx_q.copy()
    bits[1150] = 0
    base = wl.idx_q_redraw(w)
    zero = np.zeros(bits.shape[1:], np.uint16)
    out, red = nt.redraw_near_ties(bits, w.scales["idx_q"], ik, w.page_table, w.seq_lens, w.cu_q,
                                   w.cfg.topk, lambda t, a: zero if a == 0 else base(t, a),
                                   tokens=[1150])
    assert red == [1150] and np.array_equal(out[1150], base(1150, 1))
