"""The no-tie input rule of the index step: redraw query rows whose top-k
decision is closer than the GPU's accumulation error.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Why this exists. The top-k block ids must agree bit for bit with the exact
selection. The exact block scores are real numbers (``index_topk``); a GPU
accumulates each query-key dot of D exact e4m3 products in fp32, so a
computed dot can sit off the exact one by a little, and a row whose two
competing blocks score closer than that has two correct answers. The tiny
benchmark configuration asks for inputs drawn so that the top-k has no tied
block scores; the same rule is applied to every row a parity test checks.

Reading (listed in the design notes). A row -- one (index head, query token)
-- is *clear* when its exact decision gap (the score of the lowest selected
block minus that of the highest unselected one, ``index_topk.select_blocks``)
exceeds

    bound = 2 * D * 2**-23 * max_j sum_d |q_d k_jd|,

the largest amount by which fp32 accumulation of D exact products, in any
order, with round-to-nearest or truncation, can move one dot, counted twice
because two scores are compared. (A block score is a maximum of dots, and a
maximum of perturbed values moves by no more than the largest perturbation.)
The maximum runs over every key the row scores.

The rule. A token whose rows are not all clear gets a fresh idx_q row set
(all its index heads) from a seeded re-draw of the same distribution, until
every row clears the bound. Query rows are independent of one another in
the index step (a row's selection depends only on its own idx_q row and on
the shared index-K cache), so redrawing one token changes no other token's
selection. The per-tensor scale stays the one of the first draw: a redraw
whose magnitude would exceed the first draw's amax is refused and drawn
again, so the codes never saturate and the scale keeps meaning amax/448 of
the rows it was computed from.

The re-draw itself is a callable supplied by the caller (the seeded input
generator), so this module holds only the decision, not the random numbers.
"""

from __future__ import annotations

from typing import Callable, Iterable, List, Optional, Tuple

import numpy as np

from . import e4m3
from .index_topk import PAGE, index_topk, query_positions
from .quant import quantize


def accumulation_bound(q_codes: np.ndarray, key_codes: np.ndarray) -> np.ndarray:
    """Per-head comparison bound of one token's rows.

    q_codes: [H, D] e4m3 codes of the token's index queries.
    key_codes: [m, D] e4m3 codes of every key the token's rows score.
    Returns [H] float64: ``2 * D * 2**-23 * max_j sum_d |q_d k_jd|`` (0 when
    there is no key to score).
    """
    q_codes = np.asarray(q_codes)
    D = q_codes.shape[-1]
    if len(key_codes) == 0:
        return np.zeros(q_codes.shape[0])
    s = np.abs(e4m3.decode(key_codes)) @ np.abs(e4m3.decode(q_codes)).T     # [m, H]
    return 2.0 * D * 2.0 ** -23 * s.max(axis=0)


def row_bounds(idx_q_codes: np.ndarray, idx_k_codes: np.ndarray, page_table: np.ndarray,
               seq_lens: np.ndarray, cu_q: np.ndarray, tokens: Iterable[int]) -> np.ndarray:
    """[Hidx, n] bounds of the listed tokens' rows over the keys of the
    blocks each token scores (every block before its own)."""
    seq, pos = query_positions(seq_lens, cu_q)
    tok = np.asarray(list(tokens), dtype=np.int64)
    hidx, D = idx_q_codes.shape[1], idx_q_codes.shape[2]
    out = np.zeros((hidx, len(tok)))
    for n, t in enumerate(tok):
        own = int(pos[t]) // PAGE
        if own == 0:
            continue
        keys = idx_k_codes[page_table[seq[t], :own]].reshape(-1, D)
        out[:, n] = accumulation_bound(idx_q_codes[t], keys)
    return out


def near_tie_tokens(idx_q_codes, idx_k_codes, page_table, seq_lens, cu_q, topk,
                    tokens) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Tokens (of those listed) with at least one row inside its bound.

    Returns (near tokens, gaps [Hidx, n], bounds [Hidx, n]) for the listed
    tokens in their given order.
    """
    tok = np.asarray(list(tokens), dtype=np.int64)
    _, gaps = index_topk(idx_q_codes, idx_k_codes, page_table, seq_lens, cu_q, topk, tokens=tok)
    bounds = row_bounds(idx_q_codes, idx_k_codes, page_table, seq_lens, cu_q, tok)
    near = ~(gaps > bounds)
    return tok[np.any(near, axis=0)], gaps, bounds


def redraw_near_ties(idx_q_bits: np.ndarray, scale: Optional[float], idx_k_codes: np.ndarray,
                     page_table: np.ndarray, seq_lens: np.ndarray, cu_q: np.ndarray, topk: int,
                     redraw: Callable[[int, int], np.ndarray], tokens: Optional[Iterable[int]] = None,
                     max_attempts: int = 64) -> Tuple[np.ndarray, List[int]]:
    """Apply the no-tie rule to the listed tokens (all by default).

    idx_q_bits: [T, Hidx, d] bf16 bit patterns; scale: idx_q's per-tensor
    scale (kept); idx_k_codes: the e4m3 index-K cache the rows score against;
    redraw(t, attempt) -> fresh [Hidx, d] bf16 bits for token t.
    Returns (new bits, sorted list of the tokens that were redrawn). Raises
    when a token is still near a tie after ``max_attempts`` draws.
    """
    bits = np.array(idx_q_bits, copy=True)
    codes = quantize(bits, scale)
    amax_bits = int((bits.astype(np.uint16) & np.uint16(0x7FFF)).max())
    tok = np.arange(bits.shape[0]) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    pending, _, _ = near_tie_tokens(codes, idx_k_codes, page_table, seq_lens, cu_q, topk, tok)
    redrawn = set(int(t) for t in pending)
    next_draw = {}                       # per token: the next re-draw number to use
    rounds = 0
    while len(pending) > 0:
        if rounds >= max_attempts:
            raise RuntimeError(f"{len(pending)} tokens still near a tie after {max_attempts} draws")
        for t in pending:
            t = int(t)
            a = next_draw.get(t, 0)
            while True:
                fresh = np.asarray(redraw(t, a), dtype=np.uint16)
                a += 1
                if int((fresh & np.uint16(0x7FFF)).max()) <= amax_bits:
                    break
                if a > next_draw.get(t, 0) + 1000:
                    raise RuntimeError(f"no redraw of token {t} within the first draw's amax")
            next_draw[t] = a
            bits[t] = fresh
            codes[t] = quantize(fresh, scale)
        rounds += 1
        pending, _, _ = near_tie_tokens(codes, idx_k_codes, page_table, seq_lens, cu_q, topk,
                                        pending)
    return bits, sorted(redrawn)
