"""Steps a2+a3: indexer block scores and the strictly ascending block top-k.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, and where the pages say so:

* vLLM PR 45892 page, implementation step 1 and the ``indexer_msa.py``
  excerpt: prefill scores idx_q against the index-K cache with one score per
  128-token page ("fmha tile id is the M3 block id"; the score output is
  called ``max_score``), then picks the top-k blocks into
  ``topk_indices_buffer``. Reading: a block's score is the MAXIMUM of the
  query-key dot products over the keys of that block.
* Same page, step 3: the index-K cache has no head axis ([num_pages, 128,
  128]); every index head scores against the same keys.
* Same page, step 4: the buffer has shape [num_index_heads, tokens,
  topk_blocks].
* sglang PR 30971 page, implementation step 2 and review item 2: block ids are
  written strictly ascending; when a query has no more causal blocks than
  topk, the output is all of them followed by -1 padding.

Readings where the pages are silent:

* the query's own block (the one holding its position) is always selected and
  takes one of the ``topk`` slots; the other ``topk - 1`` are the highest
  scoring earlier blocks;
* equal scores are ordered by the lower block id;
* scores are ranked on the unscaled dot of the decoded codes: the per-tensor
  scales and the softmax scale are positive and common to a row, so they
  cannot change the order.

The dots of decoded e4m3 codes are exact in float64 (products are multiples of
2**-18 below 2**17.6; a 128-term sum needs at most 43 significant bits), so
these scores are the exact real numbers, independent of summation order.
"""

from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np

from . import e4m3

PAGE = 128


def query_positions(seq_lens: np.ndarray, cu_q: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Sequence id and absolute position of every query token.

    Sequence b owns query tokens cu_q[b] .. cu_q[b+1]-1, which are its last
    q_len = cu_q[b+1]-cu_q[b] tokens: positions seq_lens[b]-q_len .. seq_lens[b]-1
    (prefill without prefix: q_len == seq_len; decode: q_len == 1).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    cu_q = np.asarray(cu_q, dtype=np.int64)
    T = int(cu_q[-1])
    seq = np.empty(T, dtype=np.int64)
    pos = np.empty(T, dtype=np.int64)
    for b in range(len(seq_lens)):
        lo, hi = int(cu_q[b]), int(cu_q[b + 1])
        seq[lo:hi] = b
        pos[lo:hi] = seq_lens[b] - (hi - lo) + np.arange(hi - lo)
    return seq, pos


def block_scores(q_codes: np.ndarray, idx_k_pool: np.ndarray, pages: np.ndarray) -> np.ndarray:
    """Exact score of each listed block for each query vector.

    q_codes: [H, D] e4m3 codes of one token's index queries.
    idx_k_pool: [num_pages, 128, D] e4m3 index-K cache.
    pages: physical page of each logical block to score.
    Returns [H, len(pages)] float64: max over the block's 128 keys of q . k.
    """
    q = e4m3.decode(q_codes)                           # [H, D]
    k = e4m3.decode(idx_k_pool[np.asarray(pages, dtype=np.int64)])   # [n, 128, D]
    dots = np.einsum("hd,nkd->hnk", q, k)              # exact in float64
    return dots.max(axis=2)


def select_blocks(scores: np.ndarray, own_block: int, topk: int) -> Tuple[np.ndarray, float]:
    """Ascending top-k block ids for one query row, plus its decision gap.

    scores: exact scores of blocks 0 .. own_block-1.
    Returns (ids[topk] int32, gap) where gap is the score difference between
    the lowest selected and the highest unselected candidate (inf when there
    is no choice to make).
    """
    ids = np.full(topk, -1, dtype=np.int32)
    if own_block + 1 <= topk:
        ids[: own_block + 1] = np.arange(own_block + 1)
        return ids, float("inf")
    n_pick = topk - 1
    cand = np.arange(own_block)
    # descending score, then ascending id
    order = np.lexsort((cand, -scores))
    picked = np.sort(order[:n_pick])
    ids[:n_pick] = picked
    ids[n_pick] = own_block
    gap = float(scores[order[n_pick - 1]] - scores[order[n_pick]]) if n_pick > 0 else float("inf")
    return ids, gap


def index_topk(idx_q: np.ndarray, idx_k_pool: np.ndarray, page_table: np.ndarray,
               seq_lens: np.ndarray, cu_q: np.ndarray, topk: int,
               tokens: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """topk_indices for the listed query tokens (all by default).

    idx_q: [T, Hidx, D] codes; idx_k_pool: [num_pages, 128, D] codes;
    page_table: [B, max_pages] physical page of each logical block.
    Returns (ids [Hidx, n, topk] int32, gaps [Hidx, n] float64).
    """
    seq, pos = query_positions(seq_lens, cu_q)
    tok = np.arange(idx_q.shape[0]) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    hidx = idx_q.shape[1]
    ids = np.empty((hidx, len(tok), topk), dtype=np.int32)
    gaps = np.empty((hidx, len(tok)), dtype=np.float64)
    for n, t in enumerate(tok):
        b, p = int(seq[t]), int(pos[t])
        own = p // PAGE
        if own + 1 <= topk:
            sc = np.zeros((hidx, own))
        else:
            sc = block_scores(idx_q[t], idx_k_pool, page_table[b, :own])
        for i in range(hidx):
            ids[i, n], gaps[i, n] = select_blocks(sc[i], own, topk)
    return ids, gaps
