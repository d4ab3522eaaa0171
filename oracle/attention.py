"""Steps a4/a5: GQA sparse attention over the selected blocks, with a sink.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, and where the pages say so (sglang PR 30971 page,
implementation step 3 and the executive summary):

* every per-tensor scale is optional; a missing scale is the unit scale;
* q_scale is folded into sm_scale, so it multiplies BOTH the q.k dot and the
  per-head sink logit;
* k_scale multiplies the q.k dot only and never the sink term;
* v_scale multiplies the output;
* fp8 tensors store value/scale, and the kernel multiplies the logits back by
  the scales.

Each query row (token t, q head h) attends over the keys of the blocks its
index head selected (topk_indices, strictly ascending with -1 padding, as in
the vLLM PR 45892 page, step 2: attention reads the buffer the indexer
wrote), restricted to keys at positions <= the query's position.

Readings where the pages are silent:

* q head h reads kv head h // (Hq/Hkv) (standard GQA grouping) and index head
  h // (Hq/Hidx);
* with c = sm_scale*q_scale, l_j = c*k_scale*(q.k_j), sigma = c*sink_h:
      O       = v_scale * sum_j e^{l_j} v_j / (sum_j e^{l_j} + e^{sigma})
      max_logit = max_j l_j                       (sink excluded)
      lse     = ln(sum_j e^{l_j} + e^{sigma})     (natural log, sink included)
  so that O = v_scale * sum_j e^{l_j - lse} v_j holds exactly;
* without a sink the e^{sigma} term is absent;
* a row with no valid key has O = 0, max_logit = -inf, lse = sigma (or -inf).

Arithmetic: decoded codes in float64, exact dots, a two-pass max-subtracted
softmax in float64.
"""

from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np

from . import e4m3
from .index_topk import PAGE, query_positions


def unit(scale: Optional[float]) -> float:
    """A missing scale is the unit scale."""
    return 1.0 if scale is None else float(scale)


def attend(logits: np.ndarray, values: np.ndarray, sigma: Optional[float]) -> Tuple[np.ndarray, float, float]:
    """Softmax-with-sink of one row: returns (sum_j w_j v_j, max_logit, lse).

    logits: [n] float64; values: [n, Dv] float64; sigma: sink logit or None.
    """
    dv = values.shape[1]
    if logits.size == 0:
        return np.zeros(dv), float("-inf"), (float("-inf") if sigma is None else float(sigma))
    m = float(logits.max())
    top = m if sigma is None else max(m, float(sigma))
    w = np.exp(logits - top)
    z = float(w.sum()) + (0.0 if sigma is None else float(np.exp(sigma - top)))
    o = (w @ values) / z
    return o, m, top + float(np.log(z))


def row_keys(topk_row: np.ndarray, pos: int) -> Tuple[np.ndarray, np.ndarray]:
    """Logical (block, slot) of every key a row attends to, in position order."""
    blocks = np.unique(topk_row[topk_row >= 0])
    if blocks.size == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    kpos = (blocks[:, None] * PAGE + np.arange(PAGE)[None, :]).reshape(-1)
    kpos = kpos[kpos <= pos]
    return kpos // PAGE, kpos % PAGE


def sparse_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                     page_table: np.ndarray, seq_lens: np.ndarray, cu_q: np.ndarray,
                     topk_idx: np.ndarray, sink: Optional[np.ndarray], sm_scale: float,
                     q_scale: Optional[float] = None, k_scale: Optional[float] = None,
                     v_scale: Optional[float] = None,
                     tokens: Optional[Iterable[int]] = None):
    """Sparse attention for the listed query tokens (all by default).

    q: [T, Hq, D] codes; k_pool, v_pool: [num_pages, Hkv, 128, D] codes;
    page_table: [B, max_pages]; topk_idx: [Hidx, T, topk] int32.
    Returns (O [n, Hq, D], max_logit [n, Hq], lse [n, Hq]) in float64.
    """
    T, hq, d = q.shape
    hkv = k_pool.shape[1]
    hidx = topk_idx.shape[0]
    seq, pos = query_positions(seq_lens, cu_q)
    tok = np.arange(T) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    c = float(sm_scale) * unit(q_scale)
    c_qk = c * unit(k_scale)
    vs = unit(v_scale)

    out = np.zeros((len(tok), hq, d))
    max_logit = np.zeros((len(tok), hq))
    lse = np.zeros((len(tok), hq))
    for n, t in enumerate(tok):
        b, p = int(seq[t]), int(pos[t])
        qd = e4m3.decode(q[t])                                   # [Hq, D]
        for h in range(hq):
            i = h // (hq // hidx)
            g = h // (hq // hkv)
            blk, slot = row_keys(topk_idx[i, t], p)
            pages = page_table[b, blk]
            kk = e4m3.decode(k_pool[pages, g, slot])              # [n, D]
            vv = e4m3.decode(v_pool[pages, g, slot])
            logits = c_qk * (kk @ qd[h])
            sigma = None if sink is None else c * float(sink[h])
            o, m, l = attend(logits, vv, sigma)
            out[n, h] = vs * o
            max_logit[n, h] = m
            lse[n, h] = l
    return out, max_logit, lse
