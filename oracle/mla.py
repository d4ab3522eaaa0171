"""Step a6: sparse MLA-style prefill (MQA over per-query token indices).

TEST INFRASTRUCTURE ONLY (see the package docstring).

sglang PR 25751 page, key source excerpt of ``sparse_mla_q8kv8_prefill_fwd``:

* inputs q [s_q, h_q, d_qk], kv [s_kv, d_qk] (one latent head shared by all
  query heads), indices [s_q, topk] of kv rows, sm_scale, per-tensor q_scale
  and kv_scale, d_v, and optional attn_sink [h_q] and topk_length [s_q];
* V is the first d_v = 512 columns of the same kv rows (the wrapper rejects
  any other d_v);
* outputs out bf16 [s_q, h_q, d_v] and fp32 max_logits and lse [s_q, h_q].

The scale rules are those of the GQA path (sglang PR 30971 page, step 3):
q_scale multiplies the dot and the sink, kv_scale multiplies the dot (as the
k scale) and the output (as the v scale).

Readings where the pages are silent: the first
topk_length[t] entries of a query's index row are its keys (all topk entries
when topk_length is absent); entries that are negative are skipped; max_logit
and lse follow the GQA definitions (sink excluded from max_logit, included in
the natural-log lse).
"""

from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from . import e4m3
from .attention import attend, unit


def sparse_mla(q: np.ndarray, kv: np.ndarray, indices: np.ndarray,
               topk_length: Optional[np.ndarray], sink: Optional[np.ndarray],
               sm_scale: float, q_scale: Optional[float] = None,
               kv_scale: Optional[float] = None, d_v: int = 512,
               tokens: Optional[Iterable[int]] = None):
    """Sparse MLA for the listed query tokens (all by default).

    q: [T, H, d_qk] codes; kv: [S_kv, d_qk] codes; indices: [T, topk] int32.
    Returns (O [n, H, d_v], max_logit [n, H], lse [n, H]) in float64.
    """
    T, h, _ = q.shape
    tok = np.arange(T) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    c = float(sm_scale) * unit(q_scale)
    kvs = unit(kv_scale)
    out = np.zeros((len(tok), h, d_v))
    max_logit = np.zeros((len(tok), h))
    lse = np.zeros((len(tok), h))
    for n, t in enumerate(tok):
        row = indices[t]
        if topk_length is not None:
            row = row[: int(topk_length[t])]
        row = row[row >= 0].astype(np.int64)
        kk = e4m3.decode(kv[row])                   # [n, d_qk]
        vv = e4m3.decode(kv[row, :d_v])             # [n, d_v]
        logits = (c * kvs) * (e4m3.decode(q[t]) @ kk.T)   # [H, n]
        for hh in range(h):
            sigma = None if sink is None else c * float(sink[hh])
            o, m, l = attend(logits[hh], vv, sigma)
            out[n, hh] = kvs * o
            max_logit[n, hh] = m
            lse[n, hh] = l
    return out, max_logit, lse
