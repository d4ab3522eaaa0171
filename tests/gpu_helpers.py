"""Shared helpers of the GPU parity tests (host-side marshalling and checks)."""

from __future__ import annotations

import numpy as np
import torch

from oracle import e4m3


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def topk_decision_bound(q_codes: np.ndarray, keys_per_row, D: int) -> np.ndarray:
    """Per-row bound on how far fp32 accumulation can move a comparison of two
    block scores.

    A dot of D exact products accumulated in fp32 in any order, with round-to-
    nearest or truncation, is off by at most D * 2**-23 * sum_d |q_d k_d|; two
    scores are compared, hence the factor 2. The bound takes the largest
    sum_d |q_d k_d| over the keys the row actually scores.
    q_codes: [n, D] codes of the rows; keys_per_row(n) -> [m, D] key codes.
    """
    out = np.empty(len(q_codes))
    for n, q in enumerate(q_codes):
        k = keys_per_row(n)
        if len(k) == 0:
            out[n] = 0.0
            continue
        s = np.abs(e4m3.decode(k)) @ np.abs(e4m3.decode(q))
        out[n] = 2.0 * D * 2.0 ** -23 * s.max()
    return out


def check_topk_rows(got: np.ndarray, ref: np.ndarray, gaps: np.ndarray, bound: np.ndarray,
                    own: np.ndarray, topk: int, exact_scores=None):
    """Exact match on rows whose decision gap exceeds the bound. A near-tie row
    must still be a valid ascending top-k layout, and (when exact_scores(i, n)
    is given) every block it selected must score within the bound of every
    block it left out. Returns the number of near-tie rows."""
    clear = gaps > bound
    bad = np.nonzero(clear & np.any(got != ref, axis=-1))
    assert bad[0].size == 0, f"{bad[0].size} clear rows differ, first at {tuple(x[0] for x in bad)}"
    owns = np.broadcast_to(own, gaps.shape)
    for i, n in zip(*np.nonzero(~clear)):
        r, o = got[i, n], int(owns[i, n])
        valid = r[r >= 0]
        assert len(valid) == min(topk, o + 1) and valid[-1] == o and np.all(np.diff(valid) > 0)
        assert np.all(r[len(valid):] == -1)
        if exact_scores is not None and o + 1 > topk:
            sc = exact_scores(i, n)
            chosen = np.zeros(o, bool)
            chosen[valid[:-1]] = True
            assert sc[chosen].min() >= sc[~chosen].max() - bound[i, n], (i, n)
    return int((~clear).sum())
