"""Shared helpers of the GPU parity tests (host-side marshalling and checks)."""

from __future__ import annotations

import numpy as np
import torch

from oracle import e4m3


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def sample_tokens(T: int, n: int, seed: int) -> np.ndarray:
    """n sorted distinct query tokens of a one-sequence prefill: the first and
    last token, the last and first token on each side of a few block
    boundaries, the rest drawn uniformly."""
    fixed = [0, T - 1]
    for b in (1, 2, T // 256, T // 128 - 1):
        if 0 < b < T // 128:
            fixed += [128 * b - 1, 128 * b]
    fixed = np.unique(np.array(fixed))
    rest = np.setdiff1d(np.arange(T), fixed)
    pick = np.random.default_rng(seed).choice(rest, size=n - len(fixed), replace=False)
    return np.sort(np.concatenate([fixed, pick]))


def sample_extremes(values: np.ndarray, n: int, seed: int) -> np.ndarray:
    """n sorted distinct indices of `values` including its smallest and
    largest entry (e.g. the shortest and longest context of a batch)."""
    fixed = np.unique([int(np.argmin(values)), int(np.argmax(values))])
    rest = np.setdiff1d(np.arange(len(values)), fixed)
    pick = np.random.default_rng(seed).choice(rest, size=n - len(fixed), replace=False)
    return np.sort(np.concatenate([fixed, pick]))


def check_topk_rows(got: np.ndarray, ref: np.ndarray, gaps: np.ndarray, bound: np.ndarray,
                    own: np.ndarray, topk: int, exact_scores=None):
    """Exact match on rows whose decision gap exceeds the bound. A near-tie row
    (the callers redraw inputs so that none remain, and assert so) must still
    be a valid ascending top-k layout, and (when exact_scores(i, n) is given)
    every block it selected must score within the bound of every block it
    left out. Returns the number of near-tie rows."""
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
