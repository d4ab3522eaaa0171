"""Emulation of the GPU kernels' intended numerics (diagnostic only).

TEST INFRASTRUCTURE ONLY (see the package docstring). This is NOT a
pass/fail reference: parity is always judged against the float64 oracle in
``attention.py``. The emulation replays the precision choices of the
attention kernels' design, so that the error each choice costs against the
float64 result can be predicted on the CPU:

* scores: the dot of the decoded codes accumulated in fp32, times the folded
  scale, in log2 units (``u = fp32(dot) * fp32(c_qk * log2 e)``);
* online softmax over the selected 128-key blocks in ascending order with a
  lazy reference: the reference only moves when a block's maximum exceeds it
  by more than ``limit`` (log2 units); it then moves to that maximum minus
  ``head`` and the running sum and accumulator are rescaled;
* ``p = 2^(u - ref)`` in fp32, the row sum accumulated from the unrounded p;
* P rounded for the PV product: ``"fp32"`` (no rounding), ``"f16"``,
  ``"e4m3"`` (one term) or ``"e4m3x2"`` / ``"e4m3x3"`` (p rounded, then the
  rounded remainder, ...: the terms are summed exactly by the fp32 MMA);
* PV accumulated in fp32; the sink enters the final sum as
  ``2^(sigma log2 e - ref)``; O = v_scale * acc / l rounded to bf16;
  lse = ln 2 * (ref + log2 l); max_logit = ln 2 * max u.

Where the kernels' design fixes it: the prefill kernel keeps P in f16 and
moves the reference to the block maximum (limit 8, head 0); the decode kernel
splits P into two e4m3 terms and moves the reference to 4 below the maximum
(limit 8, head 4); the sparse-MLA kernel walks each query's index
list in 64-entry chunks with f16 P (limit 8, head 0). MUFU's approximation
error and the MMA's exact accumulation order are not modelled (both well
below the roundings above).

The sources of the method are those of ``attention.py``; the pages name fp8
P as the main error source of an fp8 attention and test it at 6e-2..1e-1
(sglang PR 30971 page, risk 6), which is what this module quantifies.
"""

from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from . import e4m3
from .attention import row_keys, unit
from .index_topk import query_positions

LOG2E = 1.4426950408889634
LN2 = 0.6931471805599453

PREFILL = {"p_format": "f16", "limit": 8.0, "head": 0.0}
DECODE = {"p_format": "e4m3x2", "limit": 8.0, "head": 4.0}


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); float64 out."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def round_p(p: np.ndarray, p_format: str) -> np.ndarray:
    """The P operand of the PV product, as float64 values."""
    p = np.asarray(p, dtype=np.float32)
    if p_format == "fp32":
        return p.astype(np.float64)
    if p_format == "f16":
        return p.astype(np.float16).astype(np.float64)
    if p_format.startswith("e4m3"):
        terms = 1 if p_format == "e4m3" else int(p_format[len("e4m3x"):])
        total = np.zeros(p.shape)
        rest = p
        for _ in range(terms):
            t = e4m3.decode(e4m3.encode(rest))
            total += t
            rest = (rest.astype(np.float64) - t).astype(np.float32)   # fp32 remainder
        return total
    raise ValueError(f"unknown P format {p_format!r}")


def emulate_row(q: np.ndarray, keys: np.ndarray, values: np.ndarray, blocks: np.ndarray,
                c_qk_log2: float, sigma_log2: Optional[float], v_scale: float,
                p_format: str, limit: float, head: float, round_out: bool = True):
    """One (token, head) row. keys/values: [n, D] decoded; blocks: [n] block id
    of each key (ascending). Returns (O [D], max_logit, lse)."""
    d = values.shape[1]
    if keys.shape[0] == 0:
        o = np.zeros(d)
        return o, float("-inf"), (float("-inf") if sigma_log2 is None else sigma_log2 * LN2)
    dots = (keys.astype(np.float32) @ q.astype(np.float32)).astype(np.float32)
    u = (dots * np.float32(c_qk_log2)).astype(np.float32)
    ref = None
    acc = np.zeros(d, dtype=np.float32)
    l = np.float32(0.0)
    for b in np.unique(blocks):
        sel = blocks == b
        ub = u[sel]
        mb = float(ub.max())
        if ref is None or mb > ref + limit:
            new_ref = mb - head
            if ref is not None:
                alpha = np.float32(2.0 ** (ref - new_ref))
                acc = (acc * alpha).astype(np.float32)
                l = np.float32(l * alpha)
            ref = new_ref
        p = np.exp2(ub.astype(np.float64) - ref).astype(np.float32)
        l = np.float32(l + np.float32(p.astype(np.float64).sum()))
        acc = (acc + (round_p(p, p_format) @ values[sel])).astype(np.float32)
    if sigma_log2 is not None:
        l = np.float32(l + np.float32(2.0 ** (sigma_log2 - ref)))
    o = (acc / l).astype(np.float32) * np.float32(v_scale)
    o = bf16_round(o) if round_out else o.astype(np.float64)
    return o, float(u.max()) * LN2, (ref + float(np.log2(np.float64(l)))) * LN2


def emulate_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                      page_table: np.ndarray, seq_lens: np.ndarray, cu_q: np.ndarray,
                      topk_idx: np.ndarray, sink: Optional[np.ndarray], sm_scale: float,
                      q_scale: Optional[float] = None, k_scale: Optional[float] = None,
                      v_scale: Optional[float] = None, tokens: Optional[Iterable[int]] = None,
                      p_format: str = "f16", limit: float = 8.0, head: float = 0.0,
                      round_out: bool = True):
    """Emulated sparse attention with the layouts of ``attention.sparse_attention``."""
    T, hq, d = q.shape
    hkv = k_pool.shape[1]
    hidx = topk_idx.shape[0]
    seq, pos = query_positions(seq_lens, cu_q)
    tok = np.arange(T) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    c = float(sm_scale) * unit(q_scale)
    c_qk_log2 = float(np.float32(c * unit(k_scale) * LOG2E))
    vs = unit(v_scale)
    out = np.zeros((len(tok), hq, d))
    max_logit = np.zeros((len(tok), hq))
    lse = np.zeros((len(tok), hq))
    for n, t in enumerate(tok):
        b, p = int(seq[t]), int(pos[t])
        qd = e4m3.decode(q[t])
        for h in range(hq):
            i = h // (hq // hidx)
            g = h // (hq // hkv)
            blk, slot = row_keys(topk_idx[i, t], p)
            pages = page_table[b, blk]
            kk = e4m3.decode(k_pool[pages, g, slot])
            vv = e4m3.decode(v_pool[pages, g, slot])
            sig = None if sink is None else float(np.float32(c * float(sink[h]) * LOG2E))
            out[n, h], max_logit[n, h], lse[n, h] = emulate_row(
                qd[h], kk, vv, blk, c_qk_log2, sig, vs, p_format, limit, head, round_out)
    return out, max_logit, lse


def emulate_mla(q: np.ndarray, kv: np.ndarray, indices: np.ndarray,
                topk_length: Optional[np.ndarray], sink: Optional[np.ndarray], sm_scale: float,
                q_scale: Optional[float] = None, kv_scale: Optional[float] = None, d_v: int = 512,
                tokens: Optional[Iterable[int]] = None, p_format: str = "f16", limit: float = 8.0,
                head: float = 0.0, chunk: int = 64, round_out: bool = True):
    """Emulated sparse MLA with the layouts of ``mla.sparse_mla``: the index
    list is walked in ``chunk``-entry pieces (the blocks of the lazy softmax)."""
    T, h, _ = q.shape
    tok = np.arange(T) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    c = float(sm_scale) * unit(q_scale)
    kvs = unit(kv_scale)
    c_qk_log2 = float(np.float32(c * kvs * LOG2E))
    out = np.zeros((len(tok), h, d_v))
    max_logit = np.zeros((len(tok), h))
    lse = np.zeros((len(tok), h))
    for n, t in enumerate(tok):
        row = indices[t]
        if topk_length is not None:
            row = row[: int(topk_length[t])]
        where = np.nonzero(row >= 0)[0]
        rows = row[where].astype(np.int64)
        kk = e4m3.decode(kv[rows])
        vv = e4m3.decode(kv[rows, :d_v])
        qd = e4m3.decode(q[t])
        for hh in range(h):
            sig = None if sink is None else float(np.float32(c * float(sink[hh]) * LOG2E))
            out[n, hh], max_logit[n, hh], lse[n, hh] = emulate_row(
                qd[hh], kk, vv, where // chunk, c_qk_log2, sig, kvs, p_format, limit, head, round_out)
    return out, max_logit, lse
