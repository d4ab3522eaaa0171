"""Seeded synthetic workloads for the five benchmark configurations.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no quantisation, scoring, selection or attention). Both
the GPU path and the test oracle take their inputs from here.

Every activation is drawn in fp32 from ``numpy.random.Generator(PCG64)``,
rounded to bfloat16 (round-to-nearest-even, via torch's CPU cast) and returned
as uint16 bit patterns. Per-tensor scales follow the recipe of each
configuration (``amax / 448`` unless stated). Each tensor has its own
sub-stream ``SeedSequence([seed, tensor_id])`` so tensors can be drawn in any
order and in chunks without changing their values.

Configurations (names used everywhere in tests and the benchmark):

=========  ==========================================================================
tiny       1 sequence x 2048 tokens, Hq/Hkv/Hidx = 8/1/1, D 128, d_idx 64, topk 8;
           all tensors N(0,1); sink N(0,1)
prefill8k  1 x 8192 tokens, 16/2/4, d_idx 128, topk 16; tensors N(0,1) * c with a
           per-tensor channel vector c log-uniform in [0.5, 4]
prefill32k 1 x 32768 tokens, as prefill8k with topk 64 and k_scale, v_scale drawn
           uniform in [0.25, 4]
decode     128 sequences, q_len 1, context lengths uniform in [4096, 65536],
           16/2/4, topk 64, pages scattered through a pool 1.25x the pages in use
mla        4096 queries at positions 28672..32767 over 32768 latent tokens,
           128 heads, d_qk 576, d_v 512, topk 2048 with topk_length uniform in
           [256, 2048]; indices a sorted sample without replacement of [0, pos]
=========  ==========================================================================
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

PAGE = 128
FP8_MAX = 448.0

# tensor ids for the per-tensor sub-streams
_Q, _K, _V, _IQ, _IK, _SINK, _C, _SCALE, _PT, _LEN, _IDX, _KV = range(12)


@dataclass(frozen=True)
class GQAConfig:
    name: str
    B: int                 # sequences
    seq_lens: tuple        # () means drawn (decode); else explicit per-sequence lengths
    q_len: int             # 0 means q_len == seq_len (prefill without prefix)
    Hq: int
    Hkv: int
    Hidx: int
    D: int
    d_idx: int
    topk: int
    dist: str              # "normal" | "channel" (N(0,1) * per-channel c)
    kv_scale_uniform: bool = False   # k/v scales drawn U[0.25, 4] instead of amax/448
    len_range: tuple = ()            # decode: (lo, hi) inclusive
    max_pages: int = 0               # page-table width (0: just enough)
    pool_factor: float = 1.0
    seed: int = 0


@dataclass(frozen=True)
class MLAConfig:
    name: str
    T: int
    S_kv: int
    H: int
    d_qk: int
    d_v: int
    topk: int
    len_range: tuple
    seed: int = 4


CONFIGS: Dict[str, object] = {
    "tiny": GQAConfig("tiny", 1, (2048,), 0, 8, 1, 1, 128, 64, 8, "normal", seed=0),
    "prefill8k": GQAConfig("prefill8k", 1, (8192,), 0, 16, 2, 4, 128, 128, 16, "channel", seed=1),
    "prefill32k": GQAConfig("prefill32k", 1, (32768,), 0, 16, 2, 4, 128, 128, 64, "channel",
                            kv_scale_uniform=True, seed=2),
    "decode": GQAConfig("decode", 128, (), 1, 16, 2, 4, 128, 128, 64, "channel",
                        len_range=(4096, 65536), max_pages=512, pool_factor=1.25, seed=3),
    "mla": MLAConfig("mla", 4096, 32768, 128, 576, 512, 2048, (256, 2048), seed=4),
}


def _rng(seed: int, tensor: int, extra: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor, extra])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (RNE) and return the uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _channel_vector(seed: int, tensor: int, dim: int) -> np.ndarray:
    g = _rng(seed, _C, tensor)
    return np.exp(g.uniform(np.log(0.5), np.log(4.0), size=dim)).astype(np.float32)


def draw_tensor(seed: int, tensor: int, shape: tuple, dist: str, chunk_rows: int = 1 << 20) -> np.ndarray:
    """bf16 bits of a tensor whose last axis is the channel axis.

    Drawn in row chunks of the flattened [rows, last] view, so large pools do
    not need an fp32 copy of the whole tensor.
    """
    last = shape[-1]
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    out = np.empty((rows, last), dtype=np.uint16)
    g = _rng(seed, tensor)
    c = _channel_vector(seed, tensor, last) if dist == "channel" else None
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = g.standard_normal((r1 - r0, last), dtype=np.float32)
        if c is not None:
            x *= c
        out[r0:r1] = to_bf16_bits(x)
    return out.reshape(shape)


def amax_scale(bits: np.ndarray) -> float:
    """Per-tensor scale amax/448 (fp32) of a bf16 tensor (input recipe)."""
    # the max magnitude of bf16 bit patterns is the max of the low 15 bits
    mag = (np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)).max()
    amax = float(bf16_bits_to_f32(np.array([mag], dtype=np.uint16))[0])
    return float(np.float32(amax) / np.float32(FP8_MAX))


def redraw_rows(seed: int, tensor_name: str, row: int, attempt: int, shape: tuple,
                dist: str) -> np.ndarray:
    """Fresh bf16 bits for one leading-axis row of a tensor (e.g. one token's
    idx_q rows, shape [Hidx, d]), drawn like ``draw_tensor`` (with the
    tensor's own channel vector for "channel") from the sub-stream
    (seed, 100 + tensor, row, attempt): a re-draw is deterministic and does
    not depend on which other rows were redrawn."""
    tid = {"q": _Q, "k": _K, "v": _V, "idx_q": _IQ, "idx_k": _IK}[tensor_name]
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 100 + tid, row, attempt])))
    last = shape[-1]
    x = g.standard_normal(shape, dtype=np.float32)
    if dist == "channel":
        x *= _channel_vector(seed, tid, last)
    return to_bf16_bits(x)


def idx_q_redraw(w: "GQAWorkload"):
    """The re-draw of one token's idx_q rows for a workload: a callable
    (token, attempt) -> bf16 bits [Hidx, d_idx]."""
    shape = w.idx_q.shape[1:]
    return lambda t, attempt: redraw_rows(w.seed, "idx_q", t, attempt, shape, w.cfg.dist)


@dataclass
class GQAWorkload:
    cfg: GQAConfig
    seq_lens: np.ndarray        # int32 [B]
    cu_q: np.ndarray            # int32 [B+1]
    page_table: np.ndarray      # int32 [B, max_pages], -1 where unused
    num_pages: int
    q: np.ndarray               # bf16 bits [T, Hq, D]
    idx_q: np.ndarray           # bf16 bits [T, Hidx, d_idx]
    k_pool: np.ndarray          # bf16 bits [num_pages, Hkv, 128, D]
    v_pool: np.ndarray          # bf16 bits [num_pages, Hkv, 128, D]
    idx_k_pool: np.ndarray      # bf16 bits [num_pages, 128, d_idx]
    sink: np.ndarray            # fp32 [Hq]
    scales: Dict[str, float] = field(default_factory=dict)   # q, k, v, idx_q, idx_k
    sm_scale: float = 0.0
    seed: int = 0

    @property
    def T(self) -> int:
        return int(self.cu_q[-1])

    @property
    def max_q_len(self) -> int:
        return int(np.max(np.diff(self.cu_q)))


def make_gqa(cfg: GQAConfig, seed: Optional[int] = None, T_override: Optional[int] = None) -> GQAWorkload:
    """Draw a GQA workload (prefill or paged decode).

    ``T_override`` shrinks a prefill configuration to T tokens (same recipe),
    for parity tests that must finish in seconds on the CPU oracle.
    """
    seed = cfg.seed if seed is None else seed
    if cfg.seq_lens:
        seq_lens = np.array(cfg.seq_lens, dtype=np.int32)
        if T_override is not None:
            seq_lens = np.array([T_override], dtype=np.int32)
    else:
        lo, hi = cfg.len_range
        seq_lens = _rng(seed, _LEN).integers(lo, hi + 1, size=cfg.B).astype(np.int32)
    B = len(seq_lens)
    q_lens = seq_lens.copy() if cfg.q_len == 0 else np.full(B, cfg.q_len, dtype=np.int32)
    cu_q = np.zeros(B + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(q_lens)
    T = int(cu_q[-1])

    blocks = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    in_use = int(blocks.sum())
    num_pages = int(math.ceil(cfg.pool_factor * in_use))
    max_pages = max(cfg.max_pages, int(blocks.max()))
    perm = _rng(seed, _PT).permutation(num_pages).astype(np.int32)
    page_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(blocks[b])
        page_table[b, :n] = perm[off:off + n]
        off += n

    q = draw_tensor(seed, _Q, (T, cfg.Hq, cfg.D), cfg.dist)
    idx_q = draw_tensor(seed, _IQ, (T, cfg.Hidx, cfg.d_idx), cfg.dist)
    k_pool = draw_tensor(seed, _K, (num_pages, cfg.Hkv, PAGE, cfg.D), cfg.dist)
    v_pool = draw_tensor(seed, _V, (num_pages, cfg.Hkv, PAGE, cfg.D), cfg.dist)
    idx_k_pool = draw_tensor(seed, _IK, (num_pages, PAGE, cfg.d_idx), cfg.dist)
    sink = _rng(seed, _SINK).standard_normal(cfg.Hq).astype(np.float32)

    scales = {name: amax_scale(arr) for name, arr in
              (("q", q), ("idx_q", idx_q), ("k", k_pool), ("v", v_pool), ("idx_k", idx_k_pool))}
    if cfg.kv_scale_uniform:
        g = _rng(seed, _SCALE)
        scales["k"] = float(np.float32(g.uniform(0.25, 4.0)))
        scales["v"] = float(np.float32(g.uniform(0.25, 4.0)))
    return GQAWorkload(cfg, seq_lens, cu_q, page_table, num_pages, q, idx_q, k_pool, v_pool,
                       idx_k_pool, sink, scales, 1.0 / math.sqrt(cfg.D), seed)


@dataclass
class MLAWorkload:
    cfg: MLAConfig
    q: np.ndarray             # bf16 bits [T, H, d_qk]
    kv: np.ndarray            # bf16 bits [S_kv, d_qk]
    indices: np.ndarray       # int32 [T, topk], -1 padded
    topk_length: np.ndarray   # int32 [T]
    sink: np.ndarray          # fp32 [H]
    scales: Dict[str, float] = field(default_factory=dict)    # q, kv
    sm_scale: float = 0.0


def make_mla(cfg: MLAConfig, seed: Optional[int] = None, T_override: Optional[int] = None,
             S_override: Optional[int] = None, topk_override: Optional[int] = None,
             len_range: Optional[tuple] = None) -> MLAWorkload:
    """Draw a sparse-MLA workload; overrides shrink it for CPU-checkable cases."""
    seed = cfg.seed if seed is None else seed
    T = cfg.T if T_override is None else T_override
    S = cfg.S_kv if S_override is None else S_override
    topk = cfg.topk if topk_override is None else topk_override
    lo, hi = cfg.len_range if len_range is None else len_range
    q = draw_tensor(seed, _Q, (T, cfg.H, cfg.d_qk), "normal")
    kv = draw_tensor(seed, _KV, (S, cfg.d_qk), "normal")
    g = _rng(seed, _IDX)
    lengths = g.integers(lo, hi + 1, size=T).astype(np.int32)
    indices = np.full((T, topk), -1, dtype=np.int32)
    for t in range(T):
        pos = S - T + t
        n = int(min(lengths[t], pos + 1, topk))
        lengths[t] = n
        pick = g.choice(pos + 1, size=n, replace=False)
        indices[t, :n] = np.sort(pick)
    sink = _rng(seed, _SINK).standard_normal(cfg.H).astype(np.float32)
    scales = {"q": amax_scale(q), "kv": amax_scale(kv)}
    return MLAWorkload(cfg, q, kv, indices, lengths, sink, scales, 1.0 / math.sqrt(cfg.d_qk))


def random_topk(seed: int, seq_lens: np.ndarray, cu_q: np.ndarray, Hidx: int, topk: int) -> np.ndarray:
    """A seeded, valid block selection [Hidx, T, topk] (int32) to drive the
    attention step on its own: for each row, the query's own block plus
    topk-1 distinct earlier blocks drawn uniformly, sorted ascending, -1
    padded when the causal blocks do not exceed topk."""
    g = _rng(seed, 200)
    seq_lens = np.asarray(seq_lens, np.int64)
    cu_q = np.asarray(cu_q, np.int64)
    T = int(cu_q[-1])
    out = np.full((Hidx, T, topk), -1, dtype=np.int32)
    for b in range(len(seq_lens)):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        for t in range(q0, q1):
            own = (int(seq_lens[b]) - (q1 - q0) + (t - q0)) // PAGE
            for i in range(Hidx):
                if own + 1 <= topk:
                    out[i, t, :own + 1] = np.arange(own + 1)
                else:
                    pick = np.sort(g.choice(own, size=topk - 1, replace=False))
                    out[i, t, :topk - 1] = pick
                    out[i, t, topk - 1] = own
    return out


def rotary_table(max_pos: int, d_rope: int, base: float = 10000.0) -> np.ndarray:
    """A standard rotary cos/sin table as a synthetic input: row p holds the
    d_rope/2 cosines then the d_rope/2 sines of p * base**(-2i/d_rope),
    evaluated in float64 and rounded to float32."""
    inv = base ** (-np.arange(0, d_rope, 2, dtype=np.float64) / d_rope)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
