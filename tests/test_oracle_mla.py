"""Pins for the oracle's sparse-MLA prefill (step a6)."""

import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import e4m3
from oracle.mla import sparse_mla


def _codes(g, shape, max_code=0x48):
    c = g.integers(0, max_code, size=shape).astype(np.uint8)
    return c | (g.integers(0, 2, size=shape).astype(np.uint8) << 7)


def test_single_key_closed_form():
    g = np.random.default_rng(1)
    T, H, dqk, dv, S = 5, 4, 72, 64, 50
    q = _codes(g, (T, H, dqk))
    kv = _codes(g, (S, dqk))
    idx = np.full((T, 8), -1, np.int32)
    idx[:, 0] = g.integers(0, S, size=T)
    idx[:, 1:4] = 3                                   # beyond topk_length: ignored
    tl = np.ones(T, np.int32)
    sink = g.standard_normal(H).astype(np.float32)
    sm, qs, kvs = 0.2, 1.3, 0.7
    o, ml, lse = sparse_mla(q, kv, idx, tl, sink, sm, qs, kvs, d_v=dv)
    for t in range(T):
        k = e4m3.decode(kv[idx[t, 0]])
        for h in range(H):
            l = sm * qs * kvs * float(e4m3.decode(q[t, h]) @ k)
            s = sm * qs * float(sink[h])
            w = math.exp(l) / (math.exp(l) + math.exp(s))
            np.testing.assert_allclose(o[t, h], kvs * w * k[:dv], rtol=1e-12, atol=1e-15)
            assert ml[t, h] == l
            assert abs(lse[t, h] - math.log(math.exp(l) + math.exp(s))) < 1e-12


def test_all_causal_indices_equal_dense_causal_mqa():
    g = np.random.default_rng(2)
    T, H, dqk, dv, S = 24, 4, 40, 32, 64
    q = _codes(g, (T, H, dqk))
    kv = _codes(g, (S, dqk))
    pos = S - T + np.arange(T)
    idx = np.full((T, S), -1, np.int32)
    for t in range(T):
        idx[t, : pos[t] + 1] = np.arange(pos[t] + 1)
    o, _, _ = sparse_mla(q, kv, idx, None, None, 0.15, None, None, d_v=dv)
    qq = torch.from_numpy(np.transpose(e4m3.decode(q), (1, 0, 2)))[None]     # [1, H, T, dqk]
    kk = torch.from_numpy(e4m3.decode(kv))[None, None].expand(1, H, S, dqk)
    vv = torch.from_numpy(e4m3.decode(kv[:, :dv]))[None, None].expand(1, H, S, dv)
    mask = torch.from_numpy(np.arange(S)[None, :] <= pos[:, None])          # causal at offset
    ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=0.15)[0]
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-13)


def test_topk_length_equals_explicit_padding_and_order_is_irrelevant():
    g = np.random.default_rng(3)
    T, H, dqk, dv, S, topk = 6, 2, 32, 16, 40, 12
    q = _codes(g, (T, H, dqk))
    kv = _codes(g, (S, dqk))
    idx = np.stack([np.sort(g.choice(S, size=topk, replace=False)) for _ in range(T)]).astype(np.int32)
    tl = g.integers(1, topk + 1, size=T).astype(np.int32)
    padded = idx.copy()
    for t in range(T):
        padded[t, tl[t]:] = -1
    shuffled = padded.copy()
    for t in range(T):
        g.shuffle(shuffled[t])
    sink = g.standard_normal(H).astype(np.float32)
    a = sparse_mla(q, kv, idx, tl, sink, 0.3, 2.0, 0.5, d_v=dv)
    b = sparse_mla(q, kv, padded, None, sink, 0.3, 2.0, 0.5, d_v=dv)
    c = sparse_mla(q, kv, shuffled, None, sink, 0.3, 2.0, 0.5, d_v=dv)
    for x, y in ((a, b), (a, c)):
        for u, w in zip(x, y):
            np.testing.assert_allclose(u, w, rtol=1e-12, atol=1e-15)
