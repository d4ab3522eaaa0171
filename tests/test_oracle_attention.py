"""Pins for the oracle's sparse GQA attention with sink (steps a4/a5).

The independent references are torch's scaled_dot_product_attention in
float64 (math backend) on the decoded values, with the sink realised as an
extra key whose additive mask is the sink logit and whose value carries a
one-hot marker channel (its output weight gives e^{sigma - lse}), and closed
forms.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import e4m3
from oracle.attention import sparse_attention


def _codes(g, shape, max_code=0x48):
    c = g.integers(0, max_code, size=shape).astype(np.uint8)       # |v| <= 4
    return c | (g.integers(0, 2, size=shape).astype(np.uint8) << 7)


def _random_topk(g, T, hidx, topk, pos):
    ids = np.full((hidx, T, topk), -1, np.int32)
    for i in range(hidx):
        for t in range(T):
            own = int(pos[t]) // 128
            if own + 1 <= topk:
                sel = list(range(own + 1))
            else:
                sel = sorted(g.choice(own, size=topk - 1, replace=False).tolist()) + [own]
            ids[i, t, :len(sel)] = sel
    return ids


def _case(seed, T, hq, hkv, hidx, topk, D=32, extra_pages=2):
    g = np.random.default_rng(seed)
    nblk = (T + 127) // 128
    n_pages = nblk + extra_pages
    pt = g.permutation(n_pages)[:nblk].astype(np.int32)[None, :]
    q = _codes(g, (T, hq, D))
    k = _codes(g, (n_pages, hkv, 128, D))
    v = _codes(g, (n_pages, hkv, 128, D))
    sink = g.standard_normal(hq).astype(np.float32)
    sl = np.array([T], np.int32)
    cu = np.array([0, T], np.int32)
    return g, q, k, v, pt, sl, cu, sink


def _logical(pool, pt, T):
    """[num_pages, Hkv, 128, D] -> [Hkv, T, D] for sequence 0."""
    blocks = pool[pt[0]]                                   # [nblk, Hkv, 128, D]
    return np.transpose(blocks, (1, 0, 2, 3)).reshape(pool.shape[1], -1, pool.shape[3])[:, :T]


def _sdpa(qv, kv, vv, allowed, scale, sigma):
    """Per-head SDPA with sink. qv [H,T,D]; kv,vv [H,S,D]; allowed [H,T,S] bool.

    Returns (O [H,T,D], lse [H,T]).
    """
    H, T, D = qv.shape
    S = kv.shape[1]
    q = torch.from_numpy(qv)[None]
    k = torch.cat([torch.from_numpy(kv), torch.zeros(H, 1, D, dtype=torch.float64)], 1)[None]
    v = torch.cat([torch.from_numpy(vv), torch.zeros(H, 1, D, dtype=torch.float64)], 1)
    marker = torch.zeros(H, S + 1, 1, dtype=torch.float64)
    marker[:, S] = 1.0
    v = torch.cat([v, marker], 2)[None]
    mask = torch.full((H, T, S + 1), -math.inf, dtype=torch.float64)
    mask[:, :, :S][torch.from_numpy(np.ascontiguousarray(allowed))] = 0.0
    mask[:, :, S] = torch.from_numpy(np.asarray(sigma, np.float64))[:, None]
    out = F.scaled_dot_product_attention(q, k, v, attn_mask=mask[None], scale=scale)[0]
    o = out[..., :D].numpy()
    lse = np.asarray(sigma, np.float64)[:, None] - np.log(out[..., D].numpy())
    return o, lse


def _reference(q, k, v, pt, T, ids, sink, sm, qs, ks, vs, hq, hkv, hidx):
    qv = np.transpose(e4m3.decode(q), (1, 0, 2))          # [Hq, T, D]
    kl = e4m3.decode(_logical(k, pt, T))                  # [Hkv, T, D]
    vl = e4m3.decode(_logical(v, pt, T))
    kv_h = kl[np.arange(hq) // (hq // hkv)]               # GQA: head h reads kv head h // group
    vv_h = vl[np.arange(hq) // (hq // hkv)]
    allowed = np.zeros((hq, T, T), bool)
    causal = np.tril(np.ones((T, T), bool))
    for h in range(hq):
        i = h // (hq // hidx)
        for t in range(T):
            sel = ids[i, t][ids[i, t] >= 0]
            blockmask = np.isin(np.arange(T) // 128, sel)
            allowed[h, t] = blockmask & causal[t]
    sigma = sm * qs * sink.astype(np.float64)
    o, lse = _sdpa(qv, kv_h, vv_h, allowed, sm * qs * ks, sigma)
    return vs * np.transpose(o, (1, 0, 2)), lse.T


@pytest.mark.parametrize("T,hq,hkv,hidx,topk", [(300, 4, 2, 2, 2), (257, 8, 1, 1, 1),
                                                (400, 4, 4, 1, 2), (130, 2, 1, 2, 3)])
def test_sparse_selection_matches_sdpa_with_block_mask(T, hq, hkv, hidx, topk):
    g, q, k, v, pt, sl, cu, sink = _case(T * 7 + hq, T, hq, hkv, hidx, topk)
    ids = _random_topk(g, T, hidx, topk, np.arange(T))
    sm, qs, ks, vs = 0.3, 0.7, 1.9, 0.45
    o, ml, lse = sparse_attention(q, k, v, pt, sl, cu, ids, sink, sm, qs, ks, vs)
    o_ref, lse_ref = _reference(q, k, v, pt, T, ids, sink, sm, qs, ks, vs, hq, hkv, hidx)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-10, atol=1e-10)
    assert np.all(lse >= ml)


def test_topk_covering_every_block_is_dense_causal_attention():
    T, hq, hkv, hidx = 384, 4, 2, 2
    g, q, k, v, pt, sl, cu, sink = _case(3, T, hq, hkv, hidx, 3)
    ids = _random_topk(g, T, hidx, 3, np.arange(T))        # 3 blocks: every causal block
    o, _, lse = sparse_attention(q, k, v, pt, sl, cu, ids, sink, 0.2, None, None, None)
    qv = np.transpose(e4m3.decode(q), (1, 0, 2))
    kl = e4m3.decode(_logical(k, pt, T))[np.arange(hq) // 2]
    vl = e4m3.decode(_logical(v, pt, T))[np.arange(hq) // 2]
    allowed = np.ascontiguousarray(np.broadcast_to(np.tril(np.ones((T, T), bool)), (hq, T, T)))
    o_ref, lse_ref = _sdpa(qv, kl, vl, allowed, 0.2, 0.2 * sink.astype(np.float64))
    np.testing.assert_allclose(o, np.transpose(o_ref, (1, 0, 2)), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.T, rtol=1e-10)


def test_single_selected_block_is_dense_attention_over_that_block():
    T = 512
    g, q, k, v, pt, sl, cu, sink = _case(4, T, 2, 1, 1, 1)
    ids = np.array([[[t // 128] for t in range(T)]], np.int32)        # topk = 1: own block
    o, _, _ = sparse_attention(q, k, v, pt, sl, cu, ids, None, 0.25, None, None, None)
    for blk in range(4):
        sl_ = slice(128 * blk, 128 * blk + 128)
        qv = torch.from_numpy(np.transpose(e4m3.decode(q[sl_]), (1, 0, 2)))[None]
        kb = torch.from_numpy(e4m3.decode(k[pt[0, blk], 0]))[None, None].expand(1, 2, 128, -1)
        vb = torch.from_numpy(e4m3.decode(v[pt[0, blk], 0]))[None, None].expand(1, 2, 128, -1)
        ref = F.scaled_dot_product_attention(qv, kb, vb, is_causal=True, scale=0.25)[0]
        np.testing.assert_allclose(o[sl_], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_sink_lowers_row_mass_by_the_closed_form():
    T = 200
    g, q, k, v, pt, sl, cu, sink = _case(5, T, 2, 1, 1, 2)
    ones = np.full_like(v, 0x38)                                       # every value = 1.0
    ids = _random_topk(g, T, 1, 2, np.arange(T))
    sm, qs = 0.3, 1.7
    o0, m0, lse0 = sparse_attention(q, k, ones, pt, sl, cu, ids, None, sm, qs, 2.0, None)
    o1, m1, lse1 = sparse_attention(q, k, ones, pt, sl, cu, ids, sink, sm, qs, 2.0, None)
    np.testing.assert_allclose(o0, 1.0, rtol=1e-13)                  # no sink: mass 1
    sigma = sm * qs * sink.astype(np.float64)                          # q_scale on the sink, k_scale not
    S = np.exp(lse0)                                                   # sum_j e^{l_j}
    mass = S / (S + np.exp(sigma)[None, :])
    np.testing.assert_allclose(o1[..., 0], mass, rtol=1e-12)
    np.testing.assert_allclose(lse1, np.logaddexp(lse0, sigma[None, :]), rtol=1e-12)
    np.testing.assert_array_equal(m0, m1)                              # max_logit excludes the sink


def test_scale_laws():
    T = 260
    g, q, k, v, pt, sl, cu, sink = _case(6, T, 4, 2, 1, 2)
    ids = _random_topk(g, T, 1, 2, np.arange(T))
    base = sparse_attention(q, k, v, pt, sl, cu, ids, sink, 0.3, 1.5, 1.0, 1.0)
    # v_scale multiplies the output only
    o_v, m_v, l_v = sparse_attention(q, k, v, pt, sl, cu, ids, sink, 0.3, 1.5, 1.0, 2.5)
    np.testing.assert_allclose(o_v, 2.5 * base[0], rtol=1e-13)
    np.testing.assert_array_equal(l_v, base[2])
    # doubling k_scale == doubling sm_scale on the dot while the sink stays put
    o_k, m_k, l_k = sparse_attention(q, k, v, pt, sl, cu, ids, sink, 0.3, 1.5, 2.0, 1.0)
    o_s, m_s, l_s = sparse_attention(q, k, v, pt, sl, cu, ids, sink / 2, 0.6, 1.5, 1.0, 1.0)
    np.testing.assert_allclose(o_k, o_s, rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(m_k, m_s, rtol=1e-13)
    np.testing.assert_allclose(l_k, l_s, rtol=1e-13)
    # q_scale and sm_scale only enter as a product
    o_q = sparse_attention(q, k, v, pt, sl, cu, ids, sink, 0.45, 1.0, 1.0, 1.0)
    np.testing.assert_allclose(o_q[0], base[0], rtol=1e-9, atol=1e-14)


def test_all_equal_keys_give_the_mass_weighted_mean_of_values():
    T = 256
    g, q, k, v, pt, sl, cu, sink = _case(7, T, 2, 1, 1, 2)
    k[:] = 0x30                                                          # every key = 0.5 * ones
    ids = _random_topk(g, T, 1, 2, np.arange(T))
    sm, qs, ks, vs = 0.1, 1.2, 0.8, 1.3
    o, ml, lse = sparse_attention(q, k, v, pt, sl, cu, ids, sink, sm, qs, ks, vs)
    qd = e4m3.decode(q)
    vl = e4m3.decode(_logical(v, pt, T))[0]
    for t in (0, 5, 127, 128, 200, 255):
        sel = ids[0, t][ids[0, t] >= 0]
        keys = [j for j in range(t + 1) if j // 128 in sel]
        for h in range(2):
            l = sm * qs * ks * 0.5 * qd[t, h].sum()
            n = len(keys)
            sigma = sm * qs * float(sink[h])
            mass = n * math.exp(l) / (n * math.exp(l) + math.exp(sigma))
            np.testing.assert_allclose(o[t, h], vs * mass * vl[keys].mean(0), rtol=1e-11, atol=1e-13)
            assert ml[t, h] == pytest.approx(l, rel=1e-14)
            assert lse[t, h] == pytest.approx(math.log(n * math.exp(l) + math.exp(sigma)), rel=1e-13)


def test_unit_scales_on_e4m3_exact_bf16_inputs_equal_bf16_attention():
    # unit scales: codes are the bf16 values themselves, so the fp8 path is
    # the plain attention of the (e4m3-exact) bf16 tensors
    T, hq = 150, 2
    g, q, k, v, pt, sl, cu, sink = _case(8, T, hq, 1, 1, 2)
    ids = _random_topk(g, T, 1, 2, np.arange(T))
    o8, _, l8 = sparse_attention(q, k, v, pt, sl, cu, ids, sink, 0.125, None, None, None)
    o_ref, l_ref = _reference(q, k, v, pt, T, ids, sink, 0.125, 1.0, 1.0, 1.0, hq, 1, 1)
    np.testing.assert_allclose(o8, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(l8, l_ref, rtol=1e-10)


def test_decode_rows_attend_to_their_sequence_prefix():
    g = np.random.default_rng(9)
    D, hq, hkv = 16, 2, 1
    n_pages = 9
    k = _codes(g, (n_pages, hkv, 128, D))
    v = _codes(g, (n_pages, hkv, 128, D))
    pt = np.array([[4, 0, 7, -1], [1, 2, 3, 5]], np.int32)
    sl = np.array([300, 512], np.int32)
    q = _codes(g, (2, hq, D))
    ids = np.array([[[0, 1, 2, -1], [0, 1, 2, 3]]], np.int32)          # everything causal
    o, _, lse = sparse_attention(q, k, v, pt, sl, np.array([0, 1, 2], np.int32), ids, None, 0.5)
    for b in range(2):
        L = int(sl[b])
        kl = e4m3.decode(_logical(k, pt[b:b + 1, :(L + 127) // 128], L))
        vl = e4m3.decode(_logical(v, pt[b:b + 1, :(L + 127) // 128], L))
        qq = torch.from_numpy(e4m3.decode(q[b]))[None, :, None, :]         # [1, hq, 1, D]
        ref = F.scaled_dot_product_attention(qq, torch.from_numpy(kl)[None].expand(1, hq, L, D),
                                             torch.from_numpy(vl)[None].expand(1, hq, L, D),
                                             scale=0.5)[0, :, 0]
        np.testing.assert_allclose(o[b], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_row_without_keys():
    T = 10
    g, q, k, v, pt, sl, cu, sink = _case(10, T, 2, 1, 1, 1)
    ids = np.full((1, T, 1), -1, np.int32)
    o, ml, lse = sparse_attention(q, k, v, pt, sl, cu, ids, sink, 0.5, 2.0, None, None)
    assert np.all(o == 0) and np.all(np.isneginf(ml))
    np.testing.assert_allclose(lse, np.broadcast_to(0.5 * 2.0 * sink.astype(np.float64), (T, 2)))
