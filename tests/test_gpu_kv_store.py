"""GPU parity of msa_kv_store_fp8 (the quantised KV-cache store that feeds
the path) against the oracle: every byte of the three pools must match,
including the slots the store must leave alone (they start as seeded random
bytes)."""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import kv_store as okv
from oracle.index_topk import query_positions
from gpu_helpers import dev, dev_bf16

pytestmark = pytest.mark.gpu


def _new_rows(w):
    """The new tokens' K, V, index-K bit patterns, read from the pools in
    logical order (the values a model would produce for those positions)."""
    seq, pos = query_positions(w.seq_lens, w.cu_q)
    pages = w.page_table[seq, pos // 128]
    slots = pos % 128
    return w.k_pool[pages, :, slots], w.v_pool[pages, :, slots], w.idx_k_pool[pages, slots]


def _random_caches(w, seed):
    g = np.random.default_rng(seed)
    c = w.cfg
    kc = g.integers(0, 256, (w.num_pages, c.Hkv, 128, c.D), dtype=np.uint8)
    vc = g.integers(0, 256, (w.num_pages, c.Hkv, 128, c.D), dtype=np.uint8)
    ic = g.integers(0, 256, (w.num_pages, 128, c.d_idx), dtype=np.uint8)
    return kc, vc, ic


def _store(msa, w, caches, k, v, ik, scales, to_dev=dev_bf16):
    kc, vc, ic = (dev(c) if c is not None else None for c in caches)
    msa.kv_store_fp8(dev(w.page_table), dev(w.seq_lens), dev(w.cu_q), kc, vc, ic,
                     k=None if k is None else to_dev(k), v=None if v is None else to_dev(v),
                     idx_k=None if ik is None else to_dev(ik),
                     k_scale=scales[0], v_scale=scales[1], idx_k_scale=scales[2])
    return kc, vc, ic


def _same(got, want):
    for g, r in zip(got, want):
        if r is None:
            continue
        np.testing.assert_array_equal(g.cpu().numpy(), r)


def test_varlen_prefill_with_prefix(msa):
    cfg = wl.GQAConfig("kv_varlen", 3, (700, 1500, 2100), 0, 16, 2, 4, 128, 128, 8, "channel",
                       pool_factor=1.2, seed=61)
    w = wl.make_gqa(cfg)
    q_lens = np.array([700, 300, 257], np.int32)
    w.cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    k, v, ik = _new_rows(w)
    caches = _random_caches(w, 1)
    scales = (w.scales["k"], None, w.scales["idx_k"])
    got = _store(msa, w, caches, k, v, ik, scales)
    msa.check_errors()
    _same(got, okv.kv_store(w.page_table, w.seq_lens, w.cu_q, *caches, k=k, v=v, idx_k=ik,
                            k_scale=scales[0], v_scale=scales[1], idx_k_scale=scales[2]))


def test_decode_batch_fp16_slices_of_a_fused_row(msa):
    # K, V and index K are column slices of one fused [T, Hq*D + 2*Hkv*D + d_idx]
    # fp16 projection output: token stride = the fused row, per-token blocks contiguous
    cfg = wl.GQAConfig("kv_dec", 64, (), 1, 16, 2, 4, 128, 128, 16, "channel",
                       len_range=(1, 5000), max_pages=48, pool_factor=1.2, seed=62)
    w = wl.make_gqa(cfg)
    T, Hkv, D, di, Hq = w.T, cfg.Hkv, cfg.D, cfg.d_idx, cfg.Hq
    g = np.random.default_rng(3)
    fused = (g.standard_normal((T, Hq * D + 2 * Hkv * D + di)) * 3).astype(np.float16)
    bits = fused.view(np.uint16)
    o_k, o_v, o_i = Hq * D, Hq * D + Hkv * D, Hq * D + 2 * Hkv * D
    k = bits[:, o_k:o_v].reshape(T, Hkv, D)
    v = bits[:, o_v:o_i].reshape(T, Hkv, D)
    ik = bits[:, o_i:]
    fd = torch.from_numpy(fused).cuda()
    kt, vt, it = fd[:, o_k:o_v].view(T, Hkv, D), fd[:, o_v:o_i].view(T, Hkv, D), fd[:, o_i:]
    assert kt.stride(0) == fused.shape[1] and not kt.is_contiguous()
    caches = _random_caches(w, 2)
    kc, vc, ic = (dev(c) for c in caches)
    msa.kv_store_fp8(dev(w.page_table), dev(w.seq_lens), dev(w.cu_q), kc, vc, ic, k=kt, v=vt, idx_k=it,
                     k_scale=0.0173, v_scale=3.25, idx_k_scale=None)
    msa.check_errors()
    want = okv.kv_store(w.page_table, w.seq_lens, w.cu_q, *caches, k=k, v=v, idx_k=ik,
                        k_scale=0.0173, v_scale=3.25, idx_k_scale=None, dtype="fp16")
    _same((kc, vc, ic), want)


def test_index_k_only_leaves_kv_untouched(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=333)
    _, _, ik = _new_rows(w)
    caches = _random_caches(w, 3)
    got = _store(msa, w, caches, None, None, ik, (None, None, w.scales["idx_k"]))
    msa.check_errors()
    _same(got, (caches[0], caches[1], okv.kv_store(w.page_table, w.seq_lens, w.cu_q, None, None,
                                                   caches[2], idx_k=ik,
                                                   idx_k_scale=w.scales["idx_k"])[2]))


def test_prefill32k_full_sequence(msa):
    # the whole 32k-token sequence stored at the size and launch shape the
    # benchmark times; every byte of the three pools checked
    w = wl.make_gqa(wl.CONFIGS["prefill32k"])
    k, v, ik = _new_rows(w)
    caches = _random_caches(w, 4)
    scales = (w.scales["k"], w.scales["v"], w.scales["idx_k"])
    got = _store(msa, w, caches, k, v, ik, scales)
    msa.check_errors()
    _same(got, okv.kv_store(w.page_table, w.seq_lens, w.cu_q, *caches, k=k, v=v, idx_k=ik,
                            k_scale=scales[0], v_scale=scales[1], idx_k_scale=scales[2]))


def test_bad_page_is_reported_and_other_sequences_stored(msa):
    cfg = wl.GQAConfig("kv_bad", 5, (), 1, 16, 2, 4, 128, 128, 8, "channel",
                       len_range=(100, 900), max_pages=8, pool_factor=1.5, seed=63)
    w = wl.make_gqa(cfg)
    k, v, ik = _new_rows(w)
    bad = 2
    pos = int(w.seq_lens[bad]) - 1
    w.page_table = w.page_table.copy()
    w.page_table[bad, pos // 128] = w.num_pages + 7
    caches = _random_caches(w, 5)
    got = _store(msa, w, caches, k, v, ik, (None, None, None))
    with pytest.raises(msa.MsaError) as e:
        msa.check_errors()
    assert e.value.status == 6
    want = [c.copy() for c in caches]
    for b in range(cfg.B):
        if b == bad:
            continue
        sl = slice(b, b + 1)
        want = list(okv.kv_store(w.page_table[sl], w.seq_lens[sl], np.array([0, 1], np.int32), *want,
                                 k=k[sl], v=v[sl], idx_k=ik[sl]))
    _same(got, want)


def test_more_new_tokens_than_cached_is_reported(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=200)
    k, v, ik = _new_rows(w)
    w.seq_lens = np.array([150], np.int32)          # 200 new tokens, 150 in the cache
    caches = _random_caches(w, 6)
    _store(msa, w, caches, k, v, ik, (None, None, None))
    with pytest.raises(msa.MsaError) as e:
        msa.check_errors()
    assert e.value.status == 6


def test_empty_batch_is_a_no_op(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=10)
    caches = _random_caches(w, 7)
    kc, vc, ic = (dev(c) for c in caches)
    empty = torch.empty((0, w.cfg.Hkv, w.cfg.D), dtype=torch.bfloat16, device="cuda")
    msa.kv_store_fp8(dev(w.page_table), dev(w.seq_lens), dev(np.zeros(2, np.int32)), kc, vc, ic,
                     k=empty, v=empty)
    msa.check_errors()
    _same((kc, vc, ic), caches)
