"""Degenerate batches on the GPU path: no query tokens at all, and a
sequence with no query tokens between two that have some (its rows of cu_q
repeat). Compared with the oracle like the other parity tests."""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, attention as oa
from gpu_helpers import dev
from test_gpu_index_topk import _run as run_index_topk

pytestmark = pytest.mark.gpu


def test_empty_batches_return_empty_outputs(msa):
    w = wl.make_gqa(wl.CONFIGS["tiny"])
    cfg = w.cfg
    k8 = dev(oq.quantize(w.k_pool, w.scales["k"]))
    v8 = dev(oq.quantize(w.v_pool, w.scales["v"]))
    ik8 = dev(oq.quantize(w.idx_k_pool, w.scales["idx_k"]))
    pt, sl = dev(w.page_table), dev(w.seq_lens)
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    iq0 = torch.empty((0, cfg.Hidx, cfg.d_idx), dtype=torch.uint8, device="cuda")
    ids = msa.index_topk(iq0, ik8, pt, sl, cu, cfg.topk, 0)
    assert tuple(ids.shape) == (cfg.Hidx, 0, cfg.topk)
    q0 = torch.empty((0, cfg.Hq, cfg.D), dtype=torch.uint8, device="cuda")
    for max_q_len in (0, 1):
        o, ml, lse = msa.sparse_attn_fwd(q0, k8, v8, pt, sl, cu, ids, dev(w.sink), w.sm_scale,
                                         w.scales["q"], w.scales["k"], w.scales["v"], max_q_len)
        assert tuple(o.shape) == (0, cfg.Hq, cfg.D) and ml.numel() == 0 and lse.numel() == 0
    m = wl.make_mla(wl.CONFIGS["mla"], T_override=2, S_override=256, topk_override=64, len_range=(1, 64))
    kv8 = dev(oq.quantize(m.kv, m.scales["kv"]))
    q0 = torch.empty((0, 128, 576), dtype=torch.uint8, device="cuda")
    idx0 = torch.empty((0, 64), dtype=torch.int32, device="cuda")
    o, ml, lse = msa.sparse_mla_fwd(q0, kv8, idx0, None, None, m.sm_scale, m.scales["q"], m.scales["kv"])
    assert tuple(o.shape) == (0, 128, 512)
    msa.check_errors()


def _varlen_with_empty_sequence():
    cfg = wl.GQAConfig("varlen_empty", 3, (700, 300, 1500), 0, 16, 2, 4, 128, 128, 8, "channel",
                       pool_factor=1.2, seed=21)
    w = wl.make_gqa(cfg)
    q_lens = np.array([200, 0, 257], np.int32)       # the middle sequence has no query token
    w.cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(w.cu_q[-1])
    w.q, w.idx_q = w.q[:T], w.idx_q[:T]
    return w


def test_index_topk_with_an_empty_sequence(msa):
    run_index_topk(msa, _varlen_with_empty_sequence())


def test_attention_with_an_empty_sequence(msa):
    w = _varlen_with_empty_sequence()
    ids = wl.random_topk(22, w.seq_lens, w.cu_q, 4, 8)
    q8, k8, v8 = (oq.quantize(w.q, w.scales["q"]), oq.quantize(w.k_pool, w.scales["k"]),
                  oq.quantize(w.v_pool, w.scales["v"]))
    o, ml, lse = msa.sparse_attn_fwd(dev(q8), dev(k8), dev(v8), dev(w.page_table), dev(w.seq_lens),
                                     dev(w.cu_q), dev(ids), dev(w.sink), w.sm_scale, w.scales["q"],
                                     w.scales["k"], w.scales["v"], w.max_q_len)
    msa.check_errors()
    ref = oa.sparse_attention(q8, k8, v8, w.page_table, w.seq_lens, w.cu_q, ids, w.sink, w.sm_scale,
                              w.scales["q"], w.scales["k"], w.scales["v"])
    og = o.float().cpu().numpy().astype(np.float64)
    assert np.abs(og - ref[0]).max() <= 4e-2
    assert np.linalg.norm(og - ref[0]) / np.linalg.norm(ref[0]) <= 1e-2
    assert np.abs(lse.cpu().numpy() - ref[2]).max() <= 2e-3
