"""The benchmark's work accounting, checked on CPU against brute-force counts.

The roofline figures divide algorithmic work by measured time, so the work
counts are checked here independently: selected causal keys (and so the
algorithmic FLOPs) by walking each row's keys one by one, the union-tile
work by explicit sets per tile, the decode step's bytes by explicit sets
per (sequence, kv head); the committed traffic figure is used only while the
kernel source matches the hash recorded beside it."""

import os

import numpy as np
import torch

import bench
from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, index_topk as oi
from oracle.attention import row_keys


def _prefill_state(T=700):
    w = wl.make_gqa(wl.CONFIGS["prefill8k"], T_override=T)
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    ids, _ = oi.index_topk(iq, ik, w.page_table, w.seq_lens, w.cu_q, w.cfg.topk)
    return {"w": w, "ids": torch.from_numpy(ids)}


def test_algorithmic_flops_count_every_selected_causal_key():
    st = _prefill_state()
    w, ids = st["w"], st["ids"].numpy()
    cfg = w.cfg
    brute = 0
    for h in range(cfg.Hq):
        i = h // (cfg.Hq // cfg.Hidx)
        for t in range(w.T):
            blk, _ = row_keys(ids[i, t], t)
            brute += 4 * cfg.D * len(blk)
    assert bench.alg_flops(st, bench.selected_keys(st)) == brute


def test_executed_flops_walk_each_tile_union():
    st = _prefill_state(T=900)
    w, ids = st["w"], st["ids"].numpy()
    cfg = w.cfg
    G = cfg.Hq // cfg.Hkv
    toks = 256 // G                         # two 128-row tiles of 128/G tokens x G heads
    hpi = cfg.Hq // cfg.Hidx
    blocks = 0
    for g in range(cfg.Hkv):
        heads = range(g * G, g * G + G)
        for t0 in range(0, w.T, toks):
            union = set()
            for t in range(t0, min(t0 + toks, w.T)):
                for h in heads:
                    union |= {int(b) for b in ids[h // hpi, t] if b >= 0}
            blocks += len(union)
    assert bench.executed_flops(st) == blocks * 2 * 128.0 * 128 * 128 * 4


def test_decode_bytes_read_each_union_block_once():
    cfg = wl.GQAConfig("acct_dec", 12, (), 1, 16, 2, 4, 128, 128, 16, "channel",
                       len_range=(100, 9000), max_pages=80, pool_factor=1.2, seed=71)
    w = wl.make_gqa(cfg)
    ids = wl.random_topk(3, w.seq_lens, w.cu_q, cfg.Hidx, cfg.topk)
    st = {"w": w, "ids": torch.from_numpy(ids), "sl": torch.from_numpy(w.seq_lens)}
    total, kv_bytes, union = bench.decode_bytes(st)
    G, hpi = cfg.Hq // cfg.Hkv, cfg.Hq // cfg.Hidx
    brute_union = 0
    for b in range(cfg.B):
        for g in range(cfg.Hkv):
            heads = {h // hpi for h in range(g * G, g * G + G)}
            brute_union += len({int(x) for i in heads for x in ids[i, b] if x >= 0})
    assert union == brute_union
    assert kv_bytes == brute_union * 2 * 128 * cfg.D
    idx_bytes = sum((int(L) - 1) // 128 for L in w.seq_lens) * 128 * cfg.d_idx
    small = w.T * (cfg.Hq * cfg.D * 3 + cfg.Hidx * cfg.d_idx * 3 + cfg.Hq * 2 * cfg.D + 8 * cfg.Hq)
    assert total == idx_bytes + kv_bytes + small


def test_committed_traffic_is_used_only_for_the_matching_source(monkeypatch, tmp_path):
    # a summary recording the hash of the kernel source it was taken on
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(
        "# a kernel\n- source_hash: `00aa11bb22cc33dd`\n- dram_bytes_per_launch: 1234.5\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "src_hash", lambda *names: "00aa11bb22cc33dd")
    assert bench.traffic_for("attn.cu", "k.md") == 1234.5
    assert bench.traffic_for("attn.cu", "missing.md") is None
    # any change to the kernel source changes its hash: the figure is then not used
    monkeypatch.setattr(bench, "src_hash", lambda *names: "0123456789abcdef")
    assert bench.traffic_for("attn.cu", "k.md") is None


def test_src_hash_follows_the_source_bytes():
    h = bench.src_hash("attn.cu", "common.cuh")
    assert len(h) == 16 and h == bench.src_hash("attn.cu", "common.cuh")
    assert h != bench.src_hash("mla.cu", "common.cuh")
