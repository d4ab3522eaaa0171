"""The whole path as one CUDA graph: quantise -> index top-k -> attention,
captured once and replayed (graph-chained launches; no host work between the
steps). The replay must reproduce the eager run bit for bit, and a replay
after new inputs are copied into the captured buffers must equal an eager
run on those inputs."""

import numpy as np
import pytest
import torch

import bench
from fp8_block_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

OUTS = ("q8", "iq8", "ids", "o", "ml", "lse")


def _setup(msa, cfg):
    wl.CONFIGS[cfg.name] = cfg
    try:
        return bench.gqa_setup(msa, wl, cfg.name, torch.device("cuda:0"))
    finally:
        del wl.CONFIGS[cfg.name]


def _snapshot(st):
    return {k: st[k].clone() for k in OUTS}


def _same(st, ref):
    for k in OUTS:
        assert torch.equal(st[k], ref[k]), k


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_graph_replay_is_bit_exact(msa, kind):
    if kind == "prefill":
        cfg = wl.GQAConfig("graph_prefill", 1, (1500,), 0, 16, 2, 4, 128, 128, 8, "channel", seed=51)
    else:
        cfg = wl.GQAConfig("graph_decode", 24, (), 1, 16, 2, 4, 128, 128, 16, "channel",
                           len_range=(100, 9000), max_pages=80, pool_factor=1.2, seed=52)
    st = _setup(msa, cfg)
    bench.run_path(msa, st)
    torch.cuda.synchronize()
    msa.check_errors()
    ref = _snapshot(st)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                 # warm-up on the capture stream's side
        bench.run_path(msa, st)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for k in OUTS:
        st[k].zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bench.run_path(msa, st)
    for k in OUTS:
        st[k].zero_()
    g.replay()
    torch.cuda.synchronize()
    msa.check_errors()
    _same(st, ref)

    # new activations in the captured input buffers: replay == eager on them
    gen = torch.Generator(device="cpu").manual_seed(53)
    st["q"].copy_((torch.randn(st["q"].shape, generator=gen) * 2).to(torch.bfloat16))
    st["iq"].copy_((torch.randn(st["iq"].shape, generator=gen) * 2).to(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    replayed = _snapshot(st)
    bench.run_path(msa, st)
    torch.cuda.synchronize()
    msa.check_errors()
    _same(st, replayed)
    assert not torch.equal(replayed["o"], ref["o"])
