"""The whole path chained on the GPU at the tiny configuration's full size:
quantise Q, idx_q and the caches, select blocks with the GPU's own index
top-k, then attend over the GPU's own selection -- each step's output is the
next step's input, and each is checked against the oracle:

* e4m3 codes and block ids bit for bit (every row; the inputs follow the
  no-tie rule, so each row has one correct selection);
* O, lse and max_logit against the oracle's attention over the oracle's own
  selection (equal to the GPU's, as just checked), at the bars of the
  attention tests.
"""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, index_topk as oi, attention as oa, no_tie
from gpu_helpers import dev, dev_bf16
from test_gpu_attention import _check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny"])
def test_whole_path_on_its_own_selection(msa, name):
    w = wl.make_gqa(wl.CONFIGS[name])
    cfg = w.cfg
    ik_ref = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    w.idx_q, red = no_tie.redraw_near_ties(w.idx_q, w.scales["idx_q"], ik_ref, w.page_table,
                                           w.seq_lens, w.cu_q, cfg.topk, wl.idx_q_redraw(w))
    # (a) quantise every fp8 operand on the GPU
    q8 = msa.quant_fp8(dev_bf16(w.q), w.scales["q"])
    iq8 = msa.quant_fp8(dev_bf16(w.idx_q), w.scales["idx_q"])
    k8 = msa.quant_fp8(dev_bf16(w.k_pool), w.scales["k"])
    v8 = msa.quant_fp8(dev_bf16(w.v_pool), w.scales["v"])
    ik8 = msa.quant_fp8(dev_bf16(w.idx_k_pool), w.scales["idx_k"])
    refs = {"q": oq.quantize(w.q, w.scales["q"]), "idx_q": oq.quantize(w.idx_q, w.scales["idx_q"]),
            "k": oq.quantize(w.k_pool, w.scales["k"]), "v": oq.quantize(w.v_pool, w.scales["v"]),
            "idx_k": ik_ref}
    for name_, got in (("q", q8), ("idx_q", iq8), ("k", k8), ("v", v8), ("idx_k", ik8)):
        assert np.array_equal(got.cpu().numpy(), refs[name_]), name_
    # (b) the GPU's own block selection
    pt, sl, cu = dev(w.page_table), dev(w.seq_lens), dev(w.cu_q)
    ids = msa.index_topk(iq8, ik8, pt, sl, cu, cfg.topk, w.max_q_len)
    ids_ref, gaps = oi.index_topk(refs["idx_q"], ik_ref, w.page_table, w.seq_lens, w.cu_q, cfg.topk)
    bound = no_tie.row_bounds(refs["idx_q"], ik_ref, w.page_table, w.seq_lens, w.cu_q, range(w.T))
    assert np.all(gaps > bound)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    # (c) attention over that selection
    o, ml, lse = msa.sparse_attn_fwd(q8, k8, v8, pt, sl, cu, ids, dev(w.sink), w.sm_scale,
                                     w.scales["q"], w.scales["k"], w.scales["v"], w.max_q_len)
    msa.check_errors()
    ref = oa.sparse_attention(refs["q"], refs["k"], refs["v"], w.page_table, w.seq_lens, w.cu_q,
                              ids_ref, w.sink, w.sm_scale, w.scales["q"], w.scales["k"],
                              w.scales["v"])
    got = (o.float().cpu().numpy().astype(np.float64), ml.cpu().numpy(), lse.cpu().numpy())
    err, rel = _check(got, ref)
    print(f"{name}: {len(red)} tokens redrawn; O max-abs {err:.2e}, rel-F {rel:.2e}")


def test_graph_replay_of_the_path_matches_the_oracle(msa):
    """The same chain (multi-tensor quantise -> index top-k -> attention, all
    launched with programmatic dependent launch) captured once as a CUDA
    graph and replayed: ids bit for bit and O / lse / max_logit against the
    oracle, on the tiny configuration."""
    import bench
    st = bench.gqa_setup(msa, wl, "tiny", torch.device("cuda:0"))
    w = st["w"]
    cfg = w.cfg
    ik_ref = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    w.idx_q, red = no_tie.redraw_near_ties(w.idx_q, w.scales["idx_q"], ik_ref, w.page_table,
                                           w.seq_lens, w.cu_q, cfg.topk, wl.idx_q_redraw(w))
    st["iq"].copy_(dev_bf16(w.idx_q))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                 # warm-up on a side stream before capture
        bench.run_path(msa, st)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for k in ("ids", "o", "ml", "lse"):
        st[k].zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bench.run_path(msa, st)
    g.replay()
    torch.cuda.synchronize()
    msa.check_errors()
    q_ref, iq_ref = oq.quantize(w.q, w.scales["q"]), oq.quantize(w.idx_q, w.scales["idx_q"])
    assert np.array_equal(st["q8"].cpu().numpy(), q_ref)
    assert np.array_equal(st["iq8"].cpu().numpy(), iq_ref)
    ids_ref, gaps = oi.index_topk(iq_ref, ik_ref, w.page_table, w.seq_lens, w.cu_q, cfg.topk)
    assert np.array_equal(st["ids"].cpu().numpy(), ids_ref)
    ref = oa.sparse_attention(q_ref, oq.quantize(w.k_pool, w.scales["k"]),
                              oq.quantize(w.v_pool, w.scales["v"]), w.page_table, w.seq_lens,
                              w.cu_q, ids_ref, w.sink, w.sm_scale, w.scales["q"], w.scales["k"],
                              w.scales["v"])
    got = (st["o"].float().cpu().numpy().astype(np.float64), st["ml"].cpu().numpy(),
           st["lse"].cpu().numpy())
    err, rel = _check(got, ref)
    print(f"graph replay: {len(red)} tokens redrawn; O max-abs {err:.2e}, rel-F {rel:.2e}")
