"""The failure path of the bounded device waits, driven without a fault.

With the library's debug switch on, every wait inside its kernels that is
not complete at its first test gives up at once: the kernel records a
timeout in the device error word, every role of the block stops waiting,
drains the copies and tensor-core operations it already issued, frees its
tensor memory and returns. This test runs each tensor-core entry point that
way on small cases and checks that

* no call faults: msa_check_errors reports MSA_ERR_TIMEOUT (or MSA_OK when
  every wait of a call completed within its first test, which may itself
  suspend the thread for a while before giving an answer), never a CUDA
  error; the prefill attention case, whose pipeline always waits longer
  than that, must report the timeout;
* with the switch off again, the same calls are exact against the oracle
  (the context is intact and nothing is left over in the shared state).
"""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq, index_topk as oi, no_tie
from gpu_helpers import dev
from test_gpu_attention import run_attention
from test_gpu_mla import _run as run_mla

pytestmark = pytest.mark.gpu


def _cases():
    pre = wl.make_gqa(wl.CONFIGS["tiny"], T_override=1300)
    dec = wl.make_gqa(wl.GQAConfig("dec", 24, (), 1, 16, 2, 4, 128, 128, 16, "channel",
                                   len_range=(1000, 9000), max_pages=80, pool_factor=1.2, seed=51))
    mla = wl.make_mla(wl.CONFIGS["mla"], T_override=12, S_override=32768, topk_override=2048,
                      len_range=(1500, 2048))
    return pre, dec, mla


def _index_call(msa, w):
    ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
    iq = oq.quantize(w.idx_q, w.scales["idx_q"])
    return msa.index_topk(dev(iq), dev(ik), dev(w.page_table), dev(w.seq_lens), dev(w.cu_q),
                          w.cfg.topk, w.max_q_len)


def _attn_call(msa, w, ids):
    q8 = oq.quantize(w.q, w.scales["q"])
    k8 = oq.quantize(w.k_pool, w.scales["k"])
    v8 = oq.quantize(w.v_pool, w.scales["v"])
    return msa.sparse_attn_fwd(dev(q8), dev(k8), dev(v8), dev(w.page_table), dev(w.seq_lens),
                               dev(w.cu_q), dev(ids), dev(w.sink), w.sm_scale, w.scales["q"],
                               w.scales["k"], w.scales["v"], w.max_q_len)


def _mla_call(msa, w):
    q8 = oq.quantize(w.q, w.scales["q"])
    kv8 = oq.quantize(w.kv, w.scales["kv"])
    return msa.sparse_mla_fwd(dev(q8), dev(kv8), dev(w.indices), dev(w.topk_length), dev(w.sink),
                              w.sm_scale, w.scales["q"], w.scales["kv"])


def _status(msa) -> int:
    torch.cuda.synchronize()
    try:
        msa.check_errors()
        return 0
    except msa.MsaError as e:
        return e.status


def test_forced_timeouts_drain_and_the_next_calls_are_exact(msa):
    pre, dec, mla = _cases()
    ids_pre = wl.random_topk(7, pre.seq_lens, pre.cu_q, pre.cfg.Hidx, pre.cfg.topk)
    ids_dec = wl.random_topk(8, dec.seq_lens, dec.cu_q, dec.cfg.Hidx, dec.cfg.topk)
    calls = {
        "index prefill": lambda: _index_call(msa, pre),
        "index decode": lambda: _index_call(msa, dec),
        "attention prefill": lambda: _attn_call(msa, pre, ids_pre),
        "attention decode": lambda: _attn_call(msa, dec, ids_dec),
        "sparse MLA": lambda: _mla_call(msa, mla),
    }
    assert _status(msa) == 0
    seen = {}
    msa.debug_force_timeouts(True)
    try:
        for name, call in calls.items():
            call()
            seen[name] = _status(msa)
    finally:
        msa.debug_force_timeouts(False)
    print("forced-timeout statuses:", seen)
    assert all(s in (0, 4) for s in seen.values()), seen
    assert seen["attention prefill"] == 4, seen
    assert _status(msa) == 0
    # the same work with the switch off: exact against the oracle
    for w in (pre, dec):
        ik = oq.quantize(w.idx_k_pool, w.scales["idx_k"])
        w.idx_q, _ = no_tie.redraw_near_ties(w.idx_q, w.scales["idx_q"], ik, w.page_table,
                                             w.seq_lens, w.cu_q, w.cfg.topk, wl.idx_q_redraw(w))
        got = _index_call(msa, w).cpu().numpy()
        msa.check_errors()
        ref, _ = oi.index_topk(oq.quantize(w.idx_q, w.scales["idx_q"]), ik, w.page_table,
                               w.seq_lens, w.cu_q, w.cfg.topk)
        assert np.array_equal(got, ref), w.cfg.name
    run_attention(msa, pre, ids_pre)
    run_attention(msa, dec, ids_dec)
    run_mla(msa, mla)
