"""The allocation-free index top-k entry point against the regular one.

msa_index_topk_noalloc serves callers that cannot allocate device memory: it
keeps its scratch in the library's fixed device array instead of a caller
workspace. Its output must equal msa_index_topk's (block ids are integer
results: bit for bit) on consecutive calls that reuse the shared scratch.
This file is collected last, and the test also passes on its own in a fresh
process (the first call sets up the scratch address).
"""

import ctypes

import numpy as np
import pytest

from fp8_block_sparse_gb300 import workloads as wl
from oracle import quant as oq

pytestmark = pytest.mark.gpu


def _inputs(cfg):
    import torch
    w = wl.make_gqa(cfg)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    iq = t(oq.quantize(w.idx_q, w.scales["idx_q"]))
    ik = t(oq.quantize(w.idx_k_pool, w.scales["idx_k"]))
    return w, iq, ik, t(w.page_table), t(w.seq_lens), t(w.cu_q)


def test_noalloc_matches_workspace_entry_on_consecutive_calls(msa):
    import torch
    cases = [
        # many short decode sequences, then a prefill that reuses the same scratch
        wl.GQAConfig("dec", 96, (), 1, 16, 2, 4, 128, 128, 16, "channel",
                     len_range=(100, 20000), max_pages=160, pool_factor=1.2, seed=21),
        wl.GQAConfig("pre", 1, (2000,), 0, 8, 1, 1, 128, 64, 8, "normal", seed=22),
    ]
    for cfg in cases:
        w, iq, ik, pt, sl, cu = _inputs(cfg)
        ref = msa.index_topk(iq, ik, pt, sl, cu, cfg.topk, w.max_q_len)
        got = msa.index_topk_noalloc(iq, ik, pt, sl, cu, cfg.topk, w.max_q_len)
        torch.cuda.synchronize()
        msa.check_errors()
        assert torch.equal(got, ref), cfg.name


def test_noalloc_rejects_sizes_beyond_its_scratch(msa):
    import torch
    lib = msa.load()
    T, Hidx, max_pages = 8192, 4, 64          # 8 MiB of scores alone: over the limit
    assert lib.msa_index_topk_workspace_size(T, Hidx, max_pages) > 8 << 20
    p = ctypes.c_void_p(256)
    out = torch.empty((Hidx, T, 16), dtype=torch.int32, device="cuda")
    st = lib.msa_index_topk_noalloc(p, p, p, p, p, 1, T, T, Hidx, 128, 16, 64, max_pages,
                                    ctypes.c_void_p(out.data_ptr()), None)
    assert st == 5
    assert b"fixed scratch" in lib.msa_last_error_string()
