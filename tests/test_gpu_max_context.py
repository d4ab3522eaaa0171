"""The largest context the path accepts: one sequence of 2048 * 128 - 5
tokens (a 2048-entry page table) in decode and as a 256-token prefill at the
end of that context. The prefill tiles then walk unions of up to all 2048
blocks. Checked against the oracle on sampled query tokens."""

import numpy as np
import pytest

from fp8_block_sparse_gb300 import workloads as wl
from test_gpu_attention import run_attention
from test_gpu_index_topk import _run as run_index_topk

pytestmark = pytest.mark.gpu

L_MAX = 2048 * 128 - 5


@pytest.mark.parametrize("q_len", [1, 256])
def test_longest_context(msa, q_len):
    cfg = wl.GQAConfig("maxctx", 1, (L_MAX,), q_len, 16, 2, 4, 128, 128, 64, "normal",
                       max_pages=2048, seed=40 + q_len)
    w = wl.make_gqa(cfg)
    assert w.page_table.shape[1] == 2048
    tok = np.arange(w.T) if w.T <= 8 else np.concatenate(
        [np.sort(np.random.default_rng(q_len).choice(w.T - 1, size=8, replace=False)), [w.T - 1]])
    run_index_topk(msa, w, tokens=tok)
    ids = wl.random_topk(41, w.seq_lens, w.cu_q, cfg.Hidx, cfg.topk)
    run_attention(msa, w, ids, tokens=tok)
