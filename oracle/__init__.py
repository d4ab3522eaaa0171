"""CPU oracle for FP8 (e4m3) top-k block-sparse attention.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, float64 restatement
of what the GPU path computes. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it;
the product library never does, and it shares no code with the CUDA kernels.

Sources (the four web pages this method is described on):

* sglang PR 30971 page, "M3 attention GEMMs fully fp8" -- the q/idx_q
  quantiser ``_quant_q_fp8``, the strictly ascending block-id top-k contract
  and the per-tensor scale semantics (implementation steps 2 and 3); the
  paged pool's K / V / index-K stores (step 4).
* vLLM PR 45892 page, "SM100 MSA indexer backend for MiniMax M3" -- indexer
  scoring reduced per 128-token page (``max_score``), the shared
  ``topk_indices_buffer[index_heads, tokens, topk]`` and the head-less fp8
  index-K cache (implementation steps 1-3).
* sglang PR 25751 page, "SM90 Q8KV8 FP8 sparse MLA prefill JIT kernel" -- the
  sparse-MLA prefill API with ``attn_sink`` and ``topk_length`` and its
  ``out / max_logits / lse`` outputs (key source excerpt).
* sglang PR 25460 page, "prefill QKV quantize hook and FP8 Triton kernel" --
  the per-tensor quantiser ``(x.to(fp32) * scale_inv).to(fp8)`` (key source
  excerpt of ``fp8_quantize``).

Modules: ``e4m3`` (codec), ``quant`` (step a1), ``index_topk`` (steps a2+a3),
``attention`` (steps a4/a5), ``mla`` (step a6). Every function is pinned by
``tests/test_oracle_*.py`` against closed forms, brute force, library special
cases or hand-made golden fixtures; none is "parity unpinned".
"""

from . import e4m3, quant, index_topk, attention, mla  # noqa: F401
