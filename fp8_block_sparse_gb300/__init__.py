"""GB300 (sm_103a) FP8 e4m3 top-k block-sparse attention.

The compute path lives in ``libmsa.so`` (hand-written CUDA kernels behind a
C ABI declared in ``include/msa.h``); this package is a thin ctypes binding
with the same entry-point names plus the seeded workload generator.
"""

from .binding import (  # noqa: F401
    load, lib_path, MsaError, check_errors, debug_force_timeouts, profile_enable, profile_last_ms,
    quant_fp8, quant_fp8_multi, kv_store_fp8, rope_quant_fp8, index_topk, index_topk_workspace_size, index_topk_noalloc,
    sparse_attn_fwd, sparse_attn_workspace_size, sparse_mla_fwd,
)
from . import workloads  # noqa: F401,E402
