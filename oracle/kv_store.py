"""The quantised KV-cache store that feeds the path (the next row after it).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, and where the pages say so:

* sglang PR 30971 page, implementation step 4 (memory_pool.py): the sparse KV
  pool's stores (``set_kv_buffer`` for K and V, ``set_index_k_buffer`` for
  the index K) write the new tokens' keys and values into the paged fp8
  pools, each with a per-tensor scale whose default is ``None``; ``None``
  means the unit scale and no division at all.
* Same page, implementation step 3: the store runs before the query
  quantiser, so the path reads the cache these stores wrote.
* vLLM PR 45892 page, implementation step 3: the index-K cache has no head
  axis, one row of ``d_idx`` codes per token slot.

Readings where the pages are silent:

* the stored code of an element is the path's quantiser rule,
  ``e4m3(fp32(x) * fp32(1 / scale))``, the same rule as the query
  quantiser. The pool's non-unit path divides in the input dtype before the
  cast; the two agree whenever the scale is absent or a power of two, and
  one rule for every fp8 operand keeps the cache and the queries coded alike.
* the slots are addressed by the batch description the attention uses: new
  token ``i`` of sequence ``b`` sits at position
  ``p = seq_lens[b] - q_len_b + i``, physical page ``page_table[b, p // 128]``,
  slot ``p % 128``. Every other slot of the pools is left as it was.
"""

from __future__ import annotations

from typing import Optional

import numpy as np

from . import quant
from .index_topk import query_positions

PAGE = 128


def slot_addresses(page_table: np.ndarray, seq_lens: np.ndarray, cu_q: np.ndarray):
    """(page, slot) of every new token, in token order.

    Raises ValueError when a position has no page-table entry or the entry is
    outside the pool, which the device reports as a data error.
    """
    seq, pos = query_positions(seq_lens, cu_q)
    page_table = np.asarray(page_table)
    pages = np.empty(len(pos), dtype=np.int64)
    for t in range(len(pos)):
        j = int(pos[t]) // PAGE
        if pos[t] < 0 or j >= page_table.shape[1]:
            raise ValueError(f"token {t}: position {int(pos[t])} has no page-table entry")
        pages[t] = int(page_table[seq[t], j])
    return pages, pos % PAGE


def kv_store(page_table: np.ndarray, seq_lens: np.ndarray, cu_q: np.ndarray,
             k_cache: Optional[np.ndarray], v_cache: Optional[np.ndarray],
             idx_k_cache: Optional[np.ndarray],
             k: Optional[np.ndarray] = None, v: Optional[np.ndarray] = None,
             idx_k: Optional[np.ndarray] = None,
             k_scale: Optional[float] = None, v_scale: Optional[float] = None,
             idx_k_scale: Optional[float] = None, dtype: str = "bf16"):
    """Returns copies of the three caches with the new tokens stored.

    k, v:   [T, Hkv, D] bf16 / fp16 bit patterns (uint16), or None to skip.
    idx_k:  [T, d_idx] bit patterns, or None to skip.
    k_cache, v_cache: [num_pages, Hkv, 128, D] e4m3 codes (uint8).
    idx_k_cache:      [num_pages, 128, d_idx] e4m3 codes.
    """
    pages, slots = slot_addresses(page_table, seq_lens, cu_q)
    out = []
    for x, cache, scale, headed in ((k, k_cache, k_scale, True), (v, v_cache, v_scale, True),
                                    (idx_k, idx_k_cache, idx_k_scale, False)):
        if cache is None:
            out.append(None)
            continue
        cache = np.array(cache, dtype=np.uint8, copy=True)
        if x is not None:
            codes = quant.quantize(x, scale, dtype)
            for t in range(len(pages)):
                page = int(pages[t])
                if page < 0 or page >= cache.shape[0]:
                    raise ValueError(f"token {t}: page {page} outside the pool")
                if headed:
                    cache[page, :, slots[t], :] = codes[t]
                else:
                    cache[page, slots[t], :] = codes[t]
        out.append(cache)
    return tuple(out)
