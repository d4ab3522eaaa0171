"""Fused rotary embedding + e4m3 quantisation of MLA-style q / k rows (the
producer that replaces step a1 for the sparse-MLA inputs).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, and where the pages say so:

* sglang PR 25460 page, implementation step 2 and the excerpt of
  ``_fused_rope_fp8_quantize``: the rotary embedding is applied to the
  ``pe`` part of each q / k head (positions index a cos/sin cache; a flag
  selects the neox layout), then the ``nope`` part and the rotated ``pe``
  part are written side by side along the last dimension as one contiguous
  e4m3 row (``out[..., :d_nope]`` and ``out[..., d_nope:]``), with a
  quantisation scale; a k_pe shared by all heads is broadcast.
* Same page, key source excerpt of ``fp8_quantize``: values are widened to
  fp32, scaled and cast to e4m3.

Readings where the pages are silent:

* ``cos_sin_cache[pos]`` holds the d_rope/2 cosines followed by the d_rope/2
  sines of that position's angles.
* neox layout: the pe vector is split into halves (x1, x2), rotated as
  (x1 c - x2 s, x2 c + x1 s); otherwise pairs of neighbours (x[2i], x[2i+1])
  are rotated by angle i.
* the rotation runs in fp32, each product and each sum rounded to fp32 (no
  fused multiply-add), and the rotated fp32 value goes straight to the
  quantiser (no rounding to the input dtype in between);
* the quantiser is the path's rule, ``e4m3(fp32(v) * fp32(1 / scale))``, no
  multiply when the scale is absent, for both parts.
"""

from __future__ import annotations

from typing import Optional

import numpy as np

from . import e4m3, quant


def _widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return quant.bf16_bits_to_f32(bits)
    if dtype == "fp16":
        return quant.f16_bits_to_f32(bits)
    raise ValueError(f"unsupported input dtype {dtype!r}")


def rope(pe: np.ndarray, cos_sin_cache: np.ndarray, positions: np.ndarray, is_neox: bool) -> np.ndarray:
    """fp32 rotary embedding of pe [rows, heads, d_rope] (fp32 values).

    Row r uses cos_sin_cache[positions[r]]; every product and every sum is
    an fp32 operation (numpy float32 arithmetic, one rounding each).
    """
    pe = np.asarray(pe, dtype=np.float32)
    d = pe.shape[-1]
    half = d // 2
    cs = np.asarray(cos_sin_cache, dtype=np.float32)[np.asarray(positions, dtype=np.int64)]
    c = cs[:, None, :half]
    s = cs[:, None, half:]
    out = np.empty_like(pe)
    if is_neox:
        x1, x2 = pe[..., :half], pe[..., half:]
        out[..., :half] = x1 * c - x2 * s
        out[..., half:] = x2 * c + x1 * s
    else:
        x1, x2 = pe[..., 0::2], pe[..., 1::2]
        out[..., 0::2] = x1 * c - x2 * s
        out[..., 1::2] = x2 * c + x1 * s
    return out


def rope_quant(nope_bits: np.ndarray, pe_bits: np.ndarray, cos_sin_cache: np.ndarray,
               positions: np.ndarray, is_neox: bool, scale: Optional[float] = None,
               dtype: str = "bf16") -> np.ndarray:
    """e4m3 codes [rows, heads, d_nope + d_rope] of nope || rope(pe).

    nope_bits: [rows, heads, d_nope] bit patterns; pe_bits: [rows, heads or 1,
    d_rope] (a single head is broadcast to every head).
    """
    nope = _widen(nope_bits, dtype)
    pe = _widen(pe_bits, dtype)
    rows, heads, d_nope = nope.shape
    if pe.shape[1] == 1 and heads > 1:
        pe = np.broadcast_to(pe, (rows, heads, pe.shape[2]))
    rotated = rope(pe, cos_sin_cache, positions, is_neox)
    s_inv = quant.scale_inverse(scale)
    out = np.empty((rows, heads, d_nope + pe.shape[2]), dtype=np.uint8)
    out[..., :d_nope] = e4m3.encode((nope * s_inv).astype(np.float32))
    out[..., d_nope:] = e4m3.encode((rotated * s_inv).astype(np.float32))
    return out
