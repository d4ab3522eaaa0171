"""Step a1: per-tensor e4m3 quantisation of Q and idx_q.

TEST INFRASTRUCTURE ONLY (see the package docstring).

sglang PR 25460 page, key source excerpt of ``fp8_quantize``: each element is
widened to fp32, multiplied by a host-side ``scale_inv`` and cast to fp8
("scale first, then convert to FP8"). sglang PR 30971 page, key source
excerpt of ``_quant_q_fp8``: the stored fp8 value is value/scale, and a
missing scale (``None``) means unit scale with no division at all.

Reading taken where the two pages differ: the multiply-by-inverse form of the
PR 25460 kernel, with the inverse computed once in fp32 on the host
(``1.0f / scale``, IEEE single division). The PR 30971 excerpt divides in the
input dtype; that form double-rounds differently and is not the one built.
"""

from __future__ import annotations

from typing import Optional

import numpy as np

from . import e4m3


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of IEEE half bit patterns (uint16) to float32."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def scale_inverse(scale: Optional[float]) -> np.float32:
    """fp32 inverse of a per-tensor scale; unit when the scale is absent."""
    if scale is None:
        return np.float32(1.0)
    return np.float32(1.0) / np.float32(scale)


def quantize(x_bits: np.ndarray, scale: Optional[float], dtype: str = "bf16") -> np.ndarray:
    """e4m3 codes of ``fp32(x) * scale_inv`` (single fp32 multiply, then RNE)."""
    if dtype == "bf16":
        x = bf16_bits_to_f32(x_bits)
    elif dtype == "fp16":
        x = f16_bits_to_f32(x_bits)
    else:
        raise ValueError(f"unsupported input dtype {dtype!r}")
    v = x * scale_inverse(scale)          # numpy float32 * float32: one IEEE rounding
    return e4m3.encode(v.astype(np.float32))
