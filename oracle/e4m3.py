"""OCP FP8 E4M3 codec ("fn" variant: no infinities), from the bit definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages store every fp8 tensor as ``torch.float8_e4m3fn`` (sglang PR 30971
page, implementation step 3: q/idx_q are cast to fp8_e4m3; vLLM PR 45892 page,
step 3: the index cache is stored as float8_e4m3fn). The format itself is the
OCP 8-bit floating point E4M3 encoding:

* bit 7 sign, bits 6..3 biased exponent E (bias 7), bits 2..0 mantissa M;
* E == 0: subnormal, value = M * 2**-9;
* otherwise value = (1 + M/8) * 2**(E-7);
* E == 15 and M == 7 is NaN; there is no infinity, so the largest finite
  magnitude is (1 + 6/8) * 2**8 = 448 (code 0x7E).

Encoding rounds to nearest, ties to even mantissa. Overflow saturates to
+-448 ("satfinite"): the pages never say what happens above 448, and the
saturating reading is the one under which every finite fp32 input has a
finite code. For |v| <= 464 (the rounding midpoint between 448 and the
absent 480) saturation and plain round-to-nearest agree.
"""

from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
MIN_NORMAL = 2.0 ** -6
SUBNORMAL_STEP = 2.0 ** -9


def decode_table() -> np.ndarray:
    """Float64 value of each of the 256 codes (NaN for 0x7F and 0xFF)."""
    codes = np.arange(256, dtype=np.int64)
    sign = codes >> 7
    exp_field = (codes >> 3) & 0xF
    man_field = codes & 0x7
    magnitude = np.where(
        exp_field == 0,
        man_field * SUBNORMAL_STEP,
        (1.0 + man_field / 8.0) * np.exp2(exp_field - 7.0),
    )
    values = np.where(sign == 1, -magnitude, magnitude)
    values[(exp_field == 15) & (man_field == 7)] = np.nan
    return values


_TABLE = decode_table()


def decode(codes: np.ndarray) -> np.ndarray:
    """Map uint8 codes to their float64 values."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(values: np.ndarray) -> np.ndarray:
    """Round float32 values to e4m3 codes (RNE, satfinite, sign of zero kept)."""
    v = np.asarray(values, dtype=np.float32).astype(np.float64)  # exact widening
    negative = np.signbit(v)
    a = np.abs(v)
    out = np.zeros(v.shape, dtype=np.uint8)

    is_nan = np.isnan(v)
    saturate = ~is_nan & (a >= MAX_FINITE)
    subnormal = ~is_nan & (a < MIN_NORMAL)
    normal = ~is_nan & ~saturate & ~subnormal

    # Subnormal range: the grid is k * 2**-9, k = 0..8; k == 8 is the smallest
    # normal (code 0x08), so the code is k itself. rint rounds half to even.
    out[subnormal] = np.rint(a[subnormal] / SUBNORMAL_STEP).astype(np.uint8)

    # Normal range: a = f * 2**e with f in [1, 2); keep 3 fraction bits.
    frac, exp2 = np.frexp(a[normal])          # a = frac * 2**exp2, frac in [0.5, 1)
    e = exp2.astype(np.int64) - 1
    q = np.rint((2.0 * frac - 1.0) * 8.0).astype(np.int64)   # 0..8, exact product
    carry = q == 8
    e = e + carry
    q = np.where(carry, 0, q)
    out[normal] = (((e + 7) << 3) | q).astype(np.uint8)

    out[saturate] = 0x7E
    out[is_nan] = 0x7F
    out |= (negative.astype(np.uint8) << 7)
    return out
