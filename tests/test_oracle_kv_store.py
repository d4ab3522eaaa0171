"""Pins for the oracle's quantised KV-cache store (the step before the path).

Each check fixes the store by something other than the oracle itself: slot
coordinates worked out by hand from the position rule, byte codes of
e4m3-exact values written out by their bit fields, torch's own fp8 cast, and
invariants (untouched slots keep their bytes; a full sequence stored through
a permuted page table reads back in logical order)."""

import numpy as np
import pytest
import torch

from oracle import kv_store as okv
from fp8_block_sparse_gb300 import workloads as wl

SENTINEL = 0x7F        # e4m3 NaN code: a saturating cast of finite data never writes it


def _bf16(x):
    return wl.to_bf16_bits(np.asarray(x, np.float32))


def _torch_codes(bits, scale):
    """torch's fp8 cast of fp32(x) * fp32(1/scale): an independent codec."""
    xf = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float()
    s_inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(1.0 if scale is None else scale,
                                                                  dtype=torch.float32)
    return (xf * s_inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _caches(num_pages, Hkv, D, d_idx):
    k = np.full((num_pages, Hkv, 128, D), SENTINEL, np.uint8)
    return k, k.copy(), np.full((num_pages, 128, d_idx), SENTINEL, np.uint8)


def test_worked_example_slots_and_codes():
    # one sequence of 130 tokens whose last 3 are new: positions 127, 128, 129
    # -> (page_table[0], slot 127), (page_table[1], slot 0), (page_table[1], slot 1)
    pt = np.array([[5, 2, -1]], np.int32)
    sl = np.array([130], np.int32)
    cu = np.array([0, 3], np.int32)
    pages, slots = okv.slot_addresses(pt, sl, cu)
    assert pages.tolist() == [5, 2, 2] and slots.tolist() == [127, 0, 1]
    # e4m3 bytes by bit field (sign | 4-bit exponent, bias 7 | 3-bit mantissa):
    # 1.5 = 0 0111 100 = 0x3C, -2 = 1 1000 000 = 0xC0, 448 = 0 1111 110 = 0x7E,
    # 0.015625 = 2^-6 = 0 0001 000 = 0x08, 2^-9 (subnormal 1/8 * 2^-6) = 0x01
    vals = np.array([1.5, -2.0, 448.0, 0.015625, 2.0 ** -9, 0.0, -0.0, 1000.0])
    want = np.array([0x3C, 0xC0, 0x7E, 0x08, 0x01, 0x00, 0x80, 0x7E], np.uint8)   # 1000 saturates
    x = np.stack([np.roll(vals, t) for t in range(3)])              # [T=3, 8]
    k = _bf16(x.reshape(3, 1, 8))
    kc, vc, ic = _caches(8, 1, 8, 8)
    kc2, vc2, ic2 = okv.kv_store(pt, sl, cu, kc, vc, ic, k=k, v=None, idx_k=_bf16(-x))
    for t, (p, s) in enumerate(zip([5, 2, 2], [127, 0, 1])):
        assert kc2[p, 0, s].tolist() == np.roll(want, t).tolist()
        neg = np.roll(want, t) ^ 0x80
        assert ic2[p, s].tolist() == neg.tolist()
    assert np.array_equal(vc2, vc)                                   # v not given: untouched
    changed = np.argwhere((kc2 != SENTINEL).any(axis=-1))
    assert sorted(map(tuple, changed.tolist())) == [(2, 0, 0), (2, 0, 1), (5, 0, 127)]


def test_prefix_continuation_positions():
    # 300 cached tokens, the last 45 new: positions 255..299 = page 1 slot 127,
    # then page 2 slots 0..43
    pt = np.array([[9, 4, 7, 0]], np.int32)
    pages, slots = okv.slot_addresses(pt, np.array([300], np.int32), np.array([0, 45], np.int32))
    assert pages.tolist() == [4] + [7] * 44
    assert slots.tolist() == [127] + list(range(44))


def test_full_sequence_reads_back_in_logical_order():
    g = np.random.default_rng(3)
    L, Hkv, D, di = 128 * 5 - 37, 2, 32, 16
    perm = g.permutation(7)[:5].astype(np.int32)
    pt = perm[None, :]
    x = _bf16(g.standard_normal((L, Hkv, D)).astype(np.float32) * 3)
    xi = _bf16(g.standard_normal((L, di)).astype(np.float32) * 3)
    kc, vc, ic = _caches(7, Hkv, D, di)
    scale = 0.0371
    kc2, vc2, ic2 = okv.kv_store(pt, np.array([L], np.int32), np.array([0, L], np.int32), kc, vc, ic,
                                 k=x, v=x, idx_k=xi, k_scale=scale, v_scale=None, idx_k_scale=2.5)
    # logical order: position p lives at page pt[p // 128], slot p % 128
    logical_k = kc2[perm].transpose(0, 2, 1, 3).reshape(-1, Hkv, D)[:L]
    logical_v = vc2[perm].transpose(0, 2, 1, 3).reshape(-1, Hkv, D)[:L]
    logical_i = ic2[perm].reshape(-1, di)[:L]
    np.testing.assert_array_equal(logical_k, _torch_codes(x, scale))
    np.testing.assert_array_equal(logical_v, _torch_codes(x, None))
    np.testing.assert_array_equal(logical_i, _torch_codes(xi, 2.5))
    # the tail of the last page and the pages outside the table keep their bytes
    assert (kc2[perm[-1], :, 128 - 37:] == SENTINEL).all()
    unused = np.setdiff1d(np.arange(7), perm)
    assert (kc2[unused] == SENTINEL).all() and (ic2[unused] == SENTINEL).all()


def test_varlen_decode_batch_touches_one_slot_per_sequence():
    g = np.random.default_rng(4)
    B, Hkv, D = 6, 2, 16
    sl = np.array([1, 128, 129, 700, 256, 5], np.int32)
    pt = g.permutation(40)[:B * 6].reshape(B, 6).astype(np.int32)
    cu = np.arange(B + 1, dtype=np.int32)
    x = _bf16(g.standard_normal((B, Hkv, D)).astype(np.float32))
    kc, vc, ic = _caches(40, Hkv, D, 16)
    kc2, _, _ = okv.kv_store(pt, sl, cu, kc, None, None, k=x)
    for b in range(B):
        p = int(sl[b]) - 1
        np.testing.assert_array_equal(kc2[pt[b, p // 128], :, p % 128], _torch_codes(x[b], None))
    assert int((kc2 != SENTINEL).any(axis=-1).sum()) == B * Hkv


@pytest.mark.parametrize("scale", [0.125, 4.0])
def test_power_of_two_scale_equals_division_in_bf16(scale):
    # the pool's own non-unit form divides in the input dtype before the cast;
    # for a power-of-two scale the division is exact, so both forms agree
    g = np.random.default_rng(5)
    x = _bf16(g.standard_normal((50, 1, 64)).astype(np.float32) * 6)   # |x / scale| < 448
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    pool_form = (xt / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    pt = np.arange(1, dtype=np.int32)[None, :]
    kc, _, _ = _caches(1, 1, 64, 16)
    kc2, _, _ = okv.kv_store(pt, np.array([50], np.int32), np.array([0, 50], np.int32), kc, None, None,
                             k=x, k_scale=scale)
    np.testing.assert_array_equal(kc2[0, 0, :50], pool_form[:, 0])


def test_missing_scale_is_unit_scale():
    g = np.random.default_rng(6)
    x = _bf16(g.standard_normal((20, 1, 32)).astype(np.float32))
    args = (np.zeros((1, 1), np.int32), np.array([20], np.int32), np.array([0, 20], np.int32))
    kc, _, _ = _caches(1, 1, 32, 16)
    a = okv.kv_store(*args, kc, None, None, k=x, k_scale=None)[0]
    b = okv.kv_store(*args, kc, None, None, k=x, k_scale=1.0)[0]
    np.testing.assert_array_equal(a, b)


def test_bad_page_and_missing_entry_are_errors():
    kc, _, _ = _caches(4, 1, 16, 16)
    x = _bf16(np.ones((1, 1, 16), np.float32))
    with pytest.raises(ValueError):
        okv.kv_store(np.array([[4]], np.int32), np.array([1], np.int32), np.array([0, 1], np.int32),
                     kc, None, None, k=x)
    with pytest.raises(ValueError):        # position 128 needs a second page-table entry
        okv.kv_store(np.array([[0]], np.int32), np.array([129], np.int32), np.array([0, 1], np.int32),
                     kc, None, None, k=x)
