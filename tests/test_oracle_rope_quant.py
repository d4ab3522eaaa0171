"""Pins for the oracle's fused rotary embedding + e4m3 quantiser (the MLA
q / kv producer): hand-worked rotations whose results are e4m3-exact, with
their bytes written out by bit fields; the identity at angle zero; a
complex-number restatement of the rotation; the relative-position property;
the neox / neighbour-pair layouts related by a permutation; torch's own fp32
arithmetic and fp8 cast; broadcast of a shared k_pe."""

import numpy as np
import pytest
import torch

from oracle import quant, rope_quant as orq
from fp8_block_sparse_gb300 import workloads as wl


def _bf16(x):
    return wl.to_bf16_bits(np.asarray(x, np.float32))


def test_hand_worked_rotation_bytes():
    # d_rope = 4, one position whose cos/sin row is (c0, c1, s0, s1) = (.5, .25, .75, 1)
    cs = np.array([[0.5, 0.25, 0.75, 1.0]], np.float32)
    pe = _bf16(np.array([[[1.0, 2.0, 3.0, 4.0]]]))
    nope = _bf16(np.zeros((1, 1, 16)))
    pos = np.zeros(1, np.int32)
    # neox: halves (1, 2), (3, 4): (1*.5-3*.75, 2*.25-4*1, 3*.5+1*.75, 4*.25+2*1)
    #   = (-1.75, -3.5, 2.25, 3.0) -> 1 0111 110, 1 1000 110, 0 1000 001, 0 1000 100
    out = orq.rope_quant(nope, pe, cs, pos, True)
    assert out[0, 0, 16:].tolist() == [0xBE, 0xC6, 0x41, 0x44]
    # neighbour pairs (1, 2) at angle 0, (3, 4) at angle 1:
    #   (1*.5-2*.75, 2*.5+1*.75, 3*.25-4*1, 4*.25+3*1) = (-1, 1.75, -3.25, 4)
    #   -> 1 0111 000, 0 0111 110, 1 1000 101, 0 1001 000
    out = orq.rope_quant(nope, pe, cs, pos, False)
    assert out[0, 0, 16:].tolist() == [0xB8, 0x3E, 0xC5, 0x48]
    assert (out[0, 0, :16] == 0).all()


@pytest.mark.parametrize("neox", [True, False])
def test_position_zero_is_plain_quantisation(neox):
    g = np.random.default_rng(1)
    cs = wl.rotary_table(8, 64)
    nope = _bf16(g.standard_normal((5, 3, 32)) * 4)
    pe = _bf16(g.standard_normal((5, 3, 64)) * 4)
    out = orq.rope_quant(nope, pe, cs, np.zeros(5, np.int32), neox, scale=0.05)
    want = quant.quantize(np.concatenate([nope, pe], axis=-1), 0.05)
    np.testing.assert_array_equal(out, want)


def test_rotation_matches_complex_multiplication():
    g = np.random.default_rng(2)
    cs = wl.rotary_table(4096, 64)
    pe = g.standard_normal((300, 4, 64)).astype(np.float32)
    pos = g.integers(0, 4096, 300)
    got = orq.rope(pe, cs, pos, True)
    z = pe[..., :32].astype(np.float64) + 1j * pe[..., 32:].astype(np.float64)
    w = cs[pos, :32].astype(np.float64) + 1j * cs[pos, 32:].astype(np.float64)
    r = z * w[:, None, :]
    want = np.concatenate([r.real, r.imag], axis=-1)
    # two fp32 products and one fp32 sum: within 3 ulp-scale roundings of |x|
    bound = 4 * 2.0 ** -24 * (np.abs(pe[..., :32]) + np.abs(pe[..., 32:]))
    err = np.abs(got - want)
    assert (err[..., :32] <= bound).all() and (err[..., 32:] <= bound).all()


def test_relative_position_property():
    g = np.random.default_rng(3)
    cs = wl.rotary_table(2048, 64)
    q = g.standard_normal((1, 1, 64)).astype(np.float32)
    k = g.standard_normal((1, 1, 64)).astype(np.float32)
    for m, n, d in ((5, 2, 100), (700, 13, 900), (0, 0, 1000)):
        a = float(np.dot(orq.rope(q, cs, [m], True).ravel(), orq.rope(k, cs, [n], True).ravel()))
        b = float(np.dot(orq.rope(q, cs, [m + d], True).ravel(), orq.rope(k, cs, [n + d], True).ravel()))
        assert abs(a - b) < 1e-4 * (1 + abs(a))


def test_neighbour_pairs_are_neox_halves_permuted():
    g = np.random.default_rng(4)
    cs = wl.rotary_table(512, 32)
    pe = g.standard_normal((40, 2, 32)).astype(np.float32)
    pos = g.integers(0, 512, 40)
    perm = np.concatenate([np.arange(0, 32, 2), np.arange(1, 32, 2)])   # evens then odds
    inter = orq.rope(pe, cs, pos, False)
    neox = orq.rope(pe[..., perm], cs, pos, True)
    np.testing.assert_array_equal(inter[..., perm], neox)


def test_torch_fp32_arithmetic_and_fp8_cast():
    g = np.random.default_rng(5)
    cs = wl.rotary_table(1024, 64)
    nope = _bf16(g.standard_normal((64, 8, 128)) * 3)
    pe = _bf16(g.standard_normal((64, 8, 64)) * 3)
    pos = g.integers(0, 1024, 64)
    scale = 0.03
    out = orq.rope_quant(nope, pe, cs, pos, True, scale=scale)
    tb = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float()
    x1, x2 = tb(pe)[..., :32], tb(pe)[..., 32:]
    c = torch.from_numpy(cs[pos, :32])[:, None, :]
    s = torch.from_numpy(cs[pos, 32:])[:, None, :]
    rot = torch.cat([torch.mul(x1, c) - torch.mul(x2, s), torch.mul(x2, c) + torch.mul(x1, s)], -1)
    s_inv = torch.tensor(1.0) / torch.tensor(scale)
    full = torch.cat([tb(nope), rot], -1) * s_inv
    assert float(full.abs().max()) < 448           # inside torch's non-NaN range
    want = full.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(out, want)


def test_shared_pe_is_broadcast_to_every_head():
    g = np.random.default_rng(6)
    cs = wl.rotary_table(256, 64)
    nope = _bf16(g.standard_normal((10, 4, 64)))
    pe1 = _bf16(g.standard_normal((10, 1, 64)))
    pos = g.integers(0, 256, 10)
    a = orq.rope_quant(nope, pe1, cs, pos, True)
    b = orq.rope_quant(nope, np.repeat(pe1, 4, axis=1), cs, pos, True)
    np.testing.assert_array_equal(a, b)


def test_missing_scale_is_unit_and_power_of_two_scale_is_exact():
    g = np.random.default_rng(7)
    cs = wl.rotary_table(64, 32)
    nope = _bf16(g.uniform(0.5, 8, (6, 2, 16)))
    pe = _bf16(g.uniform(0.5, 8, (6, 2, 32)))
    pos = g.integers(0, 64, 6)
    a = orq.rope_quant(nope, pe, cs, pos, False)
    np.testing.assert_array_equal(a, orq.rope_quant(nope, pe, cs, pos, False, scale=1.0))
    from oracle import e4m3
    half = orq.rope_quant(nope, pe, cs, pos, False, scale=2.0)
    # dividing by 2 moves every normal e4m3 value one binade down, exactly
    big = np.abs(e4m3.decode(a)) >= 2.0 ** -5
    np.testing.assert_array_equal(e4m3.decode(half)[big], e4m3.decode(a)[big] / 2)
