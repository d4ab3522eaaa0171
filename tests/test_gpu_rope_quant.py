"""GPU parity of msa_rope_quant_fp8 (fused rotary embedding + e4m3
quantisation of the sparse-MLA q / kv rows) against the oracle: every output
byte, bit for bit."""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import workloads as wl
from oracle import rope_quant as orq
from gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _bits(x, dtype):
    if dtype == "bf16":
        return wl.to_bf16_bits(np.asarray(x, np.float32))
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def _tensor(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


@pytest.mark.parametrize("neox", [True, False])
def test_mla_q_rows_slices_of_one_tensor(msa, neox):
    # q [rows, 128, 576] before rope: nope = q[..., :512], pe = q[..., 512:]
    g = np.random.default_rng(10)
    rows, H, dn, dr = 300, 128, 512, 64
    cs = wl.rotary_table(40000, dr)
    q = _bits(g.standard_normal((rows, H, dn + dr)) * 2, "bf16")
    pos = g.integers(0, 40000, rows).astype(np.int32)
    qt = _tensor(q, "bf16")
    got = msa.rope_quant_fp8(qt[..., :dn], qt[..., dn:], dev(cs), dev(pos), is_neox=neox, scale=0.011)
    msa.check_errors()
    want = orq.rope_quant(q[..., :dn], q[..., dn:], cs, pos, neox, scale=0.011)
    np.testing.assert_array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("neox", [True, False])
def test_kv_rows_one_head_fp16(msa, neox):
    g = np.random.default_rng(11)
    S, dn, dr = 1000, 512, 64
    cs = wl.rotary_table(4096, dr)
    kv_a = _bits(g.standard_normal((S, 1, dn)) * 3, "fp16")
    k_pe = _bits(g.standard_normal((S, 1, dr)) * 3, "fp16")
    pos = np.arange(S, dtype=np.int32) + 17
    got = msa.rope_quant_fp8(_tensor(kv_a, "fp16"), _tensor(k_pe, "fp16"), dev(cs), dev(pos), is_neox=neox)
    msa.check_errors()
    want = orq.rope_quant(kv_a, k_pe, cs, pos, neox, dtype="fp16")
    np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_shared_k_pe_broadcast_to_heads(msa):
    # per-head k_nope [rows, 16, 128] with one shared k_pe [rows, 1, 64]
    g = np.random.default_rng(12)
    rows, H, dn, dr = 777, 16, 128, 64
    cs = wl.rotary_table(2048, dr)
    k_nope = _bits(g.standard_normal((rows, H, dn)), "bf16")
    k_pe = _bits(g.standard_normal((rows, 1, dr)) * 5, "bf16")
    pos = g.integers(0, 2048, rows).astype(np.int32)
    got = msa.rope_quant_fp8(_tensor(k_nope, "bf16"), _tensor(k_pe, "bf16"), dev(cs), dev(pos))
    msa.check_errors()
    np.testing.assert_array_equal(got.cpu().numpy(), orq.rope_quant(k_nope, k_pe, cs, pos, True))


def test_mla_config_full_size_sampled_rows(msa):
    # the full MLA q [4096, 128, 576] at the benchmark's launch shape;
    # rows are independent, so sampled rows are checked against the oracle
    w = wl.make_mla(wl.CONFIGS["mla"])
    T, H, d = w.q.shape
    dn, dr = 512, 64
    cs = wl.rotary_table(w.cfg.S_kv, dr)
    pos = (np.arange(T) + w.cfg.S_kv - T).astype(np.int32)
    qt = _tensor(w.q, "bf16")
    got = msa.rope_quant_fp8(qt[..., :dn], qt[..., dn:], dev(cs), dev(pos), scale=w.scales["q"]).cpu().numpy()
    msa.check_errors()
    rows = np.sort(np.random.default_rng(13).choice(T, 48, replace=False))
    rows = np.concatenate([[0], rows, [T - 1]])
    want = orq.rope_quant(w.q[rows, :, :dn], w.q[rows, :, dn:], cs, pos[rows], True, scale=w.scales["q"])
    np.testing.assert_array_equal(got[rows], want)


def test_bad_position_zeroes_rope_part_and_is_reported(msa):
    g = np.random.default_rng(14)
    rows, H, dn, dr = 40, 4, 64, 32
    cs = wl.rotary_table(100, dr)
    nope = _bits(g.standard_normal((rows, H, dn)), "bf16")
    pe = _bits(g.standard_normal((rows, H, dr)), "bf16")
    pos = g.integers(0, 100, rows).astype(np.int32)
    pos[7] = 100
    got = msa.rope_quant_fp8(_tensor(nope, "bf16"), _tensor(pe, "bf16"), dev(cs), dev(pos)).cpu().numpy()
    with pytest.raises(msa.MsaError) as e:
        msa.check_errors()
    assert e.value.status == 6
    ok = np.ones(rows, bool)
    ok[7] = False
    want = orq.rope_quant(nope[ok], pe[ok], cs, pos[ok], True)
    np.testing.assert_array_equal(got[ok], want)
    assert (got[7, :, dn:] == 0).all()
    np.testing.assert_array_equal(got[7, :, :dn],
                                  orq.rope_quant(nope[7:8], pe[7:8], cs, [0], True)[0, :, :dn])


def test_zero_rows_is_a_no_op(msa):
    cs = dev(wl.rotary_table(4, 32))
    pe = torch.empty((0, 2, 32), dtype=torch.bfloat16, device="cuda")
    out = msa.rope_quant_fp8(None, pe, cs, torch.empty(0, dtype=torch.int32, device="cuda"))
    msa.check_errors()
    assert out.shape == (0, 2, 32)


@pytest.mark.parametrize("cfg", ["prefill8k", "decode"])
def test_indexer_query_rows(msa, cfg):
    # The indexer's e4m3 query produced by the fused producer: idx_q of the
    # workload [T, Hidx, 128] as nope = idx_q[..., :64] || rope(idx_q[..., 64:])
    # at the queries' positions, quantised with idx_q's per-tensor scale (the
    # split of d_idx into 64 + 64 is a reading; the pages fix only that the
    # fused kernel emits the fp8 index query directly)
    w = wl.make_gqa(wl.CONFIGS[cfg])
    T, Hi, d = w.idx_q.shape
    L = int(w.seq_lens.max())
    cs = wl.rotary_table(L, 64)
    pos = np.concatenate([np.arange(int(w.seq_lens[b]) - (int(w.cu_q[b + 1]) - int(w.cu_q[b])),
                                    int(w.seq_lens[b])) for b in range(len(w.seq_lens))]).astype(np.int32)
    iq = _tensor(w.idx_q, "bf16")
    got = msa.rope_quant_fp8(iq[..., :64], iq[..., 64:], dev(cs), dev(pos), is_neox=True,
                             scale=w.scales["idx_q"])
    msa.check_errors()
    rows = np.sort(np.random.default_rng(3).choice(T, size=min(T, 512), replace=False))
    want = orq.rope_quant(w.idx_q[rows, :, :64], w.idx_q[rows, :, 64:], cs, pos[rows], True,
                          scale=w.scales["idx_q"])
    np.testing.assert_array_equal(got.cpu().numpy()[rows], want)
