"""Host logic of the ctypes binding, without a GPU.

A fake library records what each entry point receives, and host tensors
stand in for device tensors, so these tests check the marshalling (sizes,
strides, broadcast, optional parts) and the buffer checks that keep a wrong
shape or a host buffer from reaching a kernel. The last test uses the real
library and real host tensors: every entry point refuses them (there is no
CPU path)."""

import numpy as np
import pytest
import torch

from fp8_block_sparse_gb300 import binding as bd
from fp8_block_sparse_gb300 import workloads as wl


class _FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name.endswith("_workspace_size"):
            return lambda *a: 256
        if name == "msa_last_error_string":
            return lambda: b"fake"

        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    lib = _FakeLib()
    monkeypatch.setattr(bd, "_LIB", lib)
    monkeypatch.setattr(bd, "_on_device", lambda t: True)
    monkeypatch.setattr(bd, "_stream", lambda s, d=None: None)
    return lib


def _batch(B=3, max_pages=5):
    pt = torch.zeros((B, max_pages), dtype=torch.int32)
    return pt, torch.zeros(B, dtype=torch.int32), torch.zeros(B + 1, dtype=torch.int32)


def _u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def test_index_topk_marshalling_and_checks(fake):
    pt, sl, cu = _batch()
    iq, ik = _u8(10, 4, 128), _u8(7, 128, 128)
    out = bd.index_topk(iq, ik, pt, sl, cu, 16, 10)
    assert tuple(out.shape) == (4, 10, 16)
    name, a = fake.calls[-1]
    assert name == "msa_index_topk" and a[5:13] == (3, 10, 10, 4, 128, 16, 7, 5)
    with pytest.raises(bd.MsaError):                      # cu_q must have B + 1 entries
        bd.index_topk(iq, ik, pt, sl, cu[:3], 16, 10)
    with pytest.raises(bd.MsaError):                      # out of the wrong shape
        bd.index_topk(iq, ik, pt, sl, cu, 16, 10, out=torch.zeros((4, 10, 8), dtype=torch.int32))
    with pytest.raises(bd.MsaError):                      # index-K cache with a head axis
        bd.index_topk(iq, _u8(7, 2, 128, 128), pt, sl, cu, 16, 10)
    bd.index_topk_noalloc(iq, ik, pt, sl, cu, 16, 10)
    assert fake.calls[-1][0] == "msa_index_topk_noalloc"


def test_attention_buffers_are_checked(fake):
    pt, sl, cu = _batch()
    T, Hq, Hkv, Hidx, D, topk = 12, 16, 2, 4, 128, 8
    q, kc = _u8(T, Hq, D), _u8(9, Hkv, 128, D)
    ids = torch.zeros((Hidx, T, topk), dtype=torch.int32)
    sink = torch.zeros(Hq)
    o, ml, lse = bd.sparse_attn_fwd(q, kc, kc.clone(), pt, sl, cu, ids, sink, 0.1, None, 2.0, None, T)
    assert o.dtype == torch.bfloat16 and tuple(o.shape) == (T, Hq, D) and tuple(lse.shape) == (T, Hq)
    a = fake.calls[-1][1]
    assert a[12:22] == (3, T, T, Hq, Hkv, Hidx, D, topk, 9, 5)
    bad = [dict(out=torch.zeros((T, Hq, D - 1), dtype=torch.bfloat16)),
           dict(max_logit=torch.zeros((T, Hq), dtype=torch.float64)),
           dict(lse=torch.zeros((T - 1, Hq))),
           dict(workspace=torch.zeros(64, dtype=torch.int32))]
    for kw in bad:
        with pytest.raises(bd.MsaError):
            bd.sparse_attn_fwd(q, kc, kc.clone(), pt, sl, cu, ids, sink, 0.1, None, None, None, T, **kw)
    with pytest.raises(bd.MsaError):                      # sink must have Hq entries
        bd.sparse_attn_fwd(q, kc, kc.clone(), pt, sl, cu, ids, torch.zeros(Hq - 1), 0.1, None, None, None, T)
    with pytest.raises(bd.MsaError):                      # V pool unlike the K pool
        bd.sparse_attn_fwd(q, kc, _u8(8, Hkv, 128, D), pt, sl, cu, ids, sink, 0.1, None, None, None, T)
    with pytest.raises(bd.MsaError):                      # top-k rows for another T
        bd.sparse_attn_fwd(q, kc, kc.clone(), pt, sl, cu, ids[:, :5], sink, 0.1, None, None, None, T)


def test_mla_buffers_are_checked(fake):
    T, H, S, topk = 6, 128, 300, 64
    q, kv = _u8(T, H, 576), _u8(S, 576)
    idx = torch.zeros((T, topk), dtype=torch.int32)
    o, ml, lse = bd.sparse_mla_fwd(q, kv, idx, None, torch.zeros(H), 0.04, None, None)
    assert tuple(o.shape) == (T, H, 512)
    assert fake.calls[-1][1][8:14] == (T, H, S, 576, 512, topk)
    with pytest.raises(bd.MsaError):
        bd.sparse_mla_fwd(q, kv, idx, torch.zeros(T - 1, dtype=torch.int32), None, 0.04, None, None)
    with pytest.raises(bd.MsaError):
        bd.sparse_mla_fwd(q, kv, idx, None, None, 0.04, None, None, out=torch.zeros((T, H, 576), dtype=torch.bfloat16))
    with pytest.raises(bd.MsaError):
        bd.sparse_mla_fwd(q, _u8(S, 512), idx, None, None, 0.04, None, None)


def test_quant_out_must_match(fake):
    x = torch.zeros((5, 3, 64), dtype=torch.bfloat16)
    out = bd.quant_fp8(x, 0.5)
    assert tuple(out.shape) == (5, 3, 64)
    name, a = fake.calls[-1]
    assert a[2:5] == (15, 64, 64)
    with pytest.raises(bd.MsaError):
        bd.quant_fp8(x, None, out=_u8(5, 3, 63))
    # a strided view of wider rows: rows keep their stride
    big = torch.zeros((20, 96), dtype=torch.bfloat16)
    bd.quant_fp8(big[:, :64], None, out=_u8(20, 64))
    assert fake.calls[-1][1][2:5] == (20, 64, 96)


def test_kv_store_marshalling(fake):
    pt, sl, cu = _batch()
    T, Hq, Hkv, D, di = 7, 16, 2, 128, 128
    fused = torch.zeros((T, Hq * D + 2 * Hkv * D + di), dtype=torch.bfloat16)
    k = fused[:, Hq * D:Hq * D + Hkv * D].view(T, Hkv, D)
    v = fused[:, Hq * D + Hkv * D:Hq * D + 2 * Hkv * D].view(T, Hkv, D)
    ik = fused[:, Hq * D + 2 * Hkv * D:]
    kc, vc, ic = _u8(11, Hkv, 128, D), _u8(11, Hkv, 128, D), _u8(11, 128, di)
    bd.kv_store_fp8(pt, sl, cu, kc, vc, ic, k=k, v=v, idx_k=ik, k_scale=0.5)
    a = fake.calls[-1][1]
    row = fused.shape[1]
    assert a[3] == bd.MSA_BF16 and a[4:7] == (row, row, row)
    assert a[10:17] == (3, T, 5, 11, Hkv, D, di)
    # index K only: the K / V caches are not needed, Hkv and D are unused
    bd.kv_store_fp8(pt, sl, cu, None, None, ic, idx_k=ik)
    a = fake.calls[-1][1]
    assert a[0] is None and a[1] is None and a[14:17] == (0, 16, di)
    with pytest.raises(bd.MsaError):                      # cache for another head count
        bd.kv_store_fp8(pt, sl, cu, _u8(11, 1, 128, D), vc, ic, k=k, v=v)
    with pytest.raises(bd.MsaError):                      # input given without its cache
        bd.kv_store_fp8(pt, sl, cu, None, vc, ic, k=k, v=v)
    with pytest.raises(bd.MsaError):                      # heads not contiguous within a token
        bd.kv_store_fp8(pt, sl, cu, kc, None, None, k=fused[:, :Hkv * D * 2:2].view(T, Hkv, D))
    with pytest.raises(bd.MsaError):                      # mixed dtypes
        bd.kv_store_fp8(pt, sl, cu, kc, vc, None, k=k, v=v.to(torch.float16))
    with pytest.raises(bd.MsaError):                      # index K for fewer tokens
        bd.kv_store_fp8(pt, sl, cu, kc, vc, ic, k=k, v=v, idx_k=ik[:T - 1])
    with pytest.raises(bd.MsaError):                      # V with another head count
        bd.kv_store_fp8(pt, sl, cu, kc, vc, None, k=k, v=v[:, :1])


def test_rope_quant_marshalling(fake):
    rows, H, dn, dr = 9, 4, 512, 64
    q = torch.zeros((rows, H, dn + dr), dtype=torch.bfloat16)
    cs = torch.zeros((100, dr))
    pos = torch.zeros(rows, dtype=torch.int32)
    out = bd.rope_quant_fp8(q[..., :dn], q[..., dn:], cs, pos)
    assert tuple(out.shape) == (rows, H, dn + dr)
    a = fake.calls[-1][1]
    assert a[3:11] == (rows, H, dn, dr, H * (dn + dr), dn + dr, H * (dn + dr), dn + dr)
    assert a[12] == 100 and a[14] == 1
    # one shared pe row for every head: head stride 0
    bd.rope_quant_fp8(q[..., :dn], torch.zeros((rows, 1, dr), dtype=torch.bfloat16), cs, pos, is_neox=False)
    a = fake.calls[-1][1]
    assert a[9:11] == (dr, 0) and a[14] == 0
    with pytest.raises(bd.MsaError):                      # table for another rope width
        bd.rope_quant_fp8(q[..., :dn], q[..., dn:], torch.zeros((100, 32)), pos)
    with pytest.raises(bd.MsaError):                      # pe with 2 of 4 heads
        bd.rope_quant_fp8(q[..., :dn], torch.zeros((rows, 2, dr), dtype=torch.bfloat16), cs, pos)
    with pytest.raises(bd.MsaError):
        bd.rope_quant_fp8(q[..., :dn], q[..., dn:], cs, pos, out=_u8(rows, H, dn))


def test_host_tensors_are_refused_by_the_real_library():
    from fp8_block_sparse_gb300 import build as b
    b.build()
    lib = bd.load()
    assert lib is not None
    w = wl.make_gqa(wl.CONFIGS["tiny"], T_override=130)
    pt, sl, cu = (torch.from_numpy(np.ascontiguousarray(a)) for a in (w.page_table, w.seq_lens, w.cu_q))
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    calls = [
        lambda: bd.quant_fp8(x, None),
        lambda: bd.index_topk(_u8(130, 1, 64), _u8(w.num_pages, 128, 64), pt, sl, cu, 8, 130),
        lambda: bd.sparse_attn_fwd(_u8(130, 8, 128), _u8(w.num_pages, 1, 128, 128), _u8(w.num_pages, 1, 128, 128),
                                   pt, sl, cu, torch.zeros((1, 130, 8), dtype=torch.int32), None, 0.1,
                                   None, None, None, 130),
        lambda: bd.sparse_mla_fwd(_u8(2, 128, 576), _u8(10, 576), torch.zeros((2, 4), dtype=torch.int32),
                                  None, None, 0.04, None, None),
        lambda: bd.kv_store_fp8(pt, sl, cu, None, None, _u8(w.num_pages, 128, 64),
                                idx_k=torch.zeros((130, 64), dtype=torch.bfloat16)),
        lambda: bd.rope_quant_fp8(None, torch.zeros((3, 1, 32), dtype=torch.bfloat16), torch.zeros((4, 32)),
                                  torch.zeros(3, dtype=torch.int32)),
    ]
    for c in calls:
        with pytest.raises(bd.MsaError) as e:
            c()
        assert e.value.status == 1


def test_tensors_on_two_devices_are_refused(fake):
    # the library launches on one device: a call mixing devices would hand it
    # another device's pointers, so the binding refuses it before the call
    pt, sl, cu = _batch()
    iq = torch.zeros((10, 4, 128), dtype=torch.uint8, device="meta")
    ik = _u8(7, 128, 128)
    n = len(fake.calls)
    with pytest.raises(bd.MsaError, match="one device"):
        bd.index_topk(iq, ik, pt, sl, cu, 16, 10)
    with pytest.raises(bd.MsaError, match="one device"):
        bd.index_topk_noalloc(iq, ik, pt, sl, cu, 16, 10)
    q = torch.zeros((12, 16, 128), dtype=torch.uint8, device="meta")
    kc = _u8(9, 2, 128, 128)
    ids = torch.zeros((4, 12, 8), dtype=torch.int32)
    with pytest.raises(bd.MsaError, match="one device"):
        bd.sparse_attn_fwd(q, kc, kc.clone(), pt, sl, cu, ids, None, 0.1, None, None, None, 12)
    assert len(fake.calls) == n


def test_quant_multi_marshalling(fake, monkeypatch):
    import ctypes
    seen = {}

    def capture(addr, n, x_dtype, out_dtype, stream):      # read the descriptors during the call
        d = (bd._QuantTensor * n).from_address(addr)
        seen["d"] = [(t.x, t.rows, t.cols, t.x_row_stride, t.out, t.out_row_stride,
                      None if t.scale is None else ctypes.c_float.from_address(t.scale).value)
                     for t in d]
        seen["n"], seen["dtype"] = n, x_dtype
        return 0
    monkeypatch.setattr(fake, "msa_quant_fp8_multi", capture, raising=False)
    x = torch.zeros((6, 4, 32), dtype=torch.bfloat16)
    y = torch.zeros((5, 64), dtype=torch.bfloat16)[:, :32]         # row-strided view
    oy = torch.zeros((5, 32), dtype=torch.uint8)
    outs = bd.quant_fp8_multi([(x, 0.25), (y, None, oy)])
    assert outs[1] is oy and tuple(outs[0].shape) == (6, 4, 32)
    assert seen["n"] == 2 and seen["dtype"] == bd.MSA_BF16
    assert seen["d"][0] == (x.data_ptr(), 24, 32, 32, outs[0].data_ptr(), 32, 0.25)
    assert seen["d"][1] == (y.data_ptr(), 5, 32, 64, oy.data_ptr(), 32, None)
    with pytest.raises(bd.MsaError):                                # mixed dtypes
        bd.quant_fp8_multi([(x, 1.0), (y.to(torch.float16), 1.0)])
