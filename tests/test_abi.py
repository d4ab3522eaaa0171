"""Host-side checks of libmsa.so that need no GPU: every symbol include/msa.h
declares is exported, and argument validation rejects bad calls before any
CUDA work (these calls return before touching the device)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp8_block_sparse_gb300 import build as b
    b.build()
    from fp8_block_sparse_gb300 import binding
    return binding.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "msa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_path_entry_points():
    names = declared_symbols()
    for n in ("msa_quant_fp8", "msa_index_topk", "msa_sparse_attn_fwd", "msa_sparse_mla_fwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (msa_\w+)", out))
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing
    for n in declared_symbols():
        getattr(lib, n)


def test_version_and_error_string(lib):
    assert lib.msa_version() >= 100
    assert isinstance(lib.msa_last_error_string(), bytes)


def _f(x):
    return ctypes.pointer(ctypes.c_float(x))


def test_quant_rejects_e5m2_and_bad_arguments(lib):
    dummy = ctypes.c_void_p(16)
    # e5m2 output never enters the path
    assert lib.msa_quant_fp8(dummy, 0, 4, 16, 16, dummy, 3, 16, None, None) == 2
    assert b"e5m2" in lib.msa_last_error_string()
    assert lib.msa_quant_fp8(dummy, 2, 4, 16, 16, dummy, 2, 16, None, None) == 1    # e4m3 input
    assert lib.msa_quant_fp8(dummy, 0, -1, 16, 16, dummy, 2, 16, None, None) == 1   # negative rows
    assert lib.msa_quant_fp8(dummy, 0, 4, 16, 8, dummy, 2, 16, None, None) == 1     # stride < cols
    assert lib.msa_quant_fp8(None, 0, 4, 16, 16, dummy, 2, 16, None, None) == 1     # null x
    assert lib.msa_quant_fp8(dummy, 0, 4, 16, 16, dummy, 2, 16, _f(0.0), None) == 1  # zero scale
    assert lib.msa_quant_fp8(dummy, 0, 4, 16, 16, dummy, 2, 16, _f(float("nan")), None) == 1
    assert lib.msa_quant_fp8(None, 0, 0, 16, 16, None, 2, 16, None, None) == 0      # empty: no-op


def test_index_topk_validation(lib):
    p = ctypes.c_void_p(256)
    # D unsupported, topk out of range, max_q_len out of range
    assert lib.msa_index_topk(p, p, p, p, p, 1, 128, 128, 1, 96, 8, 1, 1, p, p, 1 << 20, None) == 2
    assert lib.msa_index_topk(p, p, p, p, p, 1, 128, 128, 1, 64, 65, 1, 1, p, p, 1 << 20, None) == 2
    assert lib.msa_index_topk(p, p, p, p, p, 1, 128, 129, 1, 64, 8, 1, 1, p, p, 1 << 20, None) == 1
    assert lib.msa_index_topk(p, p, p, p, p, 1, 0, 1, 1, 64, 8, 1, 1, p, p, 0, None) == 0   # T = 0
    need = lib.msa_index_topk_workspace_size(4096, 4, 32)
    if need:
        assert lib.msa_index_topk(p, p, p, p, p, 1, 4096, 4096, 4, 64, 8, 32, 32, p, p, need - 1, None) == 5


def test_attention_validation(lib):
    p = ctypes.c_void_p(256)
    args = lambda hq, hkv, hidx, d, topk, sm=0.1: (p, p, p, p, p, p, p, None, sm, None, None, None,
                                                    1, 256, 256, hq, hkv, hidx, d, topk, 2, 2,
                                                    p, p, p, p, 1 << 30, None)
    assert lib.msa_sparse_attn_fwd(*args(16, 2, 4, 64, 16)) == 2       # head_dim 64
    assert lib.msa_sparse_attn_fwd(*args(16, 3, 4, 128, 16)) == 1      # Hq % Hkv
    assert lib.msa_sparse_attn_fwd(*args(12, 1, 4, 128, 16)) == 2      # group 12 not a power of 2
    assert lib.msa_sparse_attn_fwd(*args(16, 2, 4, 128, 65)) == 2      # topk > 64
    assert lib.msa_sparse_attn_fwd(*args(16, 2, 4, 128, 16, -1.0)) == 1
    a = list(args(16, 2, 4, 128, 16))
    a[10] = _f(-2.0)                                                   # negative k_scale
    assert lib.msa_sparse_attn_fwd(*a) == 1


def test_mla_validation(lib):
    p = ctypes.c_void_p(256)
    f = lambda dqk, dv, h, topk: lib.msa_sparse_mla_fwd(p, p, p, None, None, 0.04, None, None,
                                                         16, h, 1024, dqk, dv, topk, p, p, p, None)
    assert f(576, 256, 128, 2048) == 2          # d_v must be 512
    assert f(512, 512, 128, 2048) == 2          # d_qk must be 576
    assert f(576, 512, 64, 2048) == 2           # 128 heads


def test_empty_batches_return_ok_without_touching_pointers(lib):
    # T = 0: scalar checks only, no pointer is read and no CUDA work is issued
    null = None
    assert lib.msa_index_topk(null, null, null, null, null, 1, 0, 0, 4, 128, 64, 1, 1,
                              null, null, 0, null) == 0
    assert lib.msa_sparse_attn_fwd(null, null, null, null, null, null, null, null, 0.1, None, None, None,
                                   1, 0, 0, 16, 2, 4, 128, 64, 1, 1, null, null, null, null, 0, null) == 0
    assert lib.msa_sparse_mla_fwd(null, null, null, null, null, 0.1, None, None, 0, 128, 64, 576, 512, 2048,
                                  null, null, null, null) == 0
    # bad scalars are still rejected when T = 0
    assert lib.msa_index_topk(null, null, null, null, null, 1, 0, 0, 4, 96, 64, 1, 1,
                              null, null, 0, null) == 2                      # d_idx 96
    assert lib.msa_sparse_attn_fwd(null, null, null, null, null, null, null, null, -1.0, None, None, None,
                                   1, 0, 0, 16, 2, 4, 128, 64, 1, 1, null, null, null, null, 0, null) == 1


def test_kv_store_validation(lib):
    p = ctypes.c_void_p(256)
    null = None

    def call(k=p, v=p, ik=p, dt=0, ks=256, vs=256, iks=128, B=1, T=4, mp=2, npg=8, Hkv=2, D=128, di=128,
             kscale=None, kc=p, vc=p, ic=p):
        return lib.msa_kv_store_fp8(k, v, ik, dt, ks, vs, iks, p, p, p, B, T, mp, npg, Hkv, D, di,
                                    kscale, None, None, kc, vc, ic, None)
    assert call(dt=2) == 1                        # e4m3 input
    assert call(D=120) == 1                       # D not a multiple of 16
    assert call(di=8) == 1                        # d_idx not a multiple of 16
    assert call(ks=255) == 1                      # token stride below the row
    assert call(ks=260) == 1                      # token stride not a multiple of 8
    assert call(kc=null) == 1                     # k given without its cache
    assert call(k=ctypes.c_void_p(258)) == 1      # misaligned input
    assert call(kscale=_f(0.0)) == 1              # zero scale
    assert call(B=0) == 1
    # T = 0, or no part given: OK without reading a pointer
    assert lib.msa_kv_store_fp8(null, null, null, 0, 0, 0, 0, null, null, null, 1, 0, 1, 1, 2, 128, 128,
                                None, None, None, null, null, null, null) == 0
    assert call(k=null, v=null, ik=null) == 0


def test_rope_quant_validation(lib):
    p = ctypes.c_void_p(256)
    null = None

    def call(nope=p, pe=p, dt=0, rows=4, heads=2, dn=128, dr=64, ns=256, pe_s=128, ph=64, cs=p, mp=10,
             scale=None, out=p):
        return lib.msa_rope_quant_fp8(nope, pe, dt, rows, heads, dn, dr, ns, dn, pe_s, ph, cs, mp, p, 1,
                                      scale, out, None)
    assert call(dt=2) == 1                        # e4m3 input
    assert call(dn=120) == 1                      # d_nope not a multiple of 16
    assert call(dr=48) == 1                       # d_rope not a multiple of 32
    assert call(ns=260) == 1                      # stride not a multiple of 8
    assert call(ph=-8) == 1
    assert call(out=ctypes.c_void_p(264)) == 1    # misaligned output
    assert call(mp=0) == 1
    assert call(scale=_f(float("inf"))) == 1
    assert call(heads=0) == 1
    # rows = 0: OK without reading any pointer
    assert lib.msa_rope_quant_fp8(null, null, 0, 0, 2, 128, 64, 0, 0, 0, 0, null, 1, null, 1,
                                  None, null, null) == 0


def test_header_is_plain_c99():
    # the boundary is a C ABI: the header must compile as strict C99 on its own
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = '#include "msa.h"\nint main(void) { return (int)MSA_OK; }\n'
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-fsyntax-only", "-x", "c", "-"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_noalloc_reports_argument_errors_before_its_scratch_limit(lib):
    # sizes whose scratch would exceed the fixed array, but whose arguments are
    # invalid or unsupported: the argument error is what comes back
    p = ctypes.c_void_p(256)
    T = 1 << 20
    assert lib.msa_index_topk_noalloc(p, p, p, p, p, 1, T, T, 32, 128, 16, 64, 64, p, None) == 2
    assert lib.msa_index_topk_noalloc(p, p, p, p, p, 1, T, T, 4, 96, 16, 64, 64, p, None) == 2
    assert lib.msa_index_topk_noalloc(p, p, p, p, p, 1, T, T, 4, 128, 16, 64, 4096, p, None) == 2
    assert lib.msa_index_topk_noalloc(p, p, p, p, p, 1, T, 0, 4, 128, 16, 64, 64, p, None) == 1
    assert lib.msa_index_topk_noalloc(p, p, p, p, p, 0, T, T, 4, 128, 16, 64, 64, p, None) == 1
    # the same unsupported sizes through the workspace entry point
    assert lib.msa_index_topk(p, p, p, p, p, 1, T, T, 32, 128, 16, 64, 64, p, p, 1 << 40, None) == 2
    # valid sizes over the scratch limit: the limit is reported
    assert lib.msa_index_topk_noalloc(p, p, p, p, p, 1, T, T, 4, 128, 16, 64, 64, p, None) == 5


def test_quant_multi_validation(lib):
    class QT(ctypes.Structure):
        _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                    ("x_row_stride", ctypes.c_int64), ("out", ctypes.c_void_p),
                    ("out_row_stride", ctypes.c_int64), ("scale", ctypes.POINTER(ctypes.c_float))]
    d = (QT * 9)()
    for i in range(9):
        d[i] = QT(256, 4, 16, 16, 512, 16, None)
    arr = ctypes.cast(d, ctypes.c_void_p)
    assert lib.msa_quant_fp8_multi(arr, 0, 0, 2, None) == 1        # n out of range
    assert lib.msa_quant_fp8_multi(arr, 9, 0, 2, None) == 1
    assert lib.msa_quant_fp8_multi(None, 1, 0, 2, None) == 1
    assert lib.msa_quant_fp8_multi(arr, 2, 0, 3, None) == 2        # e5m2
    assert lib.msa_quant_fp8_multi(arr, 2, 2, 2, None) == 1        # e4m3 input
    d[1] = QT(256, 4, 16, 8, 512, 16, None)                       # stride < cols
    assert lib.msa_quant_fp8_multi(arr, 2, 0, 2, None) == 1
    d[1] = QT(256, 4, 16, 16, 512, 16, ctypes.pointer(ctypes.c_float(0.0)))
    assert lib.msa_quant_fp8_multi(arr, 2, 0, 2, None) == 1        # zero scale
    d[0] = QT(None, 0, 16, 16, None, 16, None)
    d[1] = QT(None, 4, 0, 16, None, 16, None)
    assert lib.msa_quant_fp8_multi(arr, 2, 0, 2, None) == 0        # empty entries: no-op
