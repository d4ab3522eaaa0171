"""ctypes binding of libmsa.so (declared in include/msa.h).

Argument marshalling only: tensors become device pointers, optional scales
become host float pointers (None -> NULL = unit scale), the current torch
stream becomes the launch stream. Every step of the path runs in the
library's CUDA kernels; when the library is missing, every call raises.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB: Optional[ctypes.CDLL] = None

MSA_BF16, MSA_FP16, MSA_E4M3, MSA_E5M2 = 0, 1, 2, 3
_STATUS = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_CUDA",
           4: "MSA_ERR_TIMEOUT", 5: "MSA_ERR_WORKSPACE", 6: "MSA_ERR_DATA"}


class MsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    return os.path.join(_HERE, "libmsa.so")


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_FP = ctypes.POINTER(ctypes.c_float)
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "msa_version": ([], _I),
    "msa_last_error_string": ([], ctypes.c_char_p),
    "msa_check_errors": ([_P], _I),
    "msa_profile_enable": ([_I], _I),
    "msa_debug_force_timeouts": ([_I], _I),
    "msa_profile_last_ms": ([_FP], _I),
    "msa_quant_fp8": ([_P, _I, _I64, _I64, _I64, _P, _I, _I64, _FP, _P], _I),
    "msa_quant_fp8_multi": ([_P, _I, _I, _I, _P], _I),
    "msa_kv_store_fp8": ([_P, _P, _P, _I, _I64, _I64, _I64, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                          _FP, _FP, _FP, _P, _P, _P, _P], _I),
    "msa_rope_quant_fp8": ([_P, _P, _I, _I64, _I, _I, _I, _I64, _I64, _I64, _I64, _P, _I, _P, _I,
                            _FP, _P, _P], _I),
    "msa_index_topk_workspace_size": ([_I, _I, _I], _SZ),
    "msa_index_topk": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "msa_index_topk_noalloc": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "msa_sparse_attn_workspace_size": ([_I, _I, _I, _I, _I, _I, _I, _I], _SZ),
    "msa_sparse_attn_fwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _F, _FP, _FP, _FP,
                             _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P], _I),
    "msa_sparse_mla_fwd": ([_P, _P, _P, _P, _P, _F, _FP, _FP, _I, _I, _I, _I, _I, _I,
                            _P, _P, _P, _P], _I),
}


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (once). Raises when it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise MsaError(3, f"{p} is missing; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        msg = load().msa_last_error_string()
        raise MsaError(status, msg.decode() if msg else "")


def _ptr(t: Optional[torch.Tensor]):
    # a plain int: ctypes turns it into the void* the signature declares
    return None if t is None else t.data_ptr()


def _scale(s: Optional[float]):
    # a float passed by reference (the C side reads it during the call)
    return None if s is None else ctypes.byref(ctypes.c_float(float(s)))


def _device(*tensors) -> torch.device:
    """The one device every given tensor (None entries skipped) lives on. A
    call whose tensors sit on different GPUs is refused: the library would
    launch on one device with another device's pointers."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            devs = {str(u.device) for u in tensors if u is not None}
            raise MsaError(1, f"all tensors must be on one device, got {sorted(devs)}")
    if dev is None:
        raise MsaError(1, "no tensor given")
    return dev


_NULL_CTX = contextlib.nullcontext()


def _on(dev: torch.device):
    """Makes `dev` the current device for the call (the library launches on
    the current device, and looks up per-device state there)."""
    if dev.type != "cuda" or dev.index is None or dev.index == torch.cuda.current_device():
        return _NULL_CTX
    return torch.cuda.device(dev)


def _stream(stream: Optional[torch.cuda.Stream], dev: Optional[torch.device] = None):
    """The launch stream: the given one (which must belong to `dev`), else
    torch's current stream of `dev` (of the current device when None)."""
    if stream is not None:
        if dev is not None and dev.type == "cuda" and stream.device != dev:
            raise MsaError(1, f"stream is on {stream.device}, the tensors on {dev}")
        return ctypes.c_void_p(stream.cuda_stream)
    s = torch.cuda.current_stream(dev) if dev is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _on_device(t: torch.Tensor) -> bool:
    return t.is_cuda


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> None:
    """A device tensor of this dtype, contiguous, and of this shape (when given):
    the library reads and writes exactly that extent, so a smaller or host
    buffer is refused here instead of becoming an out-of-bounds access."""
    if not _on_device(t):
        raise MsaError(1, f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise MsaError(1, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MsaError(1, f"{name} must be contiguous")
    if shape is not None and t.shape != shape:
        raise MsaError(1, f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _batch(page_table: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor):
    """(B, max_pages) of a batch description, with its three tensors checked."""
    if page_table.dim() != 2:
        raise MsaError(1, "page_table must be [B, max_pages]")
    B, max_pages = page_table.shape
    _dev(page_table, "page_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32, (B,))
    _dev(cu_q, "cu_q", torch.int32, (B + 1,))
    return B, max_pages


def check_errors(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Synchronise and raise if a kernel recorded a device-side data error
    (on the stream's device, or the current device when no stream is given)."""
    dev = stream.device if stream is not None else None
    with (_on(dev) if dev is not None else contextlib.nullcontext()):
        _check(load().msa_check_errors(_stream(stream, dev)))


def debug_force_timeouts(on: bool) -> None:
    """Debug switch of the current device: while on, every bounded wait in the
    library's kernels that is not complete at its first test gives up at once
    (the failure path: error word, drain, return). Outputs are meaningless
    meanwhile; the next check_errors reports the timeout."""
    _check(load().msa_debug_force_timeouts(1 if on else 0))


def profile_enable(on: bool = True) -> None:
    """Record events around the main attention kernel of each call (instrumentation)."""
    _check(load().msa_profile_enable(1 if on else 0))


def profile_last_ms() -> float:
    """Elapsed ms of the most recently profiled main attention kernel."""
    v = ctypes.c_float(0.0)
    _check(load().msa_profile_last_ms(ctypes.byref(v)))
    return float(v.value)


def quant_fp8(x: torch.Tensor, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """e4m3 codes of x * (1/scale) (step a1); x is bf16 or fp16, last dim contiguous."""
    lib = load()
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise MsaError(1, f"x must be bf16 or fp16, got {x.dtype}")
    if not _on_device(x):
        raise MsaError(1, "x must be a CUDA tensor")
    if x.stride(-1) != 1:
        raise MsaError(1, "x must have a contiguous last dimension")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    x2 = x.reshape(rows, cols) if x.dim() != 2 else x
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _dev(out, "out", torch.uint8)
    if out.numel() != x.numel():
        raise MsaError(1, f"out must hold {x.numel()} elements, got {out.numel()}")
    o2 = out.view(rows, cols)
    dev = _device(x, out)
    with _on(dev):
        _check(lib.msa_quant_fp8(_ptr(x2), MSA_BF16 if x.dtype == torch.bfloat16 else MSA_FP16,
                                 rows, cols, x2.stride(0) if rows else cols, _ptr(o2), MSA_E4M3,
                                 o2.stride(0) if rows else cols, _scale(scale), _stream(stream, dev)))
    return out


class _QuantTensor(ctypes.Structure):
    """msa_quant_tensor of include/msa.h (scale: a const float*, here as an address)."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("x_row_stride", ctypes.c_int64), ("out", ctypes.c_void_p),
                ("out_row_stride", ctypes.c_int64), ("scale", ctypes.c_void_p)]


QUANT_MULTI_MAX = 8
# array types made once (building a ctypes array type costs more than the call)
_QT_ARRAYS = [None] + [_QuantTensor * n for n in range(1, QUANT_MULTI_MAX + 1)]
_F32_ARRAYS = [None] + [ctypes.c_float * n for n in range(1, QUANT_MULTI_MAX + 1)]


def quant_fp8_multi(items, stream=None):
    """Several quantisations in one launch (step a for Q and idx_q together).

    items: sequence of (x, scale) or (x, scale, out) with x bf16 / fp16 (one
    dtype for all) and a contiguous last dimension; returns the e4m3 outputs,
    each byte-identical to quant_fp8(x, scale)."""
    lib = load()
    n_items = len(items)
    if not 1 <= n_items <= QUANT_MULTI_MAX:
        raise MsaError(1, f"need 1..{QUANT_MULTI_MAX} tensors, got {n_items}")
    dt = items[0][0].dtype
    if dt not in (torch.bfloat16, torch.float16):
        raise MsaError(1, f"x must be bf16 or fp16, got {dt}")
    descs = _QT_ARRAYS[n_items]()
    scales = _F32_ARRAYS[n_items]()          # the scales the descriptors point at
    s_addr = ctypes.addressof(scales)
    keep, outs = [], []
    dev = items[0][0].device
    for i, it in enumerate(items):
        x, scale = it[0], it[1]
        out = it[2] if len(it) > 2 else None
        if x.dtype != dt:
            raise MsaError(1, "all tensors must share one dtype")
        if not _on_device(x):
            raise MsaError(1, "x must be a CUDA tensor")
        if x.stride(-1) != 1:
            raise MsaError(1, "x must have a contiguous last dimension")
        cols = x.shape[-1]
        n = x.numel()
        rows = n // cols if cols else 0
        if x.is_contiguous():                  # rows of `cols` elements, back to back
            x2, xstride = x, cols
        else:
            x2 = x.reshape(rows, cols) if x.dim() != 2 else x
            xstride = x2.stride(0) if rows else cols
        if out is None:
            out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        else:
            _dev(out, "out", torch.uint8)
            if out.numel() != n:
                raise MsaError(1, f"out must hold {n} elements, got {out.numel()}")
        if x.device != dev or out.device != dev:
            raise MsaError(1, f"all tensors must be on one device, got {x.device} / {out.device} / {dev}")
        d = descs[i]
        d.x, d.rows, d.cols, d.x_row_stride = x2.data_ptr(), rows, cols, xstride
        d.out, d.out_row_stride = out.data_ptr(), cols
        if scale is not None:
            scales[i] = float(scale)
            d.scale = s_addr + 4 * i
        keep.append(x2)
        outs.append(out)
    with _on(dev):
        _check(lib.msa_quant_fp8_multi(ctypes.addressof(descs), n_items,
                                       MSA_BF16 if dt == torch.bfloat16 else MSA_FP16, MSA_E4M3,
                                       _stream(stream, dev)))
    return outs


def _token_rows(x: Optional[torch.Tensor], name: str, inner: int):
    """Token stride of x, whose per-token block of `inner` elements is contiguous."""
    if x is None:
        return 0
    if not _on_device(x) or x.dtype not in (torch.bfloat16, torch.float16):
        raise MsaError(1, f"{name} must be a bf16 or fp16 CUDA tensor")
    want, acc = [], 1
    for n in reversed(x.shape[1:]):
        want.insert(0, acc)
        acc *= n
    if acc != inner or any(n > 1 and st != w for n, st, w in zip(x.shape[1:], x.stride()[1:], want)):
        raise MsaError(1, f"{name} must be [T, ...] with {inner} contiguous elements per token")
    return x.stride(0) if x.shape[0] > 1 else inner


def kv_store_fp8(page_table: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor,
                 k_cache: Optional[torch.Tensor] = None, v_cache: Optional[torch.Tensor] = None,
                 idx_k_cache: Optional[torch.Tensor] = None, k: Optional[torch.Tensor] = None,
                 v: Optional[torch.Tensor] = None, idx_k: Optional[torch.Tensor] = None,
                 k_scale: Optional[float] = None, v_scale: Optional[float] = None,
                 idx_k_scale: Optional[float] = None, stream=None) -> None:
    """Quantise new K [T, Hkv, D], V and index K [T, d_idx] into the paged e4m3
    caches in place, at the slots the batch description gives."""
    lib = load()
    given = [x for x in (k, v, idx_k) if x is not None]
    if not given:
        return
    dt = given[0].dtype
    if any(x.dtype != dt for x in given):
        raise MsaError(1, "k, v and idx_k must share one dtype")
    B, max_pages = _batch(page_table, seq_lens, cu_q)
    for c, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (idx_k_cache, "idx_k_cache")):
        if c is not None:
            _dev(c, n, torch.uint8)
    kv = k if k is not None else v
    T = given[0].shape[0]
    if any(x.shape[0] != T for x in given):
        raise MsaError(1, "k, v and idx_k must have the same number of tokens")
    if kv is not None and (kv.dim() != 3 or (k is not None and v is not None and k.shape != v.shape)):
        raise MsaError(1, "k and v must be [T, Hkv, D] of one shape")
    if idx_k is not None and idx_k.dim() != 2:
        raise MsaError(1, "idx_k must be [T, d_idx]")
    Hkv, D = (kv.shape[1], kv.shape[2]) if kv is not None else (0, 16)
    d_idx = idx_k.shape[1] if idx_k is not None else 16
    parts = [(x, c, n, shape) for x, c, n, shape in
             ((k, k_cache, "k_cache", (Hkv, 128, D)), (v, v_cache, "v_cache", (Hkv, 128, D)),
              (idx_k, idx_k_cache, "idx_k_cache", (128, d_idx))) if x is not None]
    if any(c is None for _, c, _, _ in parts):
        raise MsaError(1, "every given input needs its cache")
    cache = parts[0][1]
    for _, c, n, shape in parts:
        if tuple(c.shape[1:]) != shape or c.shape[0] != cache.shape[0]:
            raise MsaError(1, f"{n} must be [num_pages, {', '.join(map(str, shape))}], got {tuple(c.shape)}")
    dev = _device(k, v, idx_k, k_cache, v_cache, idx_k_cache, page_table, seq_lens, cu_q)
    with _on(dev):
        _check(lib.msa_kv_store_fp8(_ptr(k), _ptr(v), _ptr(idx_k),
                                    MSA_BF16 if dt == torch.bfloat16 else MSA_FP16,
                                    _token_rows(k, "k", Hkv * D), _token_rows(v, "v", Hkv * D),
                                    _token_rows(idx_k, "idx_k", d_idx), _ptr(page_table),
                                    _ptr(seq_lens), _ptr(cu_q), B, T, max_pages, cache.shape[0], Hkv,
                                    D, d_idx, _scale(k_scale), _scale(v_scale), _scale(idx_k_scale),
                                    _ptr(k_cache), _ptr(v_cache), _ptr(idx_k_cache),
                                    _stream(stream, dev)))


def rope_quant_fp8(nope: Optional[torch.Tensor], pe: torch.Tensor, cos_sin_cache: torch.Tensor,
                   positions: torch.Tensor, is_neox: bool = True, scale: Optional[float] = None,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """e4m3 codes [rows, heads, d_nope + d_rope] of nope || rope(pe).

    nope: [rows, heads, d_nope] (or None when d_nope = 0); pe: [rows, heads or
    1, d_rope], a single head broadcast to all; last dims contiguous."""
    lib = load()
    rows, hp, d_rope = pe.shape
    heads, d_nope = (nope.shape[1], nope.shape[2]) if nope is not None else (hp, 0)
    dt = pe.dtype
    for x, n in ((nope, "nope"), (pe, "pe")):
        if x is None:
            continue
        if not _on_device(x) or x.dtype != dt or dt not in (torch.bfloat16, torch.float16):
            raise MsaError(1, f"{n} must be a bf16 or fp16 CUDA tensor like pe")
        if x.dim() != 3 or x.shape[0] != rows or (x.shape[2] > 1 and x.stride(2) != 1):
            raise MsaError(1, f"{n} must be [rows, heads, d] with a contiguous last dim")
    if hp not in (1, heads):
        raise MsaError(1, "pe must have 1 head or as many as nope")
    _dev(cos_sin_cache, "cos_sin_cache", torch.float32)
    _dev(positions, "positions", torch.int32)
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != d_rope or positions.numel() != rows:
        raise MsaError(1, "cos_sin_cache must be [max_pos, d_rope] and positions [rows]")
    if out is None:
        out = torch.empty((rows, heads, d_nope + d_rope), dtype=torch.uint8, device=pe.device)
    _dev(out, "out", torch.uint8)
    if tuple(out.shape) != (rows, heads, d_nope + d_rope):
        raise MsaError(1, f"out must be [{rows}, {heads}, {d_nope + d_rope}]")
    ns = (nope.stride(0), nope.stride(1)) if nope is not None else (0, 0)
    ps = (pe.stride(0), pe.stride(1) if hp == heads and heads > 1 else 0)
    dev = _device(nope, pe, cos_sin_cache, positions, out)
    with _on(dev):
        _check(lib.msa_rope_quant_fp8(_ptr(nope), _ptr(pe), MSA_BF16 if dt == torch.bfloat16 else MSA_FP16,
                                      rows, heads, d_nope, d_rope, ns[0], ns[1], ps[0], ps[1],
                                      _ptr(cos_sin_cache), cos_sin_cache.shape[0], _ptr(positions),
                                      1 if is_neox else 0, _scale(scale), _ptr(out),
                                      _stream(stream, dev)))
    return out


def index_topk_workspace_size(T: int, Hidx: int, max_pages: int) -> int:
    return int(load().msa_index_topk_workspace_size(T, Hidx, max_pages))


def index_topk(idx_q: torch.Tensor, idx_k_cache: torch.Tensor, page_table: torch.Tensor,
               seq_lens: torch.Tensor, cu_q: torch.Tensor, topk: int, max_q_len: int,
               out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """topk_indices [Hidx, T, topk] int32 (steps a2+a3)."""
    lib = load()
    T, Hidx, D = idx_q.shape
    num_pages = idx_k_cache.shape[0]
    _dev(idx_q, "idx_q", torch.uint8)
    _dev(idx_k_cache, "idx_k_cache", torch.uint8, (num_pages, 128, D))
    B, max_pages = _batch(page_table, seq_lens, cu_q)
    if out is None:
        out = torch.empty((Hidx, T, topk), dtype=torch.int32, device=idx_q.device)
    _dev(out, "out", torch.int32, (Hidx, T, topk))
    if workspace is None:           # (a given workspace's size is checked by the library)
        ws_bytes = index_topk_workspace_size(T, Hidx, max_pages)
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=idx_q.device)
    _dev(workspace, "workspace", torch.uint8)
    dev = _device(idx_q, idx_k_cache, page_table, seq_lens, cu_q, out, workspace)
    with _on(dev):
        _check(lib.msa_index_topk(_ptr(idx_q), _ptr(idx_k_cache), _ptr(page_table), _ptr(seq_lens),
                                  _ptr(cu_q), B, T, max_q_len, Hidx, D, topk, num_pages, max_pages,
                                  _ptr(out), _ptr(workspace), workspace.numel(),
                                  _stream(stream, dev)))
    return out


def index_topk_noalloc(idx_q: torch.Tensor, idx_k_cache: torch.Tensor, page_table: torch.Tensor,
                       seq_lens: torch.Tensor, cu_q: torch.Tensor, topk: int, max_q_len: int,
                       out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """index_topk without a workspace: the library's fixed device scratch is
    used instead (for callers that may not allocate device memory)."""
    lib = load()
    T, Hidx, D = idx_q.shape
    num_pages = idx_k_cache.shape[0]
    _dev(idx_q, "idx_q", torch.uint8)
    _dev(idx_k_cache, "idx_k_cache", torch.uint8, (num_pages, 128, D))
    B, max_pages = _batch(page_table, seq_lens, cu_q)
    if out is None:
        out = torch.empty((Hidx, T, topk), dtype=torch.int32, device=idx_q.device)
    _dev(out, "out", torch.int32, (Hidx, T, topk))
    dev = _device(idx_q, idx_k_cache, page_table, seq_lens, cu_q, out)
    with _on(dev):
        _check(lib.msa_index_topk_noalloc(_ptr(idx_q), _ptr(idx_k_cache), _ptr(page_table),
                                          _ptr(seq_lens), _ptr(cu_q), B, T, max_q_len, Hidx, D, topk,
                                          num_pages, max_pages, _ptr(out), _stream(stream, dev)))
    return out


def sparse_attn_workspace_size(B: int, T: int, max_q_len: int, Hq: int, Hkv: int, Hidx: int,
                               topk: int, max_pages: int) -> int:
    return int(load().msa_sparse_attn_workspace_size(B, T, max_q_len, Hq, Hkv, Hidx, topk, max_pages))


def sparse_attn_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    page_table: torch.Tensor, seq_lens: torch.Tensor, cu_q: torch.Tensor,
                    topk_indices: torch.Tensor, sink: Optional[torch.Tensor], sm_scale: float,
                    q_scale: Optional[float], k_scale: Optional[float], v_scale: Optional[float],
                    max_q_len: int, out=None, max_logit=None, lse=None, workspace=None,
                    stream=None):
    """Sparse GQA attention (steps a4/a5). Returns (out bf16, max_logit, lse)."""
    lib = load()
    T, Hq, D = q.shape
    if k_cache.dim() != 4 or topk_indices.dim() != 3:
        raise MsaError(1, "k_cache must be [num_pages, Hkv, 128, D] and topk_indices [Hidx, T, topk]")
    num_pages, Hkv = k_cache.shape[0], k_cache.shape[1]
    Hidx, _, topk = topk_indices.shape
    _dev(q, "q", torch.uint8)
    _dev(k_cache, "k_cache", torch.uint8, (num_pages, Hkv, 128, D))
    _dev(v_cache, "v_cache", torch.uint8, (num_pages, Hkv, 128, D))
    B, max_pages = _batch(page_table, seq_lens, cu_q)
    _dev(topk_indices, "topk_indices", torch.int32, (Hidx, T, topk))
    if sink is not None:
        _dev(sink, "sink", torch.float32, (Hq,))
    dev = q.device
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev) if out is None else out
    max_logit = torch.empty((T, Hq), dtype=torch.float32, device=dev) if max_logit is None else max_logit
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev) if lse is None else lse
    _dev(out, "out", torch.bfloat16, (T, Hq, D))
    _dev(max_logit, "max_logit", torch.float32, (T, Hq))
    _dev(lse, "lse", torch.float32, (T, Hq))
    if workspace is None:           # (a given workspace's size is checked by the library)
        ws_bytes = sparse_attn_workspace_size(B, T, max_q_len, Hq, Hkv, Hidx, topk, max_pages)
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _dev(workspace, "workspace", torch.uint8)
    dev = _device(q, k_cache, v_cache, page_table, seq_lens, cu_q, topk_indices, sink, out,
                  max_logit, lse, workspace)
    with _on(dev):
        _check(lib.msa_sparse_attn_fwd(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seq_lens), _ptr(cu_q),
            _ptr(topk_indices), _ptr(sink), float(sm_scale), _scale(q_scale), _scale(k_scale),
            _scale(v_scale), B, T, max_q_len, Hq, Hkv, Hidx, D, topk, num_pages, max_pages,
            _ptr(out), _ptr(max_logit), _ptr(lse), _ptr(workspace), workspace.numel(),
            _stream(stream, dev)))
    return out, max_logit, lse


def sparse_mla_fwd(q: torch.Tensor, kv: torch.Tensor, indices: torch.Tensor,
                   topk_length: Optional[torch.Tensor], sink: Optional[torch.Tensor],
                   sm_scale: float, q_scale: Optional[float], kv_scale: Optional[float],
                   d_v: int = 512, out=None, max_logits=None, lse=None, stream=None):
    """Sparse MLA prefill (step a6). Returns (out bf16, max_logits, lse)."""
    lib = load()
    T, H, d_qk = q.shape
    S_kv = kv.shape[0]
    if indices.dim() != 2:
        raise MsaError(1, "indices must be [T, topk]")
    topk = indices.shape[1]
    _dev(q, "q", torch.uint8)
    _dev(kv, "kv", torch.uint8, (S_kv, d_qk))
    _dev(indices, "indices", torch.int32, (T, topk))
    if topk_length is not None:
        _dev(topk_length, "topk_length", torch.int32, (T,))
    if sink is not None:
        _dev(sink, "sink", torch.float32, (H,))
    dev = q.device
    out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=dev) if out is None else out
    max_logits = torch.empty((T, H), dtype=torch.float32, device=dev) if max_logits is None else max_logits
    lse = torch.empty((T, H), dtype=torch.float32, device=dev) if lse is None else lse
    _dev(out, "out", torch.bfloat16, (T, H, d_v))
    _dev(max_logits, "max_logits", torch.float32, (T, H))
    _dev(lse, "lse", torch.float32, (T, H))
    dev = _device(q, kv, indices, topk_length, sink, out, max_logits, lse)
    with _on(dev):
        _check(lib.msa_sparse_mla_fwd(_ptr(q), _ptr(kv), _ptr(indices), _ptr(topk_length), _ptr(sink),
                                      float(sm_scale), _scale(q_scale), _scale(kv_scale), T, H, S_kv,
                                      d_qk, d_v, topk, _ptr(out), _ptr(max_logits), _ptr(lse),
                                      _stream(stream, dev)))
    return out, max_logits, lse
