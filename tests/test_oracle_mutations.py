"""The oracle's pins catch plausible mistakes: each case plants one mistake
in a copy of an oracle module's source (a wrong exponent bias or subnormal
step, truncation instead of round-to-even, a lost sign, a reciprocal taken
in the wrong precision, a mean instead of a max, the wrong tie order, a
dropped sort, an off-by-one position, a wrong head mapping, the k scale on
the sink, the sink left out of the normaliser, an off-by-one slot, swapped
cos/sin, ...), runs that module's pin tests against the copy, and expects at
least one of them to fail. Nothing here touches the GPU path."""

import inspect
import os
import types

import pytest

import oracle
import test_oracle_attention as attn_pins
import test_oracle_e4m3 as e4m3_pins
import test_oracle_index_topk as index_pins
import test_oracle_kv_store as kv_pins
import test_oracle_mla as mla_pins
import test_oracle_no_tie as no_tie_pins
import test_oracle_quant as quant_pins
import test_oracle_rope_quant as rope_pins

ORACLE_DIR = os.path.dirname(oracle.__file__)

E4M3_MUTATIONS = [
    ("SUBNORMAL_STEP = 2.0 ** -9", "SUBNORMAL_STEP = 2.0 ** -10"),
    ("np.exp2(exp_field - 7.0)", "np.exp2(exp_field - 8.0)"),
    ("out[saturate] = 0x7E", "out[saturate] = 0x7F"),
    ("q = np.rint((2.0 * frac - 1.0) * 8.0)", "q = np.floor((2.0 * frac - 1.0) * 8.0)"),
    ("out |= (negative.astype(np.uint8) << 7)", "out |= (negative.astype(np.uint8) << 6)"),
    ("out[subnormal] = np.rint(", "out[subnormal] = np.floor("),
]

QUANT_MUTATIONS = [
    ("return np.float32(1.0) / np.float32(scale)", "return np.float32(1.0 / scale)"),
    ("v = x * scale_inverse(scale)", "v = (x / np.float32(1.0 if scale is None else scale)).astype(np.float32)"),
    ("astype(np.uint32) << 16", "astype(np.uint32) << 15"),
    ("x = bf16_bits_to_f32(x_bits)", "x = f16_bits_to_f32(x_bits)"),
]

INDEX_MUTATIONS = [
    ("return dots.max(axis=2)", "return dots.mean(axis=2)"),
    ("order = np.lexsort((cand, -scores))", "order = np.lexsort((-cand, -scores))"),
    ("picked = np.sort(order[:n_pick])", "picked = order[:n_pick]"),
    ("if own_block + 1 <= topk:", "if own_block <= topk:"),
    ("pos[lo:hi] = seq_lens[b] - (hi - lo) + np.arange(hi - lo)",
     "pos[lo:hi] = seq_lens[b] - (hi - lo) - 1 + np.arange(hi - lo)"),
    ("page_table[b, :own])", "page_table[b, 1:own + 1])"),
    ('np.einsum("hd,nkd->hnk", q, k)', 'np.einsum("hd,nkd->hnk", q, k[..., ::-1])'),
]

ATTENTION_MUTATIONS = [
    ("i = h // (hq // hidx)", "i = h % hidx"),
    ("g = h // (hq // hkv)", "g = h % hkv"),
    ("else c * float(sink[h])", "else c_qk * float(sink[h])"),
    ("kpos = kpos[kpos <= pos]", "kpos = kpos[kpos < pos]"),
    ("out[n, h] = vs * o", "out[n, h] = o"),
    ("z = float(w.sum()) + (0.0 if sigma is None else float(np.exp(sigma - top)))", "z = float(w.sum())"),
    ("return o, m, top + float(np.log(z))", "return o, top, top + float(np.log(z))"),
    ("c_qk = c * unit(k_scale)", "c_qk = c"),
]

MLA_MUTATIONS = [
    ("row = row[: int(topk_length[t])]", "row = row[: int(topk_length[t]) - 1]"),
    ("vv = e4m3.decode(kv[row, :d_v])", "vv = e4m3.decode(kv[row, -d_v:])"),
    ("logits = (c * kvs) * (", "logits = c * ("),
    ("out[n, hh] = kvs * o", "out[n, hh] = o"),
    ("row = row[row >= 0]", "row = row[row >= -1]"),
    ("else c * float(sink[hh])", "else c * kvs * float(sink[hh])"),
]

KV_MUTATIONS = [
    ("pos % PAGE", "(pos + 1) % PAGE"),
    ("j = int(pos[t]) // PAGE", "j = (int(pos[t]) + 1) // PAGE"),
    ("cache[page, :, slots[t], :] = codes[t]", "cache[page, :, slots[t], :] = codes[t][::-1]"),
    ("codes = quant.quantize(x, scale, dtype)", "codes = quant.quantize(x, None, dtype)"),
    ("cache[page, slots[t], :] = codes[t]", "cache[page, slots[t] - 1, :] = codes[t]"),
]

ROPE_MUTATIONS = [
    ("out[..., :half] = x1 * c - x2 * s", "out[..., :half] = x1 * c + x2 * s"),
    ("out[..., half:] = x2 * c + x1 * s", "out[..., half:] = x2 * c - x1 * s"),
    ("c = cs[:, None, :half]\n    s = cs[:, None, half:]", "s = cs[:, None, :half]\n    c = cs[:, None, half:]"),
    ("x1, x2 = pe[..., 0::2], pe[..., 1::2]", "x2, x1 = pe[..., 0::2], pe[..., 1::2]"),
    ("out[..., 1::2] = x2 * c + x1 * s", "out[..., 1::2] = x2 * c + x1 * s * 1.0001"),
    ("e4m3.encode((rotated * s_inv).astype(np.float32))", "e4m3.encode((rotated).astype(np.float32))"),
    ("pe = np.broadcast_to(pe, (rows, heads, pe.shape[2]))",
     "pe = np.broadcast_to(pe[:, :, ::-1], (rows, heads, pe.shape[2]))"),
]


NO_TIE_MUTATIONS = [
    ("return 2.0 * D * 2.0 ** -23 * s.max(axis=0)", "return D * 2.0 ** -23 * s.max(axis=0)"),
    ("near = ~(gaps > bounds)", "near = gaps < bounds"),
    ("keys = idx_k_codes[page_table[seq[t], :own]]", "keys = idx_k_codes[page_table[seq[t], 1:own]]"),
    ("if int((fresh & np.uint16(0x7FFF)).max()) <= amax_bits:", "if True:"),
    ("pending, _, _ = near_tie_tokens(codes, idx_k_codes, page_table, seq_lens, cu_q, topk,\n"
     "                                        pending)", "pending = []"),
]


def _mutant(module: str, old: str, new: str) -> types.ModuleType:
    path = os.path.join(ORACLE_DIR, module + ".py")
    src = open(path).read()
    assert src.count(old) == 1, (module, old)
    m = types.ModuleType(f"oracle._mutant_{module}")
    m.__package__ = "oracle"
    m.__file__ = path
    exec(compile(src.replace(old, new), path, "exec"), m.__dict__)
    return m


def _cases(fn):
    """Argument sets of a pin test: the product of its parametrize marks."""
    cases = [{}]
    for mk in getattr(fn, "pytestmark", []):
        if mk.name != "parametrize":
            continue
        names, values = mk.args[0], mk.args[1]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        rows = []
        for v in values:
            v = v.values if hasattr(v, "values") and not isinstance(v, dict) else v   # pytest.param
            rows.append(dict(zip(names, v)) if len(names) > 1 else {names[0]: v[0] if isinstance(v, tuple) and len(v) == 1 else v})
        cases = [dict(c, **r) for c in cases for r in rows]
    return cases


def _pins_fail(pins, attr: str, mutant) -> bool:
    saved = getattr(pins, attr)
    setattr(pins, attr, mutant)
    try:
        for name, fn in inspect.getmembers(pins, inspect.isfunction):
            if not name.startswith("test_") or fn.__module__ != pins.__name__:
                continue
            for kw in _cases(fn):
                try:
                    fn(**kw)
                except Exception:
                    return True
        return False
    finally:
        setattr(pins, attr, saved)


def test_unmutated_oracles_pass_their_pins():
    same = lambda module: _mutant(module, "import numpy as np", "import numpy as np")
    assert not _pins_fail(e4m3_pins, "e4m3", same("e4m3"))
    assert not _pins_fail(quant_pins, "quant", same("quant"))
    assert not _pins_fail(index_pins, "ot", same("index_topk"))
    assert not _pins_fail(attn_pins, "sparse_attention", same("attention").sparse_attention)
    assert not _pins_fail(mla_pins, "sparse_mla", same("mla").sparse_mla)
    assert not _pins_fail(kv_pins, "okv", same("kv_store"))
    assert not _pins_fail(rope_pins, "orq", same("rope_quant"))
    assert not _pins_fail(no_tie_pins, "nt", same("no_tie"))


@pytest.mark.parametrize("old,new", E4M3_MUTATIONS)
def test_e4m3_pins_catch(old, new):
    assert _pins_fail(e4m3_pins, "e4m3", _mutant("e4m3", old, new))


@pytest.mark.parametrize("old,new", QUANT_MUTATIONS)
def test_quant_pins_catch(old, new):
    assert _pins_fail(quant_pins, "quant", _mutant("quant", old, new))


@pytest.mark.parametrize("old,new", INDEX_MUTATIONS)
def test_index_topk_pins_catch(old, new):
    assert _pins_fail(index_pins, "ot", _mutant("index_topk", old, new))


@pytest.mark.parametrize("old,new", ATTENTION_MUTATIONS)
def test_attention_pins_catch(old, new):
    m = _mutant("attention", old, new)
    assert _pins_fail(attn_pins, "sparse_attention", m.sparse_attention)


@pytest.mark.parametrize("old,new", MLA_MUTATIONS)
def test_mla_pins_catch(old, new):
    m = _mutant("mla", old, new)
    assert _pins_fail(mla_pins, "sparse_mla", m.sparse_mla)


@pytest.mark.parametrize("old,new", KV_MUTATIONS)
def test_kv_store_pins_catch(old, new):
    assert _pins_fail(kv_pins, "okv", _mutant("kv_store", old, new))


@pytest.mark.parametrize("old,new", ROPE_MUTATIONS)
def test_rope_quant_pins_catch(old, new):
    assert _pins_fail(rope_pins, "orq", _mutant("rope_quant", old, new))


@pytest.mark.parametrize("old,new", NO_TIE_MUTATIONS)
def test_no_tie_pins_catch(old, new):
    assert _pins_fail(no_tie_pins, "nt", _mutant("no_tie", old, new))
