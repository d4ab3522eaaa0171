#!/usr/bin/env python
"""Benchmark of the FP8 (e4m3) top-k block-sparse attention path on GB300.

One step = the whole hot path over one batch of the 32k prefill workload
(1 sequence x 32768 tokens, 16 q / 2 kv / 4 index heads, head_dim 128, top-k
64 blocks of 128 tokens): quantise Q and idx_q (one launch), index scores + ascending
top-k, sparse attention with sink. The metric is prefill tokens/s; the same
line reports the attention kernel's algorithmic TFLOP/s against the FP8
tensor peak, the paged-decode workload's HBM GB/s (eager and as one CUDA
graph replay), the sparse-MLA kernel with its fused rope + e4m3 producer, the
quantised KV-cache store of the prefill and decode workloads' new tokens, an
end-to-end figure with host buffers, and the CPU oracle timed on a bounded
sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

With N > 1 it runs under torch.distributed.run, one independent replica per
GPU (the path has no exchange step), and reports the whole-job throughput.
`--impl reference` times the CPU oracle (the only other implementation of
the path) on the same workload and prints the same JSON line.
"""

from __future__ import annotations

import argparse
import csv
import gc
import hashlib
import io
import json
import math
import os
import resource
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn prefill tokens/s + TFLOP/s (% FP8 peak) at 32k; decode HBM GB/s"
UNIT = "tokens/s"
WORKLOAD = "prefill32k"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--no-decode", action="store_true", help="skip the paged-decode measurement")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU oracle sample budget")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    p.add_argument("--no-mla", action="store_true", help="skip the sparse-MLA measurement")
    p.add_argument("--only", choices=["prefill", "decode", "mla", "kv_store"], default=None,
                   help="run only this part of the path, warm-up + steps times, untimed, and "
                        "print no result line (for profiler captures; mla also runs the rope "
                        "producer of its q, kv_store stores the --workload's new tokens)")
    p.add_argument("--workload", default=WORKLOAD, choices=["prefill32k", "prefill8k", "tiny"],
                   help="prefill workload of the step (the benchmark line uses prefill32k)")
    return p.parse_args()


# ----------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK["hbm_gbs"], "bf16_tflops": FALLBACK["bf16_tflops"],
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        rows = list(csv.reader(io.StringIO(open(self.out.name).read())))
        os.unlink(self.out.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "fp8_block_sparse_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel_file: str, profile_name: str):
    """DRAM bytes per launch from a committed ncu summary (markdown with the
    lines `source_hash: ...` and `dram_bytes_per_launch: ...`), if the summary
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip().strip("`* -")] = v.strip().strip("`* ")
    if fields.get("source_hash") != src_hash(kernel_file, "common.cuh"):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _queued_ms(fn, steps, flush):
    """Device milliseconds of each of `steps` calls of `fn`, queued back to
    back on the current stream (flush, event, call, event) with one
    synchronisation after the last: the host's launches run ahead of the GPU
    as in a serving loop, where a synchronisation per step would add the
    host's launch latency to every step."""
    import torch
    s = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(s)
        fn()
        b.record(s)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


class L2Flush:
    """Evicts the 129 MB L2 before a timed step: a 256 MB write, then a
    256 MB read, so that the lines left in L2 are clean and the step does not
    pay for writing the flush buffer back to HBM."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(32 << 20, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


# ----------------------------------------------------------------- workloads
def gqa_setup(msa, wl, name, dev, pinned=False):
    """Inputs resident in HBM (caches quantised once by the library) and
    preallocated outputs / workspaces, so a step allocates nothing."""
    import numpy as np
    import torch
    w = wl.make_gqa(wl.CONFIGS[name])
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    st = {"w": w}
    st["q_host"] = bf(w.q).pin_memory() if pinned else None
    st["iq_host"] = bf(w.idx_q).pin_memory() if pinned else None
    st["q"] = bf(w.q).to(dev)
    st["iq"] = bf(w.idx_q).to(dev)
    for key, arr, sc in (("k8", w.k_pool, "k"), ("v8", w.v_pool, "v"), ("ik8", w.idx_k_pool, "idx_k")):
        tmp = bf(arr).to(dev)
        st[key] = msa.quant_fp8(tmp, w.scales[sc])
        del tmp
    st["pt"], st["sl"], st["cu"], st["sink"] = t(w.page_table), t(w.seq_lens), t(w.cu_q), t(w.sink)
    T, cfg = w.T, w.cfg
    B, max_pages = w.page_table.shape
    st["q8"] = torch.empty((T, cfg.Hq, cfg.D), dtype=torch.uint8, device=dev)
    st["iq8"] = torch.empty((T, cfg.Hidx, cfg.d_idx), dtype=torch.uint8, device=dev)
    st["ids"] = torch.empty((cfg.Hidx, T, cfg.topk), dtype=torch.int32, device=dev)
    st["ws_idx"] = torch.empty(max(1, msa.index_topk_workspace_size(T, cfg.Hidx, max_pages)),
                               dtype=torch.uint8, device=dev)
    st["ws_attn"] = torch.empty(max(1, msa.sparse_attn_workspace_size(
        B, T, w.max_q_len, cfg.Hq, cfg.Hkv, cfg.Hidx, cfg.topk, max_pages)), dtype=torch.uint8, device=dev)
    st["o"] = torch.empty((T, cfg.Hq, cfg.D), dtype=torch.bfloat16, device=dev)
    st["ml"] = torch.empty((T, cfg.Hq), dtype=torch.float32, device=dev)
    st["lse"] = torch.empty((T, cfg.Hq), dtype=torch.float32, device=dev)
    if pinned:
        st["o_host"] = torch.empty(st["o"].shape, dtype=torch.bfloat16).pin_memory()
        st["lse_host"] = torch.empty(st["lse"].shape, dtype=torch.float32).pin_memory()
        st["ml_host"] = torch.empty(st["ml"].shape, dtype=torch.float32).pin_memory()
    return st


LAUNCHES_PREFILL = 1 + 3 + 3     # quant (Q and idx_q, one launch); index: plan, score, select; attn: plan, V^T, attention
LAUNCHES_DECODE = 1 + 2 + 2      # quant (q and idx_q, one launch); index: score, select; attn: decode, combine


def run_path(msa, st, q_in=None, iq_in=None):
    w = st["w"]
    cfg = w.cfg
    msa.quant_fp8_multi([(st["q"] if q_in is None else q_in, w.scales["q"], st["q8"]),
                         (st["iq"] if iq_in is None else iq_in, w.scales["idx_q"], st["iq8"])])
    msa.index_topk(st["iq8"], st["ik8"], st["pt"], st["sl"], st["cu"], cfg.topk, w.max_q_len,
                   out=st["ids"], workspace=st["ws_idx"])
    msa.sparse_attn_fwd(st["q8"], st["k8"], st["v8"], st["pt"], st["sl"], st["cu"], st["ids"], st["sink"],
                        w.sm_scale, w.scales["q"], w.scales["k"], w.scales["v"], w.max_q_len,
                        out=st["o"], max_logit=st["ml"], lse=st["lse"], workspace=st["ws_attn"])


def selected_keys(st):
    """Per (index head, token): number of causal keys in its selected blocks,
    and the executed key count of the kernel's 128-row union tiles."""
    import torch
    w = st["w"]
    ids = st["ids"].long()
    T = w.T
    pos = torch.arange(T, device=ids.device)        # one sequence, no prefix
    own = pos // 128
    valid = ids >= 0
    keys = torch.where(ids < own[None, :, None], 128, (pos % 128 + 1)[None, :, None])
    n = (keys * valid).sum(-1)                       # [Hidx, T]
    return n


def alg_flops(st, n_keys):
    w = st["w"]
    cfg = w.cfg
    heads_per_idx = cfg.Hq // cfg.Hidx
    return 4.0 * cfg.D * heads_per_idx * float(n_keys.sum().item())


def executed_flops(st):
    """FLOPs the union-tile kernel issues: a CTA holds two 128-row tiles
    (2 x 128/G tokens x the G heads of one kv head) that walk the union of
    their rows' selections, 128 x 128 x 128 x 4 per tile per union block."""
    import torch
    w = st["w"]
    cfg = w.cfg
    G = cfg.Hq // cfg.Hkv
    toks = 256 // G
    ids = st["ids"]
    T = w.T
    hpi = cfg.Hq // cfg.Hidx
    total = 0
    nblk = (T + 127) // 128
    for g in range(cfg.Hkv):
        i0, i1 = (g * G) // hpi, (g * G + G - 1) // hpi
        sel = ids[i0:i1 + 1]                                          # [ni, T, topk]
        ntile = (T + toks - 1) // toks
        pad = ntile * toks - T
        s = sel.permute(1, 0, 2).reshape(T, -1)
        if pad:
            s = torch.cat([s, torch.full((pad, s.shape[1]), -1, dtype=s.dtype, device=s.device)])
        s = s.reshape(ntile, -1).long()
        onehot = torch.zeros((ntile, nblk + 1), dtype=torch.bool, device=s.device)
        onehot.scatter_(1, torch.where(s >= 0, s, nblk), True)
        total += int(onehot[:, :nblk].sum().item())
    return total * 2 * 128.0 * 128 * 128 * 4


def decode_bytes(st):
    """Algorithmic HBM bytes of one decode step: index-K pages scored (blocks
    before each query's own block) + K and V pages of each (sequence, kv
    head)'s union of selected blocks + the small q / output / table traffic."""
    import torch
    w = st["w"]
    cfg = w.cfg
    own = (st["sl"].long() - 1) // 128
    idx_bytes = float(own.sum().item()) * 128 * cfg.d_idx
    G = cfg.Hq // cfg.Hkv
    hpi = cfg.Hq // cfg.Hidx
    ids = st["ids"].long()
    maxb = int(w.page_table.shape[1])
    union = 0
    for g in range(cfg.Hkv):
        i0, i1 = (g * G) // hpi, (g * G + G - 1) // hpi
        s = ids[i0:i1 + 1].permute(1, 0, 2).reshape(ids.shape[1], -1)
        oh = torch.zeros((s.shape[0], maxb + 1), dtype=torch.bool, device=s.device)
        oh.scatter_(1, torch.where(s >= 0, s, maxb), True)
        union += int(oh[:, :maxb].sum().item())
    kv_bytes = union * 2.0 * 128 * cfg.D
    small = w.T * (cfg.Hq * cfg.D * 3 + cfg.Hidx * cfg.d_idx * 3 + cfg.Hq * 2 * cfg.D + 8 * cfg.Hq)
    return idx_bytes + kv_bytes + small, kv_bytes, union


def mla_measure(msa, wl, dev, steps, flush, pk, only=None):
    """Sparse-MLA prefill workload: quantise Q + MLA kernel per step (with
    `only` = n: just run the step n times, untimed)."""
    import numpy as np
    import torch
    w = wl.make_mla(wl.CONFIGS["mla"])
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q = bf(w.q)
    kv8 = msa.quant_fp8(bf(w.kv), w.scales["kv"])
    idx, tl, sink = t(w.indices), t(w.topk_length), t(w.sink)
    T, H = w.q.shape[0], w.q.shape[1]
    q8 = torch.empty(w.q.shape, dtype=torch.uint8, device=dev)
    o = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    ml = torch.empty((T, H), dtype=torch.float32, device=dev)
    ls = torch.empty((T, H), dtype=torch.float32, device=dev)

    def step():
        msa.quant_fp8(q, w.scales["q"], out=q8)
        msa.sparse_mla_fwd(q8, kv8, idx, tl, sink, w.sm_scale, w.scales["q"], w.scales["kv"],
                           out=o, max_logits=ml, lse=ls)

    cs = t(wl.rotary_table(w.cfg.S_kv, 64))
    pos = t((np.arange(T) + w.cfg.S_kv - T).astype(np.int32))
    rq = lambda: msa.rope_quant_fp8(q[..., :512], q[..., 512:], cs, pos, is_neox=True,
                                    scale=w.scales["q"], out=q8)
    if only is not None:
        for _ in range(only):
            step()
        for _ in range(only):
            rq()
        torch.cuda.synchronize()
        msa.check_errors()
        return None
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    kern = []
    msa.profile_enable(False)                  # timed steps as a caller runs them, queued
    ms = _queued_ms(step, steps, flush)
    msa.profile_enable(True)                   # the MLA kernel alone
    for _ in range(steps):
        flush()
        step()
        kern.append(msa.profile_last_ms())
    msa.check_errors()
    # the fused producer of the same q: rotary embedding of q[..., 512:] and
    # e4m3 of nope || rope(pe), one launch per step
    for _ in range(3):
        rq()
    torch.cuda.synchronize()
    r_ms = _queued_ms(rq, steps, flush)
    msa.check_errors()
    r_bytes = 3 * q.numel() + 4 * T * (64 + 1)
    rm = statistics.mean(r_ms)
    rope = {"kernel": "rope_quant_kernel", "rows": T, "heads": H, "d_nope": 512, "d_rope": 64, "ms": rm,
            "gbs": r_bytes / (rm / 1e3) / 1e9, "frac_of_hbm": r_bytes / (rm / 1e3) / 1e9 / pk["hbm_gbs"],
            "algorithmic_bytes": r_bytes, "traffic": traffic_for("quant.cu", "rope_quant_kernel_mla_q.md")}
    flops = float(np.sum(w.topk_length.astype(np.float64))) * H * (2 * 576 + 2 * 512)
    k = statistics.mean(kern)
    fp8_peak = 2.0 * pk["bf16_tflops"]
    return {"workload": "mla", "queries": T, "heads": H, "ms_per_step": statistics.mean(ms),
            "tokens_per_s": T / (statistics.mean(ms) / 1e3),
            "kernel": "mla_prefill_kernel", "kernel_ms": k, "tflops_algorithmic": flops / (k / 1e3) / 1e12,
            "frac_of_fp8_peak": flops / (k / 1e3) / 1e12 / fp8_peak, "algorithmic_flop": flops,
            "traffic": traffic_for("mla.cu", "mla_prefill_kernel_mla.md"),
            "peak_basis": f"{pk['source']} bf16 burst x2", "rope_quant": rope}


def kv_store_measure(msa, w, dev, steps, flush, pk, only=None):
    """The quantised KV-cache store of a workload's new tokens (K, V and index
    K of every query row into the paged e4m3 pools), one launch per step
    (with `only` = n: just run it n times, untimed)."""
    import numpy as np
    import torch
    c = w.cfg
    T = w.T
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    g = torch.Generator(device="cpu").manual_seed(7)
    k = (torch.randn((T, c.Hkv, c.D), generator=g) * 2).to(torch.bfloat16).to(dev)
    v = (torch.randn((T, c.Hkv, c.D), generator=g) * 2).to(torch.bfloat16).to(dev)
    ik = (torch.randn((T, c.d_idx), generator=g) * 2).to(torch.bfloat16).to(dev)
    kc = torch.zeros((w.num_pages, c.Hkv, 128, c.D), dtype=torch.uint8, device=dev)
    vc, ic = torch.zeros_like(kc), torch.zeros((w.num_pages, 128, c.d_idx), dtype=torch.uint8, device=dev)
    pt, sl, cu = t(w.page_table), t(w.seq_lens), t(w.cu_q)

    def step():
        msa.kv_store_fp8(pt, sl, cu, kc, vc, ic, k=k, v=v, idx_k=ik,
                         k_scale=w.scales["k"], v_scale=w.scales["v"], idx_k_scale=w.scales["idx_k"])

    if only is not None:
        for _ in range(only):
            step()
        torch.cuda.synchronize()
        msa.check_errors()
        return None
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ms = _queued_ms(step, steps, flush)
    msa.check_errors()
    # algorithmic bytes: 2 B read + 1 B written per element, plus the batch description
    elems = T * (2 * c.Hkv * c.D + c.d_idx)
    nbytes = 3 * elems + 4 * (w.page_table.size + w.seq_lens.size + w.cu_q.size)
    m = statistics.mean(ms)
    del kc, vc, ic, k, v, ik
    return {"workload": c.name, "tokens": T, "kernel": "kv_store_kernel", "ms": m,
            "gbs": nbytes / (m / 1e3) / 1e9, "frac_of_hbm": nbytes / (m / 1e3) / 1e9 / pk["hbm_gbs"],
            "algorithmic_bytes": nbytes, "peak_basis": pk["source"],
            "traffic": traffic_for("quant.cu", "kv_store_kernel_prefill32k.md") if c.name == "prefill32k" else None}


# ----------------------------------------------------------------- CPU oracle
def oracle_codes(w):
    from oracle import quant as oq
    return (oq.quantize(w.k_pool, w.scales["k"]), oq.quantize(w.v_pool, w.scales["v"]),
            oq.quantize(w.idx_k_pool, w.scales["idx_k"]))


def oracle_sample(w, caches, budget_s, order_seed=0, max_tokens=None):
    """Time the oracle over the whole path for a deterministic sample of query
    tokens until `budget_s` seconds of wall time. Returns (tokens, seconds, cores)."""
    import numpy as np
    from oracle import quant as oq, index_topk as oi, attention as oa
    k8, v8, ik8 = caches
    cfg = w.cfg
    T = w.T
    order = np.random.default_rng(order_seed).permutation(T)
    if max_tokens is not None:
        order = order[:max_tokens]
    q8 = np.zeros((T, cfg.Hq, cfg.D), np.uint8)
    iq8 = np.zeros((T, cfg.Hidx, cfg.d_idx), np.uint8)
    ids = np.full((cfg.Hidx, T, cfg.topk), -1, np.int32)
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    done = 0
    for t in order:
        tt = np.array([t])
        q8[t] = oq.quantize(w.q[t], w.scales["q"])
        iq8[t] = oq.quantize(w.idx_q[t], w.scales["idx_q"])
        sel, _ = oi.index_topk(iq8, ik8, w.page_table, w.seq_lens, w.cu_q, cfg.topk, tokens=tt)
        ids[:, t] = sel[:, 0]
        oa.sparse_attention(q8, k8, v8, w.page_table, w.seq_lens, w.cu_q, ids, w.sink, w.sm_scale,
                            w.scales["q"], w.scales["k"], w.scales["v"], tokens=tt)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    wall = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu = (r1.ru_utime - r0.ru_utime) + (r1.ru_stime - r0.ru_stime)
    return done, wall, max(1, round(cpu / max(wall, 1e-9)))


# ----------------------------------------------------------------- arms
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def world_max(ms: float, world: int, device=None) -> float:
    """Largest per-rank duration over the job (the slowest replica sets the
    job's time); the process group must be initialised when world > 1."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, steps: int, job_ms: float) -> float:
    """Whole-job throughput: every replica processes its own units each step."""
    return units_per_rank * world * steps / (job_ms / 1e3)


def reference_arm(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from fp8_block_sparse_gb300 import workloads as wl
    w = wl.make_gqa(wl.CONFIGS[WORKLOAD])
    caches = oracle_codes(w)
    per_step = 4.0
    for k in range(args.warmup):
        oracle_sample(w, caches, 0.5, order_seed=1000 + k)
    toks, secs, cores = 0, 0.0, 1
    for k in range(args.steps):
        n, s, c = oracle_sample(w, caches, per_step, order_seed=k)
        toks += n
        secs += s
        cores = max(cores, c)
    value = toks / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": w.T, "Hq": 16, "Hkv": 2, "Hidx": 4, "head_dim": 128,
                   "topk": 64, "page": 128},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{toks} query tokens (whole path per token), {per_step:.0f} s per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _e2e(msa, st, args, world, dev, h2d, d2h, barrier, T):
    """End to end through the public API with host buffers: each step copies
    its Q and idx_q in from pinned host memory, runs the path and copies O,
    lse and max_logit back. The copies run on two copy streams (in and out)
    against double-buffered device inputs and outputs, so step k+1's inputs
    arrive and step k-1's outputs leave while step k computes; the timed
    region runs from before the first copy in to after the last copy out,
    after one untimed pass through both buffer sets."""
    import torch
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    bufs = [{k: st[k] for k in ("q", "iq", "o", "lse", "ml")},
            {k: torch.empty_like(st[k]) for k in ("q", "iq", "o", "lse", "ml")}]
    outs = [{"o": st["o_host"], "lse": st["lse_host"], "ml": st["ml_host"]},
            {k: torch.empty_like(st[k + "_host"]).pin_memory() for k in ("o", "lse", "ml")}]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # untimed warm-up of both buffer sets: the first DMA to or from a pinned
    # buffer maps its pages (several ms for 134 MB), which no step pays again
    for b in range(2):
        bufs[b]["q"].copy_(st["q_host"], non_blocking=True)
        bufs[b]["iq"].copy_(st["iq_host"], non_blocking=True)
        run_path(msa, dict(st, **bufs[b]))
        for key in ("o", "lse", "ml"):
            outs[b][key].copy_(bufs[b][key], non_blocking=True)
    torch.cuda.synchronize()
    e0.record(comp)
    up.wait_stream(comp)
    down.wait_stream(comp)

    def copy_in(k):
        b = k % 2
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(ev_done[b])          # step k-2 has read buffer b's inputs
            bufs[b]["q"].copy_(st["q_host"], non_blocking=True)
            bufs[b]["iq"].copy_(st["iq_host"], non_blocking=True)
            ev_in[b].record(up)

    copy_in(0)
    for k in range(args.steps):
        b = k % 2
        if k + 1 < args.steps:
            copy_in(k + 1)
        comp.wait_event(ev_in[b])
        if k >= 2:
            comp.wait_event(ev_out[b])             # step k-2's outputs have left buffer b
        run_path(msa, dict(st, **bufs[b]))
        ev_done[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[b])
            for key in ("o", "lse", "ml"):
                outs[b][key].copy_(bufs[b][key], non_blocking=True)
            ev_out[b].record(down)
    comp.wait_stream(down)
    e1.record(comp)
    barrier()
    e2e_ms = world_max(e0.elapsed_time(e1), world, dev)
    return {"value": job_throughput(T, world, args.steps, e2e_ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "two copy streams, double-buffered device inputs and outputs",
            "host_copy_gbs": _host_copy_rates(st)}


def _host_copy_rates(st):
    """This box's pinned-memory copy rates on the step's own buffers (one
    H2D of Q and one D2H of O, timed alone): the context of the e2e number,
    which such rates bound from below."""
    import torch
    a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize()
    a.record()
    st["q"].copy_(st["q_host"], non_blocking=True)
    b.record()
    st["o_host"].copy_(st["o"], non_blocking=True)
    c.record()
    torch.cuda.synchronize()
    return {"h2d": st["q_host"].numel() * 2 / (a.elapsed_time(b) / 1e3) / 1e9,
            "d2h": st["o_host"].numel() * 2 / (b.elapsed_time(c) / 1e3) / 1e9}


def native_arm(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    import fp8_block_sparse_gb300 as msa
    from fp8_block_sparse_gb300 import workloads as wl
    msa.load()
    pk = peaks()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    if args.only is not None:
        # one part of the path, untimed, for profiler captures
        n = args.warmup + args.steps
        if args.only == "mla":
            mla_measure(msa, wl, dev, 0, None, pk, only=n)
        elif args.only == "kv_store":
            kv_store_measure(msa, wl.make_gqa(wl.CONFIGS[args.workload]), dev, 0, None, pk, only=n)
        else:
            part = gqa_setup(msa, wl, args.workload if args.only == "prefill" else "decode", dev)
            for _ in range(n):
                run_path(msa, part)
            torch.cuda.synchronize()
            msa.check_errors()
        return 0

    st = gqa_setup(msa, wl, args.workload, dev, pinned=True)
    flush = L2Flush(dev)
    msa.profile_enable(True)
    # no garbage-collector pause inside a timed region: a pause between two
    # calls of a step leaves the GPU idle inside the step's events
    gc.collect()
    gc.disable()
    for _ in range(max(3, args.warmup)):
        run_path(msa, st)
    torch.cuda.synchronize()
    msa.check_errors()

    # ---- device-timed region: inputs resident, L2 flushed before every step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    cuts = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    attn_ms = []
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    clocks = Clocks(gpu_id)
    clocks.start()
    barrier()
    # the timed steps run as a caller runs them: no event between the calls
    # (an event recorded between two launches ends their programmatic
    # overlap), the library's profile events off
    msa.profile_enable(False)
    s = torch.cuda.current_stream()
    for k in range(args.steps):
        flush()
        ev[k][0].record(s)
        run_path(msa, st)
        ev[k][1].record(s)
    barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = world_max(sum(step_ms), world, dev)
    msa.check_errors()

    # ---- where a step's time goes: the same steps again, with events between
    # the calls and the library's events around the attention kernel
    msa.profile_enable(True)
    for k in range(args.steps):
        flush()
        c = cuts[k]
        c[0].record(s)
        msa.quant_fp8_multi([(st["q"], st["w"].scales["q"], st["q8"]),
                             (st["iq"], st["w"].scales["idx_q"], st["iq8"])])
        c[1].record(s)
        w = st["w"]
        msa.index_topk(st["iq8"], st["ik8"], st["pt"], st["sl"], st["cu"], w.cfg.topk, w.max_q_len,
                       out=st["ids"], workspace=st["ws_idx"])
        c[2].record(s)
        msa.sparse_attn_fwd(st["q8"], st["k8"], st["v8"], st["pt"], st["sl"], st["cu"], st["ids"],
                            st["sink"], w.sm_scale, w.scales["q"], w.scales["k"], w.scales["v"],
                            w.max_q_len, out=st["o"], max_logit=st["ml"], lse=st["lse"],
                            workspace=st["ws_attn"])
        c[3].record(s)
        attn_ms.append(msa.profile_last_ms())
    quant_ms = statistics.mean(c[0].elapsed_time(c[1]) for c in cuts)
    index_ms = statistics.mean(c[1].elapsed_time(c[2]) for c in cuts)
    attn_call_ms = statistics.mean(c[2].elapsed_time(c[3]) for c in cuts)
    kern_ms = statistics.mean(attn_ms)
    msa.check_errors()

    # ---- the quantiser's kernel alone (library events around its launch;
    # the step's quantise breakdown above also holds the host time of the call)
    qk_ms = []
    for _ in range(args.steps):
        flush()
        msa.quant_fp8_multi([(st["q"], st["w"].scales["q"], st["q8"]),
                             (st["iq"], st["w"].scales["idx_q"], st["iq8"])])
        qk_ms.append(msa.profile_last_ms())
    msa.check_errors()
    # ---- the index step's kernels alone (scoring through selection)
    ik_ms = []
    for _ in range(args.steps):
        flush()
        w = st["w"]
        msa.index_topk(st["iq8"], st["ik8"], st["pt"], st["sl"], st["cu"], w.cfg.topk, w.max_q_len,
                       out=st["ids"], workspace=st["ws_idx"])
        ik_ms.append(msa.profile_last_ms())
    msa.check_errors()
    q_bytes = 3.0 * (st["q"].numel() + st["iq"].numel())
    qk = statistics.mean(qk_ms)
    quant_kernel = {"kernel": "quant_multi_kernel", "ms": qk, "algorithmic_bytes": q_bytes,
                    "gbs": q_bytes / (qk / 1e3) / 1e9, "frac_of_hbm": q_bytes / (qk / 1e3) / 1e9 / pk["hbm_gbs"],
                    "traffic": traffic_for("quant.cu", "quant_multi_kernel_prefill32k.md")}

    T = st["w"].T
    value = job_throughput(T, world, args.steps, total_ms)
    n_keys = selected_keys(st)
    flops = alg_flops(st, n_keys)
    exe = executed_flops(st)
    fp8_peak = 2.0 * pk["bf16_tflops"]
    achieved = flops / (kern_ms / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
            "frac": achieved / fp8_peak,
            "traffic": traffic_for("attn.cu", "attn_prefill_kernel_prefill32k.md"),
            "kernel": "attn_prefill_kernel",
            "peak_basis": f"{pk['source']} bf16 burst {pk['bf16_tflops']:.0f} TF/s x2 (nominal fp8/bf16 ratio)",
            "algorithmic_flop_per_launch": flops, "executed_flop_per_launch": exe,
            "executed_tflops": exe / (kern_ms / 1e3) / 1e12, "kernel_ms": kern_ms}

    # ---- end to end through the public API with host buffers
    h2d = st["q_host"].numel() * 2 + st["iq_host"].numel() * 2
    d2h = st["o_host"].numel() * 2 + st["lse_host"].numel() * 4 + st["ml_host"].numel() * 4
    e2e = None
    msa.profile_enable(False)          # end to end as a caller runs it
    barrier()
    if not args.no_e2e:
        e2e = _e2e(msa, st, args, world, dev, h2d, d2h, barrier, T)

    # ---- the quantised KV-cache store of this workload's new tokens
    kv_store = [kv_store_measure(msa, st["w"], dev, args.steps, flush, pk)]

    # ---- paged decode workload: HBM GB/s
    decode = None
    if not args.no_decode:
        del st
        torch.cuda.empty_cache()
        ds = gqa_setup(msa, wl, "decode", dev)
        for _ in range(3):
            run_path(msa, ds)
        torch.cuda.synchronize()
        d_kern = []
        msa.profile_enable(False)                  # timed steps as a caller runs them, queued
        d_ms = _queued_ms(lambda: run_path(msa, ds), args.steps, flush)
        msa.profile_enable(True)                   # the attention kernel alone
        for k in range(args.steps):
            flush()
            run_path(msa, ds)
            d_kern.append(msa.profile_last_ms())
        msa.check_errors()
        # the same step captured once as a CUDA graph (quantise -> index top-k
        # -> attention chained without host work between launches) and replayed
        msa.profile_enable(False)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run_path(msa, ds)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run_path(msa, ds)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        g_ms = _queued_ms(graph.replay, args.steps, flush)
        msa.check_errors()
        del graph
        msa.profile_enable(True)
        kv_store.append(kv_store_measure(msa, ds["w"], dev, args.steps, flush, pk))
        total_b, kv_b, union = decode_bytes(ds)
        step_ms_d = statistics.mean(d_ms)
        kern_d = statistics.mean(d_kern)
        step_ms_g = statistics.mean(g_ms)
        decode = {"workload": "decode", "batch": ds["w"].T, "ms_per_step": step_ms_d,
                  "tokens_per_s": ds["w"].T / (step_ms_d / 1e3),
                  "hbm_gbs": total_b / (step_ms_d / 1e3) / 1e9,
                  "frac_of_hbm": total_b / (step_ms_d / 1e3) / 1e9 / pk["hbm_gbs"],
                  "attn_kernel": {"kernel": "attn_decode_kernel", "ms": kern_d,
                                  "gbs": kv_b / (kern_d / 1e3) / 1e9,
                                  "frac_of_hbm": kv_b / (kern_d / 1e3) / 1e9 / pk["hbm_gbs"],
                                  "traffic": traffic_for("attn.cu", "attn_decode_kernel_decode.md")},
                  "algorithmic_bytes_per_step": total_b, "kv_union_blocks": union,
                  "peak_hbm_gbs": pk["hbm_gbs"], "peak_basis": pk["source"],
                  "graph_replay": {"ms_per_step": step_ms_g, "tokens_per_s": ds["w"].T / (step_ms_g / 1e3),
                                   "hbm_gbs": total_b / (step_ms_g / 1e3) / 1e9}}
        del ds

    mla = None
    if not args.no_mla:
        torch.cuda.empty_cache()
        mla = mla_measure(msa, wl, dev, args.steps, flush, pk)

    gc.enable()

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        w = wl.make_gqa(wl.CONFIGS[args.workload])
        caches = oracle_codes(w)
        n, secs, cores = oracle_sample(w, caches, args.cpu_seconds)
        cpu = {"value": n / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n} query tokens of {args.workload} (quantise, index top-k, attention), {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": args.workload, "tokens": T, "Hq": 16, "Hkv": 2, "Hidx": 4, "head_dim": 128,
                       "d_idx": 128, "topk": 64, "page": 128, "parallelism": f"replicas x{world}",
                       "l2": "flushed before every timed step: 256 MB write, then 256 MB read (the step starts with clean lines, so the flush's write-back is not charged to it)"},
            "roofline": roof,
            "prefill_tflops_algorithmic": flops / (total_ms / args.steps / 1e3) / 1e12,
            "breakdown_ms": {"quant": quant_ms, "index_topk": index_ms, "attention_call": attn_call_ms,
                             "attention_kernel": kern_ms},
            "quant_kernel": quant_kernel,
            "index_kernels_ms": statistics.mean(ik_ms),
            "decode": decode,
            "mla": mla,
            "kv_store": kv_store,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": LAUNCHES_PREFILL * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    return native_arm(args)


if __name__ == "__main__":
    sys.exit(main())
