#!/usr/bin/env python
"""Benchmark: query-tokens/s of one DSA layer group with IndexShare on GB300.

A step is one indexshare_group_forward call (every hot-path step: indexer
scoring and top-K on F layers, gather + sparse MLA on every layer) over one
batch of seeded synthetic inputs already resident in HBM.  Default workload:
the 8192-token causal prefill, layers F,S,S,S, H=64, K=2048.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   (the CPU oracle, timed on a sample)

Rank 0 prints one JSON line.  Under torchrun (N > 1) every rank runs its own
replica of the workload (no data-path collective); value = all ranks' query
tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "query-tokens/s per 4-layer F+3S DSA group (prefill & decode); % TC/HBM roofline"
UNIT = "query-tokens/s"
DESCR = {
    "tiny": "tiny prefill: 1 sequence, T=512 causal, layers FSSS, H=16, K=64, integer-valued bf16",
    "prefill8k": "prefill 8K: 1 sequence, T=8192 causal, layers FSSS, H=64, latent 512 + rope 64, "
                 "indexer 32x128, K=2048, bf16 N(0,1)/sqrt(d)",
    "decode64": "decode: 64 sequences x 1 query, context U[98304,131072], layers FSSS, H=64, K=2048, bf16",
    "chunked": "chunked prefill: 4096 queries after a 131072-token prefix, layers FSSSFSSS, H=64, "
               "K=2048, bf16",
    "decode1m": "1M decode: 4 sequences x 1 query, context 1048576, layers FSSS, H=64, K=2048, "
                "FP8 E4M3 + Hadamard indexer keys/queries",
    "prefill2k": "profiling case: prefill of 2560 tokens, layers FSSS, H=64, K=2048, bf16",
    "chunked1k": "profiling case: chunked prefill of 1024 queries after a 131072-token prefix, "
                 "layers FSSS, H=64, K=2048, bf16",
    "decode8": "profiling case: decode of 8 sequences x 1 query, context U[98304,131072], FSSS, "
               "H=64, K=2048, bf16",
}
# ncu DRAM traffic of the dominant kernel (bytes per launch), with the hash of
# the kernel sources it was measured on; ignored once the sources change.
NCU_TRAFFIC = {
    # ncu dram read+write of sparse_mla_persistent_kernel<64, 0> on the 2560-token prefill launch
    # (204.5 MB read + 124.5 MB written), scaled by tokens to the 8192-token launch (q/out
    # traffic is per token; the kv cache is a few MB)
    "sparse_mla": {"bytes": 1.0529e+09, "workload": "prefill8k", "src": "8d356aa34dc94187"},
}

def kernel_src_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "dsa_indexer_indexshare_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KSRC = {"sparse_mla": ["sparse_mla.cu", "ptx.cuh", "common.cuh"],
        "indexer": ["indexer.cu", "ptx.cuh", "common.cuh"],
        "topk": ["topk.cu", "ptx.cuh", "common.cuh"]}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


# a timed region shorter than this runs at the burst clock; longer ones settle
# under the power cap, so their tensor-bound kernels are graded against the
# sustained peak
SUSTAINED_AFTER_S = 3.0


def measure_fp8_peak(dev):
    """Dense E4M3 x E4M3 -> bf16 GEMM throughput (TFLOP/s, best of 10
    8192^3 products through cuBLASLt), the denominator of a tensor-bound FP8
    indexer; None where the library call is unavailable."""
    import torch
    try:
        n = 8192
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        return round(2.0 * n ** 3 / (best / 1e3) / 1e12, 1)
    except Exception:  # noqa: BLE001 - report the nominal ratio instead
        return None


# ---------------------------------------------------------------- algorithmic work
def algorithmic(lay, cfg, fp8, kv_row_bytes=1152):
    """Per-launch algorithmic FLOPs / bytes of each kernel for this layout."""
    pos = lay.q_pos.astype(np.int64)
    vis = pos + 1
    H, K = cfg["H"], cfg["K"]
    nvalid = np.minimum(vis, K)
    # keys scanned by the indexer: every visible position of each query
    # (decode: one query per sequence, so each key row is read once)
    idx_flops = 2.0 * 32 * 128 * vis.sum()
    kbytes_per_pos = 128 * (1 if fp8 else 2) + (4 if fp8 else 0)
    seq_len = np.array([lay.q_pos[lay.q_start[b + 1] - 1] + 1 if lay.q_start[b + 1] > lay.q_start[b]
                        else 0 for b in range(lay.num_seqs)], np.int64)
    # prefill rows beyond 16K positions take the select-only F layer (the
    # library's rule): no score matrix; the top-K reads each row's sampled
    # scores and its candidate list (at least K keys and positions: counted as
    # 2K) and writes K indices
    max_q = int(np.diff(lay.q_start).max()) if lay.num_seqs else 0
    select_only = max_q > 1 and 16384 < lay.max_len <= 2 * 1024 * 1024
    idx_bytes = (seq_len.sum() * kbytes_per_pos + lay.num_q * 32 * (128 * (1 if fp8 else 2) + 4)
                 + (0 if select_only else vis.sum() * 4))
    if select_only:
        tiles = (vis - 1) // 128 + 1
        sampled = np.minimum(tiles, np.clip(tiles // 64, 32, 64)) * 128
        topk_bytes = (sampled * 4).sum() + lay.num_q * (2 * K * 8 + K * 4)
    else:
        topk_bytes = vis.sum() * 4 + lay.num_q * K * 4
    mla_flops = 2.0 * H * (576 + 512) * nvalid.sum()
    # distinct cache rows a launch must read: per sequence, at most its length
    rows_read = sum(min(int(nvalid[lay.q_start[b]:lay.q_start[b + 1]].sum()), int(seq_len[b]))
                    for b in range(lay.num_seqs))
    mla_bytes = rows_read * kv_row_bytes + lay.num_q * H * (576 + 512) * 2
    return {"indexer": {"flops": idx_flops, "bytes": float(idx_bytes)},
            "topk": {"flops": 0.0, "bytes": float(topk_bytes)},
            "sparse_mla": {"flops": mla_flops, "bytes": float(mla_bytes)}}


def tensor_peak(peaks, fp8_indexer=False, timed_s=0.0):
    """(TFLOP/s, description) of the tensor-core peak a kernel is graded
    against: the burst bf16 GEMM for a timed region shorter than
    SUSTAINED_AFTER_S, the sustained one otherwise; for the FP8 indexer the
    measured E4M3 GEMM, else the bf16 peak times the nominal 2x ratio."""
    sustained = timed_s >= SUSTAINED_AFTER_S
    bf16 = peaks["bf16_sustained"] if sustained else peaks["bf16"]
    kind = "sustained" if sustained else "burst"
    if not fp8_indexer:
        return bf16, f"{peaks['src']} {kind} bf16 GEMM"
    if peaks.get("fp8"):
        f = peaks["fp8"] * (peaks["bf16_sustained"] / peaks["bf16"] if sustained else 1.0)
        return f, f"measured E4M3 GEMM ({kind})"
    return 2.0 * bf16, f"{peaks['src']} {kind} bf16 GEMM x 2 (nominal FP8 ratio)"


def kernel_bound(name, work, peaks, fp8, timed_s=0.0):
    """Roofline bound of a kernel: whichever of tensor / HBM time is larger.
    Returns (bound, peak, unit, peak description)."""
    tc, tc_src = tensor_peak(peaks, fp8 and name == "indexer", timed_s)
    t_tc = work["flops"] / (tc * 1e12) if work["flops"] else 0.0
    t_hbm = work["bytes"] / (peaks["hbm"] * 1e9)
    if t_tc >= t_hbm:
        return "tensor", tc, "TFLOP/s", tc_src
    return "hbm", peaks["hbm"], "GB/s", f"{peaks['src']} HBM copy"


def step_units(types, steps):
    """Work units in the timed steps: an F layer for the indexer and the
    top-K (whatever number of launches it takes: the select-only F layer of
    long prefill rows is a sample, a capture and a resolve launch), a layer
    for the sparse MLA."""
    nf = types.count("F")
    return {"indexer": nf * steps, "topk": nf * steps, "sparse_mla": len(types) * steps}


def kernel_records(prof, work, peaks, fp8, timed_s, c2c_gbs=None, units=None):
    """Per-kernel roofline records from the library's live CUDA-event
    profile of the timed steps.  work[name] is the algorithmic work of one
    unit: of one F layer / layer (units[name] of them were timed) where
    units is given, else of one launch."""
    kernels = {}
    units = units or {}
    for name in ("indexer", "topk", "sparse_mla", "append", "hot_plan", "hot_fetch"):
        if name not in work or name not in prof:
            continue
        ms, n = prof[name]
        if n == 0:
            continue
        u = units.get(name) or n
        avg_s = ms / u / 1e3
        if name == "hot_fetch":  # reads over NVLink-C2C: against the measured host->device copy
            bound, peak, unit, src = "c2c", c2c_gbs, "GB/s", "measured host->device copy"
        else:
            bound, peak, unit, src = kernel_bound(name, work[name], peaks, fp8, timed_s)
        ach = (work[name]["flops"] / avg_s / 1e12) if bound == "tensor" else (
            work[name]["bytes"] / avg_s / 1e9)
        kernels[name] = {"launches": n, "ms_per_launch": round(ms / n, 4), "units": u,
                         "ms_per_unit": round(ms / u, 4), "ms_total": round(ms, 4), "share": None,
                         "bound": bound, "achieved": round(ach, 2), "peak": peak, "unit": unit,
                         "frac": round(ach / peak, 4), "peak_src": src}
    ktot = sum(v["ms_total"] for v in kernels.values())
    for v in kernels.values():
        v["share"] = round(v["ms_total"] / ktot, 4) if ktot else None
    return kernels


def scan_gather_record(kernels, work, peaks):
    """HBM-bound (decode) groups: the index scans and the sparse gathers of
    the timed steps together, algorithmic bytes over their summed times;
    None when either kernel is not HBM-bound."""
    if not all(kernels.get(k, {}).get("bound") == "hbm" for k in ("indexer", "sparse_mla")):
        return None
    byt = sum(work[k]["bytes"] * kernels[k]["units"] for k in ("indexer", "sparse_mla"))
    sec = sum(kernels[k]["ms_total"] / 1e3 for k in ("indexer", "sparse_mla"))
    ach = byt / sec / 1e9
    return {"achieved": round(ach, 1), "peak": peaks["hbm"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm"], 4),
            "what": "indexer scans + sparse-MLA gathers of the timed steps"}


# ---------------------------------------------------------------- replicas
def slowest_rank_ms(ms: float, world: int, device=None) -> float:
    """The largest of every rank's timed milliseconds (replicas report the
    slowest rank's time); a no-op for a single process.  Works with the nccl
    (device tensor) and gloo (host tensor) backends."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank_step: int, steps: int, world: int, slowest_ms: float) -> float:
    """Whole-job query-tokens/s: every replica processes the same workload."""
    return world * tokens_per_rank_step * steps / (slowest_ms / 1e3)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 9]
        if self.bus_id:
            mine = [r for r in rows if self.bus_id.endswith(r[1].lower()[-12:]) or
                    r[1].lower().endswith(self.bus_id[-12:])]
            rows = mine or rows
        idx0 = rows[0][0] if rows else None
        rows = [r for r in rows if r[0] == idx0]
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.strip() == "Active"})
        load = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- inputs
def page_caches(lay, layers, block_rows, dev, seed=0):
    """Move every per-position cache (kv, k_idx, k_scale) into a paged pool:
    each sequence's blocks of block_rows positions go to a seeded random
    permutation of physical blocks.  Returns the block table and the
    physical row of every logical (contiguous) row, on the device."""
    import numpy as np
    import torch
    R = int(block_rows)
    lens = [int(n) for n in lay.seq_len]
    nblk = [(n + R - 1) // R for n in lens]
    bps = (lay.max_len + R - 1) // R
    total = sum(nblk)
    ids = np.random.default_rng(5000 + seed).permutation(total)
    table = np.full((len(lens), bps), -1, np.int32)
    phys = np.empty(lay.rows, np.int64)  # physical row of every logical (contiguous) row
    k = 0
    for b, n in enumerate(lens):
        table[b, :nblk[b]] = ids[k:k + nblk[b]]
        s = np.arange(n)
        phys[int(lay.seq_row0[b]) + s] = table[b, s // R].astype(np.int64) * R + s % R
        k += nblk[b]
    phys_d = torch.from_numpy(phys).to(dev)
    for L in layers:
        for key in ("kv", "k_idx", "k_scale"):
            if key in L:
                src = L[key]
                dst = torch.zeros((total * R,) + tuple(src.shape[1:]), dtype=src.dtype, device=dev)
                dst.index_copy_(0, phys_d, src)
                L[key] = dst
                del src
    torch.cuda.synchronize(dev)
    return table, phys_d


def make_appends(lay, layers, cfg, fp8, batch, dev, theta=8e6):
    """Per F layer, the cache-append work of one step's new tokens: the new
    indexer queries (pre-RoPE, bf16) are rotated (and FP8-quantised) into the
    layer's q_idx, and the new tokens' keys are rotated (and quantised) into
    their cache rows.  Returns the calls and the algorithmic bytes they move."""
    import math

    import torch

    import dsa_indexer_indexshare_gb300 as dsa
    freq = np.power(float(theta), -2.0 * np.arange(32) / 64)
    nq = lay.num_q
    seq = torch.from_numpy(np.repeat(np.arange(lay.num_seqs), np.diff(lay.q_start)).astype(np.int32)).to(dev)
    ws = dsa.workspace(256, dev)
    calls = []
    nbytes = 0.0
    for l, L in enumerate(layers):
        if "q_idx" not in L:
            continue
        g = torch.Generator(device=dev)
        g.manual_seed(9000 + l)
        q_raw = (torch.randn((nq, 32, 128), generator=g, device=dev) / math.sqrt(128)).to(torch.bfloat16)
        k_new = (torch.randn((nq, 128), generator=g, device=dev) / math.sqrt(128)).to(torch.bfloat16)

        def call(L=L, q_raw=q_raw, k_new=k_new):
            dsa.dsa_indexer_prepare_queries(q_raw, batch, freq, fp8=fp8, q_out=L["q_idx"],
                                            q_scale=L.get("q_scale"), ws=ws)
            dsa.dsa_indexer_append_keys(k_new, seq, batch.q_pos, batch, L["k_idx"], freq,
                                        k_scale=L.get("k_scale"), ws=ws)
        calls.append(call)
        out = 128 + 4 if fp8 else 256  # bytes written per vector
        nbytes += nq * 32 * (256 + out) + nq * 4 + nq * (256 + out + 8)
    return calls, nbytes, ws


def setup(workload, dev, seed=0, paged=0, kv_fp8=False):
    import torch

    import dsa_indexer_indexshare_gb300 as dsa
    import synth

    cfg = dict(synth.WORKLOADS[workload])
    lay = synth.workload_layout(workload, seed)
    types = cfg["layers"]
    fp8 = bool(cfg.get("fp8"))
    layers = synth.device_layers(lay, types, cfg["H"], device=dev, seed=seed,
                                 ints=bool(cfg.get("ints")))
    if fp8:  # the FP8 indexer consumes Hadamard-rotated E4M3 codes from the library's quantiser
        for L in layers:
            if "q_idx" in L:
                qc, qs = dsa.dsa_fp8_quantize(L["q_idx"])
                kc, ks = dsa.dsa_fp8_quantize(L["k_idx"])
                L.update(q_idx=qc, q_scale=qs, k_idx=kc, k_scale=ks)
        torch.cuda.synchronize(dev)
    if kv_fp8:  # FP8 KV latent rows (656 B) from the library's quantiser
        for L in layers:
            L["kv"] = dsa.dsa_kv_fp8_quantize(L["kv"])
        torch.cuda.synchronize(dev)
    phys = None
    if paged:
        table, phys = page_caches(lay, layers, paged, dev, seed)
        batch = dsa.Batch(lay.q_start, lay.q_pos, None, lay.max_len, device=dev,
                          block_table=table, block_rows=paged)
    else:
        batch = dsa.Batch(lay.q_start, lay.q_pos, lay.seq_row0, lay.max_len, device=dev)
    return cfg, lay, layers, batch, fp8, phys


def ablation_layers(cfg, layers, types):
    """The layers of a group run as `types`: the workload's own layers, or for
    the every-layer-indexer ablation each layer with the indexer inputs of
    the F layer that leads its group."""
    if types == cfg["layers"]:
        return layers
    out = []
    last_f = None
    for l, c in enumerate(cfg["layers"]):
        if c == "F":
            last_f = layers[l]
        d = dict(layers[l])
        for k_ in ("q_idx", "w", "k_idx", "q_scale", "k_scale"):
            if k_ in last_f:
                d[k_] = last_f[k_]
        out.append(d)
    return out


def make_group_for(dsa, cfg, lay, layers, batch, types, dev):
    """(Group, workspace, index buffer) of one group configuration."""
    import torch
    g = dsa.Group(types, ablation_layers(cfg, layers, types), k=cfg["K"], scale=1 / 16)
    ws = dsa.workspace(g.workspace_size(batch), dev)
    idx = torch.empty((lay.num_q, cfg["K"]), dtype=torch.int32, device=dev)
    return g, ws, idx


def measure_workload(dsa, name, args, dev, peaks, stream, flush):
    """One more workload of the configs, timed like the headline one (device-
    resident inputs, L2 flushed between steps, CUDA events, clocks sampled
    during the timed steps), with its per-kernel roofline records, the
    scan + gather HBM fraction of decode groups and the every-layer-indexer
    ablation.  Its device memory is released before returning."""
    import torch
    cfg, lay, layers, batch, fp8, _ = setup(name, dev)
    steps = max(5, args.steps if cfg["kind"] == "decode" else min(args.steps, 10))
    group, ws, idx = make_group_for(dsa, cfg, lay, layers, batch, cfg["layers"], dev)
    run = lambda: dsa.indexshare_group_forward(group, batch, idx, ws=ws)
    for _ in range(args.warmup):
        run()
        flush()
    dsa.status_fetch(ws)
    torch.cuda.synchronize(dev)
    dsa.launch_counts_reset()
    clk = ClockSampler(getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None))
    clk.start()
    time.sleep(0.3)
    times = time_steps(run, steps, 0, flush, stream)
    clocks = clk.stop()
    launches = sum(dsa.launch_counts().values())
    prof, ms_prof = profile_steps(dsa, run, steps, flush, stream)
    dsa.status_fetch(ws)
    total_ms = sum(times)
    work = algorithmic(lay, cfg, fp8)
    kernels = kernel_records(prof, work, peaks, fp8, total_ms / 1e3,
                             units=step_units(cfg["layers"], steps))
    rec = {"workload": DESCR[name], "value": round(lay.num_q * steps / (total_ms / 1e3), 1),
           "unit": UNIT, "steps": steps, "warmup": args.warmup,
           "ms_per_step": round(total_ms / steps, 4), "ms_per_step_profiled": round(ms_prof, 4),
           "layers": cfg["layers"],
           "dtype": "bf16" + ("+fp8-indexer" if fp8 else ""), "kernels": kernels,
           "scan_gather_hbm": scan_gather_record(kernels, work, peaks), "gpu_launches": launches,
           "clocks": clocks}
    types_all = "F" * len(cfg["layers"])
    g2, ws2, idx2 = make_group_for(dsa, cfg, lay, layers, batch, types_all, dev)
    t2 = time_steps(lambda: dsa.indexshare_group_forward(g2, batch, idx2, ws=ws2), steps,
                    args.warmup, flush, stream)
    dsa.status_fetch(ws2)
    rec["ablation"] = {"layers": types_all, "value": round(lay.num_q * steps / (sum(t2) / 1e3), 1),
                       "ms_per_step": round(sum(t2) / steps, 4),
                       "indexshare_speedup": round(sum(t2) / total_ms, 3)}
    del group, ws, idx, g2, ws2, idx2, layers, batch
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return rec


def profile_steps(dsa, run, steps, flush, stream):
    """Per-kernel durations: `steps` more steps with the library's CUDA events
    recorded around every launch: ({kind: (total_ms, launches)}, the pass's
    ms per step).  Those events cost a 1M-context decode step about a sixth of
    its time, so throughput and ms_per_step come from the plain timed pass
    before this one."""
    dsa.dsa_profile_enable(True)
    try:
        t = time_steps(run, steps, 0, flush, stream)
    finally:
        dsa.dsa_profile_enable(False)
    return dsa.dsa_profile_collect(), sum(t) / steps


def time_steps(run, steps, warmup, flush, stream, after=None):
    import torch
    for _ in range(warmup):
        run()
        flush()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        evs.append((a, b))
        if after is not None:
            after()  # bookkeeping outside the timed events
        flush()  # outside the timed events: L2 is cold at every step
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


# ---------------------------------------------------------------- hot / cold KV
class HotMode:
    """--hot SLOTS: every layer's cache moves to pinned host memory (the cold
    store, read by the GPU over NVLink-C2C); each layer keeps SLOTS hot rows
    per sequence in HBM; one HotState per F layer.  Each step runs
    indexshare_group_forward_hot with the next step number; with
    --hot-rotate R the F layers' indexer queries cycle through R seeded sets."""

    def __init__(self, dsa, args, cfg, lay, layers, batch, fp8, dev):
        import math

        import torch
        self.dsa, self.lay, self.dev, self.slots = dsa, lay, dev, int(args.hot)
        self.rotate = max(1, int(args.hot_rotate))
        self.row_bytes = 656 if args.kv_fp8 else 1152
        types = cfg["layers"]
        self.cold = []
        for L in layers:  # device cache -> pinned host memory, then the hot rows replace it
            h = torch.empty(L["kv"].shape, dtype=L["kv"].dtype, pin_memory=True)
            h.copy_(L["kv"])
            self.cold.append(h)
            shape = (lay.num_seqs * self.slots, L["kv"].shape[1])
            L["kv"] = torch.zeros(shape, dtype=h.dtype, device=dev)
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        # the device reads every host page of the cold store once (setup,
        # outside the timed region); its cost is reported in `hot`
        t0 = time.perf_counter()
        if not args.hot_no_touch:
            dsa.dsa_hot_touch(self.cold, stride=65536, device=dev)
        torch.cuda.synchronize(dev)
        self.touch_s = round(time.perf_counter() - t0, 3) if not args.hot_no_touch else None
        self.spans = [dsa.HotState(lay.num_seqs, self.slots, lay.max_len, dev) for c in types if c == "F"]
        self.hg = dsa.HotGroup(self.spans, self.cold, num_q=lay.num_q, k=cfg["K"], device=dev)
        self.groups = []
        for r in range(self.rotate):
            ls = [dict(L) for L in layers]
            if r > 0:
                g = torch.Generator(device=dev)
                g.manual_seed(7000 + r)
                for L in ls:
                    if "q_idx" in L:
                        q = (torch.randn((lay.num_q, 32, 128), generator=g, device=dev)
                             / math.sqrt(128)).to(torch.bfloat16)
                        if fp8:
                            qc, qs = dsa.dsa_fp8_quantize(q)
                            L.update(q_idx=qc, q_scale=qs)
                        else:
                            L["q_idx"] = q
            self.groups.append(dsa.Group(types, ls, k=cfg["K"], scale=1 / 16))
        self.ws = dsa.workspace(self.groups[0].workspace_size(batch), dev)
        self.idx_buf = torch.empty((lay.num_q, cfg["K"]), dtype=torch.int32, device=dev)
        self.batch = batch
        self.n = 0
        self.fetched = torch.zeros((), dtype=torch.int64, device=dev)
        self.selected = int(np.minimum(lay.q_pos.astype(np.int64) + 1, cfg["K"]).sum()) * len(self.spans)
        self.c2c_gbs = self.measure_c2c()

    def step(self):
        g = self.groups[self.n % self.rotate]
        self.dsa.indexshare_group_forward_hot(g, self.batch, self.hg, self.n, self.idx_buf, ws=self.ws)
        self.n += 1

    def count_reset(self):
        self.fetched.zero_()

    def count(self):
        for s in self.spans:
            self.fetched += s.fetch_count.sum()

    def measure_c2c(self):
        """Host -> device copy rate from pinned memory (1 GiB, copy engine)."""
        import torch
        h = self.cold[0].view(torch.uint8).reshape(-1)
        n = min(h.numel(), 1 << 30)
        d = torch.empty(n, dtype=torch.uint8, device=self.dev)
        for _ in range(2):
            d.copy_(h[:n], non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(4):
            d.copy_(h[:n], non_blocking=True)
        b.record()
        torch.cuda.synchronize(self.dev)
        return round(4 * n / (a.elapsed_time(b) / 1e3) / 1e9, 1)

    def work(self, steps, prof):
        """Algorithmic bytes per launch of the hot kernels: the plan reads the
        index buffer and writes the rows; the swap-in reads the fetched rows
        from host memory (one launch per F span)."""
        fetched = float(self.fetched.item())
        self.fetched_total = fetched
        per_span_layers = len(self.cold) / max(1, len(self.spans))
        nfetch = max(1, prof.get("hot_fetch", (0, 0))[1])
        nplan = max(1, prof.get("hot_plan", (0, 0))[1])
        K = self.idx_buf.shape[1]
        plan_bytes = float(self.lay.num_q * K * 8) * len(self.spans) * steps / nplan
        fetch_bytes = fetched * per_span_layers * self.row_bytes / nfetch
        return {"hot_plan": {"flops": 0.0, "bytes": plan_bytes},
                "hot_fetch": {"flops": 0.0, "bytes": fetch_bytes}}

    def describe(self):
        return (f"hot/cold: {self.slots} hot rows per sequence and layer in HBM, the full caches "
                f"({self.row_bytes} B rows) in pinned host memory read over NVLink-C2C; "
                f"{self.rotate} rotating indexer query set(s)")

    def summary(self, steps, kernels=None):
        fetched = getattr(self, "fetched_total", float(self.fetched.item()))
        sel = self.selected * steps
        fk = (kernels or {}).get("hot_fetch")
        return {"cold_touch_s": self.touch_s,
                "swap_in_gbs": fk["achieved"] if fk else None,
                "swap_in_frac_of_h2d_copy": fk["frac"] if fk else None,
                "slots": self.slots, "rotate": self.rotate, "selected_rows": sel,
                "fetched_rows": int(fetched), "hit_rate": round(1 - fetched / sel, 4) if sel else None,
                "fetched_bytes_per_step": int(fetched * len(self.cold) / max(1, len(self.spans))
                                              * self.row_bytes / steps),
                "h2d_copy_gbs": self.c2c_gbs}


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(workload, lay, layers, cfg, fp8, nrows, seed=1, phys=None):
    """Host copies of a sampled set of query rows (and the caches they read,
    in contiguous order: a paged cache is read back through `phys`)."""
    import torch
    rng = np.random.default_rng(seed)
    nq = lay.num_q
    K = cfg["K"]
    fixed = [r for r in (0, K - 2, K - 1, K, nq - 1) if 0 <= r < nq]
    rest = rng.choice(nq, size=max(0, min(nq, nrows) - len(fixed)), replace=False)
    rows = np.unique(np.concatenate([fixed, rest]).astype(np.int64))[:max(nrows, 1)]

    def hb(t):  # bf16 tensor -> uint16 bits
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    host = []
    rt = torch.as_tensor(rows, device=layers[0]["q_lat"].device)
    for L in layers:
        if phys is not None:
            L = {k: (v.index_select(0, phys) if k in ("kv", "k_idx", "k_scale") else v)
                 for k, v in L.items()}
        if L["kv"].dtype == torch.uint8:  # FP8 KV rows: the oracle reads their dequantised rows
            import oracle
            kv_host = oracle.kv_fp8_dequantize(L["kv"].cpu().numpy())
        else:
            kv_host = hb(L["kv"])
        d = {"q_lat": hb(L["q_lat"].index_select(0, rt)), "q_rope": hb(L["q_rope"].index_select(0, rt)),
             "kv": kv_host}
        if "q_idx" in L:
            if fp8:
                d.update(q_idx=L["q_idx"].index_select(0, rt).cpu().numpy(),
                         q_scale=L["q_scale"].index_select(0, rt).cpu().numpy(),
                         k_idx=L["k_idx"].cpu().numpy(), k_scale=L["k_scale"].cpu().numpy())
            else:
                d.update(q_idx=hb(L["q_idx"].index_select(0, rt)), k_idx=hb(L["k_idx"]))
            d["w"] = L["w"].index_select(0, rt).cpu().numpy()
        host.append(d)
    return rows, host


def run_oracle(lay, host, rows, cfg, fp8):
    import oracle
    pos, key0 = oracle.row_metadata(lay.q_start, lay.q_pos, lay.seq_row0, rows)
    t0 = time.perf_counter()
    oracle.group_forward(cfg["layers"], host, np.arange(len(rows), dtype=np.int32), pos, key0,
                         lay.max_len, cfg["K"], 1 / 16, idx_dtype=1 if fp8 else 0)
    return time.perf_counter() - t0


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill8k", choices=list(DESCR))
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-slots", type=int, default=3,
                    help="buffer sets of the end-to-end leg (uploads / group call / read-back overlap)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=0)
    ap.add_argument("--with-append", action="store_true",
                    help="each step also rotates (and FP8-quantises) the new tokens' indexer "
                         "queries and appends their keys to the caches of every F layer")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="FP8 KV latent caches (656-byte rows: E4M3 latent in four scaled groups, "
                         "bf16 RoPE key)")
    ap.add_argument("--hot", type=int, default=0, metavar="SLOTS",
                    help="hot/cold KV: SLOTS hot rows per sequence in HBM per layer, the full "
                         "caches in pinned host memory, missing rows swapped in every step")
    ap.add_argument("--hot-rotate", type=int, default=1, metavar="R",
                    help="with --hot: step i uses the i mod R-th of R indexer query sets, so "
                         "R > 1 changes the selected rows from step to step")
    ap.add_argument("--hot-no-touch", action="store_true",
                    help="with --hot: skip the one-time device read of every host page of the "
                         "cold store (first swap-ins then pay for first page accesses)")
    ap.add_argument("--extra-workloads", default=None, metavar="NAMES",
                    help="comma-separated workloads timed after the main one, each recorded "
                         "under 'workloads' (default with the prefill8k workload: "
                         "decode64,chunked,decode1m; '' for none; N = 1 only)")
    ap.add_argument("--paged", type=int, default=0, metavar="ROWS",
                    help="paged caches: blocks of ROWS positions (a multiple of 128) in a "
                         "permuted pool, addressed through a block table")
    args = ap.parse_args()

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        return reference_arm(args)

    import torch.distributed as dist
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import dsa_indexer_indexshare_gb300 as dsa
    peaks = load_peaks()
    peaks["fp8"] = measure_fp8_peak(dev)
    if args.extra_workloads is None:
        plain = not (args.hot or args.paged or args.kv_fp8 or args.with_append)
        args.extra_workloads = ("decode64,chunked,decode1m"
                                if args.workload == "prefill8k" and plain else "")
    cfg, lay, layers, batch, fp8, phys = setup(args.workload, dev, paged=args.paged,
                                               kv_fp8=args.kv_fp8)
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.fill_(1)

    def make_group(types):
        return make_group_for(dsa, cfg, lay, layers, batch, types, dev)

    hot = None
    if args.hot:
        hot = HotMode(dsa, args, cfg, lay, layers, batch, fp8, dev)
        group, ws, idx_buf = hot.groups[0], hot.ws, hot.idx_buf
        args.no_ablation = args.no_e2e = args.no_cpu = True  # those legs read device caches
    else:
        group, ws, idx_buf = make_group(cfg["layers"])
    appends, append_bytes, append_ws = ([], 0.0, None)
    if args.with_append:
        appends, append_bytes, append_ws = make_appends(lay, layers, cfg, fp8, batch, dev)

    def run():
        for a in appends:
            a()
        if hot is not None:
            hot.step()
        else:
            dsa.indexshare_group_forward(group, batch, idx_buf, ws=ws)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- timed region
    for _ in range(args.warmup):
        run()
        flush()
    dsa.status_fetch(ws)
    barrier()
    dsa.launch_counts_reset()
    # hot/cold: the hot state advances every step, so its kernels are profiled
    # in the timed pass itself (steps of milliseconds: the events cost ~1 %)
    dsa.dsa_profile_enable(hot is not None)
    try:
        bus = getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None)
    except Exception:
        bus = None
    clk = ClockSampler(bus)
    clk.start()
    time.sleep(0.3)
    barrier()
    wall0 = time.perf_counter()
    if hot is not None:
        hot.count_reset()
    times = time_steps(run, args.steps, 0, flush, stream,
                       after=hot.count if hot is not None else None)
    barrier()
    wall = time.perf_counter() - wall0
    clocks = clk.stop()
    dsa.dsa_profile_enable(False)
    launches = sum(dsa.launch_counts().values())
    if hot is not None:
        prof, ms_prof = dsa.dsa_profile_collect(), sum(times) / args.steps
    else:
        prof, ms_prof = profile_steps(dsa, run, args.steps, flush, stream)
    dsa.status_fetch(ws)

    total_ms = slowest_rank_ms(sum(times), world, dev)
    tokens_per_step = lay.num_q
    value = replica_throughput(tokens_per_step, args.steps, world, total_ms)

    # ---- per-kernel roofline (live CUDA events around each launch)
    work = algorithmic(lay, cfg, fp8, 656 if args.kv_fp8 else 1152)
    if appends:  # two launches (queries, keys) per F layer per step
        work["append"] = {"flops": 0.0, "bytes": append_bytes / (2 * len(appends))}
        dsa.status_fetch(append_ws)
    if hot is not None:
        work.update(hot.work(args.steps, prof))
    kernels = kernel_records(prof, work, peaks, fp8, total_ms / 1e3,
                             hot.c2c_gbs if hot is not None else None,
                             units=step_units(cfg["layers"], args.steps))
    scan_gather = scan_gather_record(kernels, work, peaks)
    # the dominant on-GPU kernel (the hot swap-in is bound by the host link and
    # reported in "hot")
    top = max((k for k in kernels if not k.startswith("hot_")),
              key=lambda k: kernels[k]["ms_total"])
    tk = kernels[top]
    traffic = None
    if top in NCU_TRAFFIC and NCU_TRAFFIC[top].get("src") == kernel_src_hash(KSRC[top]) and \
            NCU_TRAFFIC[top].get("workload") == args.workload:
        traffic = NCU_TRAFFIC[top]["bytes"]
    roofline = {"kernel": top, "bound": tk["bound"], "achieved": tk["achieved"], "peak": tk["peak"],
                "unit": tk["unit"], "frac": tk["frac"], "traffic": traffic,
                "peak_src": tk["peak_src"],
                "units_per_launch": (work[top]["flops"] if tk["bound"] == "tensor" else work[top]["bytes"])}

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
            "ms_per_step_profiled": round(ms_prof, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" + ("+fp8-indexer" if fp8 else "") + ("+fp8-kv" if args.kv_fp8 else ""),
            "data": "synthetic (seeded N(0,1)/sqrt(d) bf16, device-resident)",
            "config": {"workload": DESCR[args.workload], "global_batch": world * tokens_per_step,
                       "seq_len": int(lay.max_len), "layers": cfg["layers"],
                       "parallelism": "replicas" if world > 1 else "single-gpu",
                       "kv_layout": (hot.describe() if hot is not None else
                                     f"paged: blocks of {args.paged} positions, permuted pool, "
                                     "block table" if args.paged else "contiguous"),
                       "kv_dtype": ("FP8 E4M3 latent, 656-byte rows" if args.kv_fp8
                                    else "bf16, 1152-byte rows"),
                       "step": ("indexer query RoPE/FP8 + key cache append per F layer, then the "
                                "group" if args.with_append else "the group forward"),
                       "l2": "flushed between steps (256 MiB write, outside the timed events)",
                       "kernel_times": ("CUDA events around every launch, in the timed steps"
                                        if hot is not None else
                                        "CUDA events around every launch, in a second pass of the "
                                        "same steps (not in the timed pass)")},
            "roofline": roofline, "kernels": kernels, "gpu_launches": launches,
            "scan_gather_hbm": scan_gather, "fp8_peak_tflops": peaks.get("fp8"),
            "hot": hot.summary(args.steps, kernels) if hot is not None else None,
            "clocks": clocks, "wall_s_timed": round(wall, 3)}

    # ---- IndexShare ablation: every layer runs its own indexer
    if not args.no_ablation:
        types_all = "F" * len(cfg["layers"])
        g2, ws2, idx2 = make_group(types_all)
        t2 = time_steps(lambda: dsa.indexshare_group_forward(g2, batch, idx2, ws=ws2),
                        args.steps, args.warmup, flush, stream)
        dsa.status_fetch(ws2)
        v2 = tokens_per_step * args.steps / (sum(t2) / 1e3)
        line["ablation"] = {"layers": types_all, "value": round(world * v2, 1),
                            "ms_per_step": round(sum(t2) / args.steps, 4),
                            "indexshare_speedup": round(sum(t2) / total_ms, 3)}
        del g2, ws2, idx2

    # ---- end to end through the public API with host buffers
    if not args.no_e2e:
        line["e2e"] = e2e_arm(dsa, group, batch, layers, idx_buf, ws, lay, args, dev, stream, world,
                              phys=phys)

    # ---- the other workloads of the configs, each timed the same way (N = 1)
    extras = [w for w in (args.extra_workloads.split(",") if args.extra_workloads else []) if w]
    if extras and world == 1:
        del group, ws, idx_buf
        line["workloads"] = {}
        for name in extras:
            line["workloads"][name] = measure_workload(dsa, name, args, dev, peaks, stream, flush)

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only)
    if not args.no_cpu and rank == 0 and world == 1:
        import oracle
        # at least one query row per host core (the oracle spreads rows over cores)
        nrows = args.cpu_rows or max(oracle.num_threads(), {
            "tiny": 512, "prefill8k": 480, "decode64": 4, "chunked": 24, "decode1m": 1,
            "prefill2k": 48, "decode8": 4, "chunked1k": 24}[args.workload])
        rows, host = oracle_sample(args.workload, lay, layers, cfg, fp8, nrows, phys=phys)
        secs = run_oracle(lay, host, rows, cfg, fp8)
        line["cpu_baseline"] = {"value": round(len(rows) / secs, 3), "unit": UNIT,
                                "cores": oracle.num_threads(), "cpu": cpu_model(), "kind": "oracle",
                                "sample": f"{len(rows)} query rows of the same workload (full group, "
                                          f"all layers), {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def e2e_arm(dsa, group, batch, layers, idx_buf, ws, lay, args, dev, stream, world, phys=None):
    """Same metric through indexshare_group_forward, with every step's inputs
    copied from pinned host memory and the outputs copied back inside the
    timed region.  A step's inputs are its per-query tensors and the cache
    rows of its own tokens (position q_pos[t] of each query: every row for a
    prefill, one row per sequence for a decode step); the rest of each cache
    is state that stays on the device.  Three sets of device buffers, with
    uploads, the group call and the read-back on three streams, let step
    i+1's uploads and step i-1's read-back overlap step i's group call."""
    import torch
    cache_keys = ("kv", "k_idx", "k_scale")
    query_keys = ("q_lat", "q_rope", "q_idx", "w", "q_scale")
    seq_of = np.repeat(np.arange(lay.num_seqs), np.diff(lay.q_start))
    rows_new = (lay.seq_row0[seq_of].astype(np.int64) + lay.q_pos.astype(np.int64))
    rows_dev = torch.from_numpy(rows_new).to(dev)
    if phys is not None:  # paged caches: the physical rows of those positions
        rows_dev = phys.index_select(0, rows_dev)
    NSLOT = max(2, args.e2e_slots)
    slots = []
    for sl in range(NSLOT):
        if sl == 0:
            dl, g, wsl, idx = layers, group, ws, idx_buf
        else:
            dl = [{k_: torch.empty_like(v) if k_ in query_keys else v for k_, v in L.items()}
                  for L in layers]
            g = dsa.Group(group.layer_types, dl, k=group.k, scale=1 / 16)
            wsl = dsa.workspace(g.workspace_size(batch), dev)
            idx = torch.empty_like(idx_buf)
        ups = []  # (pinned host, device destination, rows to scatter or None)
        for L in dl:
            for k_, v in L.items():
                if k_ in query_keys:
                    ups.append((torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v), v, None))
                elif k_ in cache_keys:
                    new_rows = v.index_select(0, rows_dev)
                    ups.append((torch.empty(new_rows.shape, dtype=v.dtype, pin_memory=True).copy_(new_rows),
                                v, torch.empty_like(new_rows)))
        outs_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in g.outs]
        slots.append({"ups": ups, "g": g, "ws": wsl, "idx": idx, "outs_h": outs_h,
                      "up": torch.cuda.Event(), "done": torch.cuda.Event(), "down": torch.cuda.Event()})
    h2d = sum(h.numel() * h.element_size() for h, _, _ in slots[0]["ups"])
    d2h = sum(o.numel() * o.element_size() for o in slots[0]["outs_h"])
    s_up, s_comp, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)

    def step(i):
        sl = slots[i % NSLOT]
        if i >= NSLOT:  # the slot's previous step has been computed and read back
            s_up.wait_event(sl["down"])
        with torch.cuda.stream(s_up):
            for h, d, stage in sl["ups"]:
                if stage is None:
                    d.copy_(h, non_blocking=True)
                else:  # the new tokens' cache rows, then scattered to their rows
                    stage.copy_(h, non_blocking=True)
                    d.index_copy_(0, rows_dev, stage)
            sl["up"].record(s_up)
        s_comp.wait_event(sl["up"])
        dsa.indexshare_group_forward(sl["g"], batch, sl["idx"], ws=sl["ws"], stream=s_comp)
        sl["done"].record(s_comp)
        s_down.wait_event(sl["done"])
        with torch.cuda.stream(s_down):
            for o_h, o_d in zip(sl["outs_h"], sl["g"].outs):
                o_h.copy_(o_d, non_blocking=True)
            sl["down"].record(s_down)

    steps = max(4, args.steps // 2)
    for i in range(NSLOT):
        step(i)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for i in range(NSLOT, NSLOT + steps):
        step(i)
    for sl in slots:  # the end waits for the last read-back of every slot
        s_comp.wait_event(sl["down"])
    b.record(s_comp)
    torch.cuda.synchronize(dev)
    for sl in slots:
        dsa.status_fetch(sl["ws"])
    ms = slowest_rank_ms(a.elapsed_time(b), world, dev)
    return {"value": round(replica_throughput(lay.num_q, steps, world, ms), 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / steps, 3),
            "inputs": "per-query tensors + the cache rows of the step's tokens",
            "pipelining": f"{NSLOT} buffer sets; uploads, group call and read-back on three streams"}


def reference_arm(args):
    """The CPU oracle as the reference arm: each step runs the full group on a
    bounded sample of the workload's query rows."""
    import oracle
    import synth
    cfg = dict(synth.WORKLOADS[args.workload])
    lay = synth.workload_layout(args.workload)
    fp8 = bool(cfg.get("fp8"))
    # at least one query row per host core (the oracle spreads rows over cores)
    nrows = args.cpu_rows or max(oracle.num_threads(), {
        "tiny": 64, "prefill8k": 8, "decode64": 1, "chunked": 4, "decode1m": 1, "prefill2k": 8,
        "decode8": 1, "chunked1k": 4}[args.workload])
    sub, rows, host = reference_inputs(lay, cfg, fp8, nrows)
    for _ in range(args.warmup):
        run_oracle(sub, host, rows, cfg, fp8)
    t = 0.0
    for _ in range(args.steps):
        t += run_oracle(sub, host, rows, cfg, fp8)
    value = len(rows) * args.steps / t
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t / args.steps, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": DESCR[args.workload], "layers": cfg["layers"]},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(),
                         "cpu": cpu_model(),
                         "kind": "oracle",
                         "sample": f"{len(rows)} query rows per step of the same workload"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def reference_inputs(lay, cfg, fp8, nrows):
    """Host inputs for the oracle arm: a sampled set of query rows and the
    caches of their sequences, drawn with the seeded host generator.  Returns
    a sub-layout holding just those sequences, the sampled rows in it, and the
    per-layer host tensors (query tensors hold the sampled rows only)."""
    import oracle
    import synth
    rng = np.random.default_rng(1)
    K = cfg["K"]
    fixed = [r for r in (lay.num_q - 1, K, K - 1) if 0 <= r < lay.num_q]
    pick = rng.choice(lay.num_q, min(nrows, lay.num_q), replace=False)
    rows = np.sort(np.unique(np.concatenate([fixed, pick]))[:nrows]).astype(np.int64)
    seq = np.searchsorted(lay.q_start, rows, side="right") - 1
    useq = list(np.unique(seq))
    lens = [int(lay.q_pos[lay.q_start[b + 1] - 1]) + 1 for b in useq]
    counts = [int(lay.q_start[b + 1] - lay.q_start[b]) for b in useq]
    sub = synth.make_layout(lens, counts)
    sub_rows = np.array([sub.q_start[useq.index(b)] + (r - lay.q_start[b]) for r, b in zip(rows, seq)],
                        np.int64)
    g = synth.HostGen(0)
    n = len(rows)
    host = []
    for l, tch in enumerate(cfg["layers"]):
        base = 100 * (l + 1)
        d = {"q_lat": g.gauss_bf16(base, (n, cfg["H"], 512), 512),
             "q_rope": g.gauss_bf16(base + 1, (n, cfg["H"], 64), 64),
             "kv": np.concatenate([g.gauss_bf16(base + 2, (sub.rows, 512), 512),
                                   g.gauss_bf16(base + 3, (sub.rows, 64), 64)], axis=1)}
        if tch == "F":
            q = g.gauss_bf16(base + 10, (n, 32, 128), 128)
            k = g.gauss_bf16(base + 12, (sub.rows, 128), 128)
            d["w"] = g.gauss_f32(base + 11, (n, 32), 32)
            if fp8:
                qc, qs = oracle.fp8_quantize_rows(q.reshape(-1, 128))
                kc, ks = oracle.fp8_quantize_rows(k)
                d.update(q_idx=qc.reshape(n, 32, 128), q_scale=qs.reshape(n, 32), k_idx=kc,
                         k_scale=ks)
            else:
                d.update(q_idx=q, k_idx=k)
        host.append(d)
    return sub, sub_rows, host


if __name__ == "__main__":
    main()
