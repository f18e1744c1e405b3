#!/usr/bin/env python
"""Benchmark of the packed-sequence varlen causal attention hot path on GB300.

One step = the whole path over one batch of synthetic packs: host packing
planner (next-fit), then per pack the metadata kernel, the forward (contract
check, tile plan, attention) and the backward (contract check, tile plans,
rowsum, dK/dV, dQ).  The batch is the first 16 next-fit packs of 8192 tokens
(segment lengths uniform in [32, 2048], tail padded to 8192), Hq = Hkv = 32,
d = 128, bf16, causal.  Every pack's q/k/v/dO (256 MB) is larger than L2, so
no flush is needed between steps.

Metric: in-segment causal FLOPs per second, fwd 4*d*Hq*E + bwd 10*d*Hq*E with
E = sum over real documents of l(l+1)/2 (the tail pad segment is computed but
not credited), in TFLOP/s.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload sft8k|gqa16k|long64k|tiny4k] [--packs P]
(--workload picks another configuration of seeded_inputs; sft8k is the benchmark.)
For N > 1 launch with torch.distributed.run; each rank runs its own packs
(independent replicas, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "varlen causal attn fwd+bwd TFLOP/s (in-segment FLOPs), % of GB300 bf16 peak"
UNIT = "TFLOP/s"
WORKLOAD = "sft8k"
PACKS_PER_STEP = 16        # --packs changes it (small cases for profiling)


def kernel_traffic(kernel: str):
    """DRAM bytes per launch (read + write) of `kernel` from the committed ncu record, or None
    when there is none or the kernel's source changed since it was captured."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic_sft8k.json")
    try:
        rec = json.load(open(path))["kernels"][kernel]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
    except (OSError, KeyError, ValueError):
        return None
    if hashlib.sha1(src).hexdigest() != rec["source_sha1"]:
        return None
    return rec["bytes"] if WORKLOAD == "sft8k" else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


WINDOW = None  # causal local window of the run (--window), None for none


def edges(lengths):
    """Causal in-segment edges: query i of a segment sees min(i, w) + 1 keys under a window w."""
    if WINDOW is None:
        return sum(l * (l + 1) // 2 for l in lengths)
    w = WINDOW
    tot = 0
    for l in lengths:
        m = min(l - 1, w)
        tot += (m + 1) * (m + 2) // 2 + max(0, l - 1 - w) * (w + 1)
    return tot


def batch_packs_of(name: str, rank: int, planners, packs_per_step: int | None = None):
    """Doc lengths (without pad) of this rank's packs of workload `name`, with the workload.

    ``planners = (next_fit, best_fit_decreasing)``, each ``(lengths, capacity)`` -> packs
    as index lists: the library's for our arm, the oracle's for the CPU legs.  Without
    `packs_per_step`, all of the workload's packs.
    """
    w = si.WORKLOADS[name]
    raw = si.raw_lengths(name).tolist()
    planner = host_planner(w, planners)
    packs = [raw] if planner is None else [[raw[i] for i in p] for p in planner(raw, w.capacity)]
    if w.packs_used:  # e.g. tiny4k is the first row only: the rest of its draws are a partial row
        packs = packs[:w.packs_used]
    if packs_per_step is None:
        return packs, list(range(len(packs))), w
    idx = rank_pack_indices(rank, packs_per_step, len(packs))
    return [packs[i] for i in idx], idx, w


def batch_packs(rank: int, planners):
    """This rank's packs of the current workload (PACKS_PER_STEP of them)."""
    return batch_packs_of(WORKLOAD, rank, planners, PACKS_PER_STEP)


def rank_pack_indices(rank: int, packs_per_step: int, n_packs: int):
    """Weak scaling without a data-path exchange: rank r takes the workload's packs
    r*P .. r*P + P - 1 (wrapping around the workload's packs)."""
    return [(rank * packs_per_step + i) % n_packs for i in range(packs_per_step)]


def aggregate(elapsed_ms: float, step_flops: float, steps: int, dist=None, device="cpu"):
    """Whole-job figures: the elapsed time is the maximum over ranks, the work the sum over
    ranks (ranks process different packs).  Returns (max_ms, total_flops)."""
    import torch
    if dist is None:
        return elapsed_ms, step_flops * steps
    mx = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    sm = torch.tensor([step_flops * steps], dtype=torch.float64, device=device)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx.item()), float(sm.item())


def host_planner(w, planners):
    """The workload's packing planner (None for a fixed segment list)."""
    if w.strategy == "fixed":
        return None
    return planners[1] if w.strategy == "best_fit_decreasing" else planners[0]


# Causal packs whose mean segment length is below TOKEN_MEAN run their segments of at most
# TOKEN_SHORT tokens as token tiles.
TOKEN_SHORT, TOKEN_MEAN = 64, 256


def flops_of(docs, pad_to, d, Hq):
    e_doc = edges(docs)
    pad = pad_to - sum(docs)
    e_all = e_doc + (edges([pad]) if pad > 0 else 0)
    segs = list(docs) + ([pad] if pad > 0 else [])
    tok = sum(segs) < TOKEN_MEAN * len(segs)
    return {"fwd": 4 * d * Hq * e_doc, "bwd": 10 * d * Hq * e_doc,
            "e_doc": e_doc, "e_all": e_all, "t_tok": sum(x for x in segs if x <= TOKEN_SHORT) if tok else 0}


def kernel_bytes_of(t_all, t_tok, d, Hq, Hkv):
    """Algorithmic HBM bytes per kernel: every input row read once and every output row
    written once (bf16 rows of d per head, fp32 lse and D), over all t_all rows, or over the
    t_tok rows of token-tiled segments for the token forward kernel."""
    q, kv = 2 * d * Hq, 2 * d * Hkv
    fwd_row = q + 2 * kv + q + 4 * Hq                # q, k, v -> o, lse
    return {"fwd": t_all * fwd_row, "fwd_tok": t_tok * fwd_row,
            "bwd_prep": t_all * (2 * q + 4 * Hq),    # o, dO -> D
            "bwd_dkdv": t_all * (2 * q + 2 * kv + 8 * Hq + 2 * kv),  # q, dO, k, v, lse, D -> dk, dv
            "bwd_dq": t_all * (2 * q + 2 * kv + 8 * Hq + q)}         # q, dO, k, v, lse, D -> dq


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows]
        pw = [num(r[3]) for r in rows]
        busy = [s for s, p in zip(sm, pw) if p == p and p > 0.25 * max(pw)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ our arm

def measure(args, name, packs_per_step, rank, world, dev, va, lib, dist, barrier, attribution=True):
    """Times `args.steps` steps of workload `name` (`packs_per_step` packs per step, inputs
    resident on the device), then the same steps again with every launch bracketed by CUDA
    events for the per-kernel attribution (not part of the timed value)."""
    global WORKLOAD, PACKS_PER_STEP
    saved = WORKLOAD, PACKS_PER_STEP
    WORKLOAD, PACKS_PER_STEP = name, packs_per_step
    try:
        import torch
        planners = (va.pack_next_fit, va.pack_best_fit_decreasing)
        packs, idx, w = batch_packs(rank, planners)
        plan_host = host_planner(w, planners)
        d, Hq, Hkv, T = w.d, w.Hq, w.Hkv, w.pad_to or sum(packs[0])
        fl = [flops_of(p, T, d, Hq) for p in packs]
        step_flops = sum(f["fwd"] + f["bwd"] for f in fl)
        ins = []
        for pi, docs in zip(idx, packs):
            q, k, v, do = si.tensors(T, Hq, Hkv, d, seed_offset=1000 * pi)
            ins.append(tuple(x.to(dev) for x in (q, k, v, do)))
        lens_dev = [torch.tensor(p, dtype=torch.int32, device=dev) for p in packs]
        all_docs = [L for p in packs for L in p]
        B = [len(p) + (1 if sum(p) < T else 0) for p in packs]
        mxs = [max(p + ([T - sum(p)] if sum(p) < T else [])) for p in packs]
        ws_f = torch.empty(va.workspace_size(T, max(B), Hq, Hkv, d, T, False), dtype=torch.uint8, device=dev)
        ws_b = torch.empty(va.workspace_size(T, max(B), Hq, Hkv, d, T, True), dtype=torch.uint8, device=dev)
        outs = [(torch.empty_like(i[0]), torch.empty((Hq, T), dtype=torch.float32, device=dev),
                 torch.empty_like(i[0]), torch.empty_like(i[1]), torch.empty_like(i[2])) for i in ins]

        def step():
            # host planner over the batch's documents (its packs match the resident lengths)
            if plan_host is not None:
                plan_host(all_docs, w.capacity)
            for p in range(len(packs)):
                q, k, v, do = ins[p]
                o, lse, dq, dk, dv = outs[p]
                cu, _, _, _, _ = va.build_metadata(lens_dev[p], pad_to=T, T_capacity=T)
                cu = cu[:B[p] + 1]
                va.varlen_attn_fwd(q, k, v, cu, mxs[p], None, True, out=o, lse=lse, workspace=ws_f, window=WINDOW)
                va.varlen_attn_bwd(q, k, v, o, lse, do, cu, mxs[p], None, True, dq=dq, dk=dk, dv=dv,
                                   window=WINDOW, workspace=ws_b)

        for _ in range(args.warmup):
            step()
        barrier()
        if va.read_status(ws_f) or va.read_status(ws_b):
            raise RuntimeError(f"device status error during the {name} warm-up")

        # the timed region: no per-kernel events inside it
        lc0 = lib.varlen_launch_count()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(torch.cuda.current_device()) as clocks:
            barrier()
            start.record()
            for _ in range(args.steps):
                step()
            stop.record()
            barrier()
        launches = lib.varlen_launch_count() - lc0
        elapsed_ms = start.elapsed_time(stop)
        per_kernel = {}
        if attribution:
            import ctypes
            n_launch_cap = args.steps * len(packs) * 16 + 64
            lib.varlen_profile_enable(n_launch_cap)
            for _ in range(args.steps):
                step()
            barrier()
            ids = (ctypes.c_int32 * n_launch_cap)()
            ms = (ctypes.c_float * n_launch_cap)()
            cnt = ctypes.c_int32()
            lib.varlen_profile_read(ids, ms, n_launch_cap, ctypes.byref(cnt))
            lib.varlen_profile_enable(0)
            for i in range(cnt.value):
                kname = lib.varlen_kernel_name(ids[i]).decode()
                t, c = per_kernel.get(kname, (0.0, 0))
                per_kernel[kname] = (t + ms[i], c + 1)
        max_ms, total_flops = aggregate(elapsed_ms, step_flops, args.steps, dist, dev)
        del ins, outs, ws_f, ws_b
        return {"value": total_flops / (max_ms * 1e-3) / 1e12, "max_ms": max_ms, "step_flops": step_flops,
                "per_kernel": per_kernel, "fl": fl, "packs": packs, "idx": idx, "w": w, "T": T,
                "launches": launches, "clocks": clocks.summary(), "plan_host": plan_host,
                "n_packs": len(packs)}
    finally:
        WORKLOAD, PACKS_PER_STEP = saved


def kernel_rates(m, steps):
    """Forward and backward kernel rates from the per-kernel attribution (CUDA events)."""
    pk, fl = m["per_kernel"], m["fl"]
    w = m["w"]
    e_doc = sum(f["e_doc"] for f in fl) * steps
    fwd_t = pk.get("fwd", (0.0, 1))[0] + pk.get("fwd_tok", (0.0, 1))[0]
    bwd_t = sum(pk.get(k, (0.0, 0))[0] for k in ("bwd_prep", "bwd_dkdv", "bwd_dq"))
    fwd = 4 * w.d * w.Hq * e_doc / (fwd_t * 1e-3) / 1e12 if fwd_t else None
    bwd = 10 * w.d * w.Hq * e_doc / (bwd_t * 1e-3) / 1e12 if bwd_t else None
    return fwd, bwd


def run_ours(args, rank, world, local_rank):
    import torch
    import packed_sequence_varlen_gb300 as va
    from packed_sequence_varlen_gb300 import _lib

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = _lib.load()
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    m = measure(args, WORKLOAD, PACKS_PER_STEP, rank, world, dev, va, lib, dist, barrier)
    packs, idx, w, T, fl, per_kernel = m["packs"], m["idx"], m["w"], m["T"], m["fl"], m["per_kernel"]
    d, Hq, Hkv = w.d, w.Hq, w.Hkv
    max_ms, value, step_flops = m["max_ms"], m["value"], m["step_flops"]

    # roofline of the dominant kernel: algorithmic flops per launch / launch time.  The kernels
    # run inside a sub-second timed region, so the burst peak is the denominator.
    peaks = load_peaks()
    e_all = sum(f["e_all"] for f in fl) * args.steps
    e_doc = sum(f["e_doc"] for f in fl) * args.steps
    kernel_flops = {"fwd": 4 * d * Hq * e_all, "bwd_dkdv": 8 * d * Hq * e_all,
                    "bwd_dq": 6 * d * Hq * e_all}
    kernel_bytes = kernel_bytes_of(T * len(fl) * args.steps, sum(f["t_tok"] for f in fl) * args.steps,
                                   d, Hq, Hkv)
    dom = max(per_kernel, key=lambda k: per_kernel[k][0])
    roof = None
    # the kernel's bound: the larger of its ideal tensor time and its ideal HBM time
    hbm_bound = dom in kernel_bytes and (dom not in kernel_flops or
                                         kernel_bytes[dom] / (peaks["hbm_gbs"] * 1e9) >
                                         kernel_flops[dom] / (peaks["bf16_tflops"] * 1e12))
    if hbm_bound:
        ach = kernel_bytes[dom] / (per_kernel[dom][0] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                "peak_kind": f"HBM copy, {peaks['source']}", "traffic": kernel_traffic(dom),
                "launches": per_kernel[dom][1],
                "avg_launch_us": round(per_kernel[dom][0] / per_kernel[dom][1] * 1e3, 2)}
    elif dom in kernel_flops:
        ach = kernel_flops[dom] / (per_kernel[dom][0] * 1e-3) / 1e12
        ach_doc = ach * e_doc / e_all
        roof = {"bound": "tensor", "kernel": dom, "achieved": round(ach, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / peaks["bf16_tflops"], 4),
                "peak_kind": f"bf16 burst, {peaks['source']} (kernel timed inside a sub-second region)",
                "work": "all computed edges (tail pad segment included)",
                "achieved_doc_edges": round(ach_doc, 2), "frac_doc_edges": round(ach_doc / peaks["bf16_tflops"], 4),
                "frac_of_sustained": round(ach / peaks["bf16_tflops_sustained"], 4),
                "traffic": kernel_traffic(dom),
                "launches": per_kernel[dom][1],
                "avg_launch_us": round(per_kernel[dom][0] / per_kernel[dom][1] * 1e3, 2)}
    kernel_table = {k: {"launches": c, "total_ms": round(t, 3),
                        "share": round(t / max(sum(x[0] for x in per_kernel.values()), 1e-9), 4)}
                    for k, (t, c) in sorted(per_kernel.items(), key=lambda kv: -kv[1][0])}
    fwd_tflops, bwd_tflops = kernel_rates(m, args.steps)
    # boundary metadata and the forward's check + map, per pack
    n_calls = len(fl) * args.steps
    plan_us = sum(t for k, (t, _) in per_kernel.items() if k.startswith("metadata") or k == "validate_plan")
    plan_us = plan_us * 1e3 / n_calls if n_calls else None

    # the second target configuration, over every BFD bin (default sft8k run only)
    second = None
    if WORKLOAD == "sft8k" and WINDOW is None and not args.no_gqa16k:
        n_bins = len(batch_packs_of("gqa16k", rank, (va.pack_next_fit, va.pack_best_fit_decreasing))[0])
        g = measure(args, "gqa16k", n_bins, 0, world, dev, va, lib, dist, barrier)
        gf, gb = kernel_rates(g, args.steps)
        second = {"workload": f"gqa16k: all {n_bins} BFD bins of 16384 tokens per step "
                              f"({g['w'].description}), causal, fwd+bwd",
                  "fwd_bwd_tflops": round(g["value"], 2),
                  "pct_of_bf16_peak_burst": round(100 * g["value"] / world / peaks["bf16_tflops"], 2),
                  "ms_per_step": round(g["max_ms"] / args.steps, 3),
                  "fwd_kernel_tflops": round(gf, 2) if gf else None,
                  "fwd_kernel_pct_of_burst": round(100 * gf / peaks["bf16_tflops"], 2) if gf else None,
                  "bwd_kernels_tflops": round(gb, 2) if gb else None,
                  "gpu_launches": int(g["launches"]), "clocks": g["clocks"]}

    e2e = run_e2e(args, va, dev, packs, idx, w, step_flops, dist, barrier, m["plan_host"]) if not args.no_e2e else None

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(max_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {PACKS_PER_STEP} pack(s) of {T} tokens per step ({w.description}), "
                               "causal" + (f", local window {WINDOW} (in-window FLOPs)" if WINDOW is not None else "")
                               + ", fwd+bwd",
                   "tokens_per_step": PACKS_PER_STEP * T, "packs_per_step": PACKS_PER_STEP,
                   "l2": f"inputs larger than L2 ({T * (2 * Hq + 2 * Hkv) * d * 2 // 2**20} MB per pack)",
                   "parallelism": f"replicas x{world}",
                   "pct_of_bf16_peak_burst": round(100 * value / world / peaks["bf16_tflops"], 2),
                   "fwd_kernel_tflops": round(fwd_tflops, 2) if fwd_tflops else None,
                   "fwd_kernel_pct_of_burst": round(100 * fwd_tflops / peaks["bf16_tflops"], 2) if fwd_tflops else None,
                   "bwd_kernels_tflops": round(bwd_tflops, 2) if bwd_tflops else None,
                   "metadata_and_fwd_plan_us_per_pack": round(plan_us, 2) if plan_us else None,
                   "gqa16k": second},
        "e2e": e2e,
        "gpu_launches": int(m["launches"]),
        "kernels": kernel_table,
        "roofline": roof,
        "clocks": m["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
        if second is not None:
            result["config"]["gqa16k"]["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget, name="gqa16k")
    return result


def link_bandwidth(dev, nbytes: int = 256 << 20, reps: int = 5):
    """Pinned host <-> device copy bandwidth (GB/s): H2D alone, D2H alone, and each direction
    while both run at once on their own streams (how the e2e step uses the link)."""
    import torch
    h_up = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_dn = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_up = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_dn = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / reps

    def both():
        with torch.cuda.stream(s1):
            d_up.copy_(h_up, non_blocking=True)
        with torch.cuda.stream(s2):
            h_dn.copy_(d_dn, non_blocking=True)
    return {"h2d": round(nbytes / timed(lambda: d_up.copy_(h_up, non_blocking=True)) / 1e9, 1),
            "d2h": round(nbytes / timed(lambda: h_dn.copy_(d_dn, non_blocking=True)) / 1e9, 1),
            "concurrent_each": round(nbytes / timed(both) / 1e9, 1)}


def run_e2e(args, va, dev, packs, idx, w, step_flops, dist, barrier, plan_host):
    """Same step through the public API from pinned HOST buffers: H2D of every pack's q/k/v/dO
    and lengths, the step, D2H of dq/dk/dv, all inside the timed region.  Copies run on their
    own streams with two device buffer sets used in turn, continuously across steps: pack
    p+1 uploads and pack p-1 downloads while pack p computes (H2D and D2H use opposite link
    directions); a set is reused only after its previous pack computed (inputs) and
    downloaded (gradients).  Two sets measured faster than three (24.5 against 35 ms per
    sft8k step: with three, the uploads themselves ran at about 150 GB/s instead of 170)."""
    import torch
    d, Hq, Hkv, T = w.d, w.Hq, w.Hkv, w.pad_to or sum(packs[0])
    host_in = []
    for pi in idx:
        q, k, v, do = si.tensors(T, Hq, Hkv, d, seed_offset=1000 * pi)
        host_in.append(tuple(x.pin_memory() for x in (q, k, v, do)))
    host_len = [torch.tensor(p, dtype=torch.int32).pin_memory() for p in packs]
    host_out = [tuple(torch.empty((T, H, d), dtype=torch.bfloat16).pin_memory() for H in (Hq, Hkv, Hkv))
                for _ in range(len(packs))]
    nbuf = 2
    dev_in = [[torch.empty((T, H, d), dtype=torch.bfloat16, device=dev) for H in (Hq, Hkv, Hkv, Hq)]
              for _ in range(nbuf)]
    lens_dev = [torch.empty(max(len(p) for p in packs), dtype=torch.int32, device=dev) for _ in range(nbuf)]
    o = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    g = [[torch.empty((T, H, d), dtype=torch.bfloat16, device=dev) for H in (Hq, Hkv, Hkv)] for _ in range(nbuf)]
    all_docs = [L for p in packs for L in p]
    h2d = sum(x.numel() * x.element_size() for t in host_in for x in t) + sum(x.numel() * 4 for x in host_len)
    d2h = sum(x.numel() * x.element_size() for t in host_out for x in t)
    s_up, s_cmp, s_dn = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n = len(packs)
    done = [None] * nbuf   # the last pack that used buffer set b has computed
    down = [None] * nbuf   # ... and its gradients are downloaded

    def step():
        if plan_host is not None:
            plan_host(all_docs, w.capacity)
        for p in range(n):
            b = p % nbuf
            with torch.cuda.stream(s_up):
                if done[b] is not None:
                    s_up.wait_event(done[b])
                for dst, src in zip(dev_in[b], host_in[p]):
                    dst.copy_(src, non_blocking=True)
                lens_dev[b][:len(packs[p])].copy_(host_len[p], non_blocking=True)
                up = torch.cuda.Event()
                up.record(s_up)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(up)
                if down[b] is not None:
                    s_cmp.wait_event(down[b])
                k_ = len(packs[p])
                cu, _, _, _, _ = va.build_metadata(lens_dev[b][:k_], pad_to=T, T_capacity=T)
                Bp = k_ + (1 if sum(packs[p]) < T else 0)
                mxs = max(packs[p] + ([T - sum(packs[p])] if sum(packs[p]) < T else []))
                cu = cu[:Bp + 1]
                q, k, v, do = dev_in[b]
                va.varlen_attn_fwd(q, k, v, cu, mxs, None, True, out=o, lse=lse, window=WINDOW)
                va.varlen_attn_bwd(q, k, v, o, lse, do, cu, mxs, None, True, dq=g[b][0], dk=g[b][1], dv=g[b][2],
                                   window=WINDOW)
                done[b] = torch.cuda.Event()
                done[b].record(s_cmp)
            with torch.cuda.stream(s_dn):
                s_dn.wait_event(done[b])
                for dst, src in zip(host_out[p], g[b]):
                    dst.copy_(src, non_blocking=True)
                down[b] = torch.cuda.Event()
                down[b].record(s_dn)

    def drain():
        for s_ in (s_up, s_cmp, s_dn):
            torch.cuda.current_stream(dev).wait_stream(s_)

    for _ in range(max(1, args.warmup)):
        step()
    drain()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    drain()
    barrier()
    dt = time.perf_counter() - t0
    max_ms, total_flops = aggregate(dt * 1e3, step_flops, args.steps, dist, dev)
    link = link_bandwidth(dev)
    bound_ms = max(h2d / link["concurrent_each"], d2h / link["concurrent_each"]) / 1e6
    return {"value": round(total_flops / (max_ms * 1e-3) / 1e12, 3), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(max_ms / args.steps, 3),
            "link_gbs": link, "link_bound_ms_per_step": round(bound_ms, 3),
            "frac_of_link_bound": round(bound_ms / (max_ms / args.steps), 4),
            "overlap": "H2D, compute and D2H on three streams, two device buffer sets used in turn across steps"}


# ------------------------------------------------------------------ oracle timing

def cpu_baseline(budget_s: float = 12.0, steps: int | None = None, name: str | None = None):
    """The float64 CPU oracle as it stands, on pack 0 of the workload, one kv head at a time
    (the oracle then computes that kv head's whole group of g q heads): the forward alone,
    then forward + backward.  FLOPs count real-document edges of every q head computed."""
    from oracle import attention as oa
    from oracle import packing as op
    name = name or WORKLOAD
    packs, idx, w = batch_packs_of(name, 0, (op.next_fit, op.best_fit_decreasing), 1)
    docs = packs[0]
    T = w.pad_to or sum(docs)
    segs = docs + ([T - sum(docs)] if sum(docs) < T else [])
    cu = np.cumsum([0] + segs)
    q, k, v, do = si.tensors(T, w.Hq, w.Hkv, w.d, seed_offset=1000 * idx[0])
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    g = w.Hq // w.Hkv
    per_kv_fwd = 4 * w.d * g * edges(docs)      # the g q heads of one kv head, real documents only
    per_kv_all = 14 * w.d * g * edges(docs)
    heads, t_fwd, t_total, times = 0, 0.0, 0.0, []
    while (steps is None and t_total < budget_s and heads < w.Hkv) or (steps is not None and heads < steps):
        h = heads % w.Hkv
        t0 = time.perf_counter()
        o, lse = oa.varlen_forward(qq, kk, vv, cu, None, True, [h], window=WINDOW)
        t1 = time.perf_counter()
        oa.varlen_backward(qq, kk, vv, o, lse, dd, cu, None, True, [h], window=WINDOW)
        dt = time.perf_counter() - t0
        times.append(dt)
        t_fwd += t1 - t0
        t_total += dt
        heads += 1
    value = per_kv_all * heads / t_total / 1e12
    return {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "fwd_value": per_kv_fwd * heads / t_fwd / 1e12,
            "sample": f"{name} pack 0 ({len(docs)} documents + pad, T={T}), {heads} of {w.Hkv} kv heads "
                      f"({heads * g} of {w.Hq} q heads), fwd and fwd+bwd, numpy float64 (BLAS on all cores)",
            "seconds": round(t_total, 2), "step_times_s": [round(x, 3) for x in times]}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, one kv head of pack 0 per step."""
    if rank != 0:
        return None
    from oracle import attention as oa
    from oracle import packing as op
    packs, idx, w = batch_packs(0, (op.next_fit, op.best_fit_decreasing))
    docs = packs[0]
    T = w.pad_to or sum(docs)
    segs = docs + ([T - sum(docs)] if sum(docs) < T else [])
    cu = np.cumsum([0] + segs)
    q, k, v, do = si.tensors(T, w.Hq, w.Hkv, w.d, seed_offset=1000 * idx[0])
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    per_step = 14 * w.d * (w.Hq // w.Hkv) * edges(docs)   # one kv head: its g q heads

    def step(i):
        h = i % w.Hkv
        o, lse = oa.varlen_forward(qq, kk, vv, cu, None, True, [h], window=WINDOW)
        oa.varlen_backward(qq, kk, vv, o, lse, dd, cu, None, True, [h], window=WINDOW)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt / 1e12
    sample = (f"{WORKLOAD} pack 0 ({len(docs)} documents + pad, T={T}), one of {w.Hkv} kv heads "
              f"({w.Hq // w.Hkv} q heads) per step, fwd+bwd, numpy float64 (BLAS on all cores)")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": f"{WORKLOAD}: one kv head of pack 0 per step (bounded sample)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ cross-attention

def run_cross(args, rank, world, local_rank):
    """Cross-attention (prefix-cache shape): every sft8k segment's queries attend to a P-token
    prefix followed by the segment itself (lk = lq + P, causal aligned bottom-right).  One step =
    forward + backward over `--packs` packs; the boundaries are built once, outside the step.
    FLOPs count the visible edges of every segment (the tail pad included): i + P + 1 keys for
    query i."""
    import torch
    import packed_sequence_varlen_gb300 as va
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    global WORKLOAD
    WORKLOAD = "sft8k"
    packs, idx, w = batch_packs(rank, (va.pack_next_fit, va.pack_best_fit_decreasing))
    P, T, d, Hq, Hkv = args.cross_prefix, w.pad_to, w.d, w.Hq, w.Hkv
    ins, edges_all = [], 0
    for pi, docs in zip(idx, packs):
        segs = docs + ([T - sum(docs)] if sum(docs) < T else [])
        cuq = [0]
        cuk = [0]
        for x in segs:
            cuq.append(cuq[-1] + x)
            cuk.append(cuk[-1] + x + P)
            edges_all += x * (x + 1) // 2 + x * P
        q, _, _, do = si.tensors(T, Hq, Hkv, d, seed_offset=1000 * pi)
        _, k, v, _ = si.tensors(cuk[-1], Hq, Hkv, d, seed_offset=1000 * pi + 1)
        ins.append((q.to(dev), k.to(dev), v.to(dev), do.to(dev),
                    torch.tensor(cuq, dtype=torch.int32, device=dev), torch.tensor(cuk, dtype=torch.int32, device=dev),
                    max(segs), max(segs) + P))
    step_flops = 14 * d * Hq * edges_all
    ws_f = torch.empty(1 << 26, dtype=torch.uint8, device=dev)
    ws_b = torch.empty(1 << 28, dtype=torch.uint8, device=dev)

    def step():
        for q, k, v, do, cq, ck, mq, mk in ins:
            o, lse = va.varlen_attn_fwd_cross(q, k, v, cq, ck, mq, mk, None, True, workspace=ws_f)
            va.varlen_attn_bwd_cross(q, k, v, o, lse, do, cq, ck, mq, mk, None, True, workspace=ws_b)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if va.read_status(ws_f) or va.read_status(ws_b):
        raise RuntimeError("device-detected error in the cross-attention run")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    peaks = load_peaks()
    value = step_flops / (ms * 1e-3) / 1e12
    return {"metric": "varlen causal cross-attention fwd+bwd TFLOP/s (visible edges)", "value": round(value, 3),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"cross: {len(packs)} sft8k pack(s) of {T} queries, each segment's keys a "
                                   f"{P}-token prefix + the segment (Hq=Hkv={Hq}, d={d}), causal bottom-right",
                       "pct_of_bf16_peak_burst": round(100 * value / peaks["bf16_tflops"], 2)},
            "e2e": None, "clocks": clocks.summary()}


# ------------------------------------------------------------------ packed loss

def run_loss(args, rank, world, local_rank):
    """Token-weighted cross entropy + logit gradient over the packed stream (the packed loss
    layout): one step = targets formed inside each segment and the loss over `--packs` sft8k
    packs of 8192 tokens with bf16 logits over `--vocab` classes.  HBM-bound: the algorithmic
    bytes are the eligible rows' logits read once, every gradient row written once, targets."""
    import torch
    import packed_sequence_varlen_gb300 as va
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    planners = (va.pack_next_fit, va.pack_best_fit_decreasing)
    global WORKLOAD
    WORKLOAD = "sft8k"
    packs, idx, w = batch_packs(rank, planners)
    T1, V = w.pad_to, args.vocab
    segs = [p + ([T1 - sum(p)] if sum(p) < T1 else []) for p in packs]
    cu = [0]
    for p in segs:
        for x in p:
            cu.append(cu[-1] + x)
    T = cu[-1]
    gen = torch.Generator().manual_seed(11 + rank)
    ids = torch.randint(0, V, (T,), generator=gen, dtype=torch.int32).to(dev)
    cud = torch.tensor(cu, dtype=torch.int32, device=dev)
    dgen = torch.Generator(device=dev).manual_seed(12 + rank)  # seeded, drawn on the device
    logits = torch.empty((T, V), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, T, 1024):  # N(0, 3^2), in slices
        n = min(1024, T - r0)
        logits[r0:r0 + n] = (3 * torch.randn(n, V, generator=dgen, device=dev)).to(torch.bfloat16)
    grad = torch.empty_like(logits)
    ws = torch.empty(va._lib.load().varlen_token_ce_workspace_size(T), dtype=torch.uint8, device=dev)
    lib = va._lib.load()

    def step():
        tg = va.loss_targets(ids, cud)
        return va.token_ce(logits, tg, grad=grad, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n_elig = int(step()[1].item())
    l0 = lib.varlen_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    launches = lib.varlen_launch_count() - l0
    alg = n_elig * V * 2 + T * V * 2 + 3 * T * 4  # logits (eligible rows), grad, ids/targets
    gbs = alg / (ms * 1e-3) / 1e9
    peaks = load_peaks()
    res = {"metric": "packed token-weighted CE + logit gradient, algorithmic HBM GB/s", "value": round(gbs, 1),
           "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic",
           "config": {"workload": f"loss: {len(packs)} sft8k pack(s) of {T1} tokens (T={T}), V={V}, "
                                  f"bf16 logits N(0, 9), targets formed inside each segment ({n_elig} eligible)",
                      "l2": f"inputs larger than L2 ({T * V * 2 // 2**20} MB of logits)"},
           "e2e": None, "gpu_launches": int(launches),
           "roofline": {"bound": "hbm", "kernel": "token_ce", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                        "peak_kind": f"HBM copy, {peaks['source']}", "traffic": None},
           "clocks": clocks.summary()}
    if not args.no_cpu_baseline:
        import time
        from oracle import loss as ol
        rows = 128  # bounded sample: the oracle on the first rows, scaled by bytes
        z = logits[:rows].double().cpu().numpy()
        tg = va.loss_targets(ids, cud)[:rows].cpu().numpy()
        t0 = time.perf_counter()
        ol.token_weighted_loss(z, tg, tg != -100)
        dt = time.perf_counter() - t0
        b = int((tg != -100).sum()) * V * 2 + rows * V * 2 + 3 * rows * 4
        res["cpu_baseline"] = {"value": round(b / dt / 1e9, 3), "unit": "GB/s", "cores": os.cpu_count(),
                               "kind": "oracle", "sample": f"first {rows} rows of the same logits, float64 numpy"}
    return res


def main():
    global PACKS_PER_STEP
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gqa16k", action="store_true",
                    help="skip the second target configuration (gqa16k, every BFD bin) of the default run")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--packs", type=int, default=16,
                    help="packs per step (16 is the benchmark; fewer for profiling cases)")
    ap.add_argument("--workload", choices=["sft8k", "gqa16k", "long64k", "tiny4k"], default="sft8k",
                    help="configuration (sft8k is the benchmark; the others are for measurement)")
    ap.add_argument("--window", type=int, default=None,
                    help="causal local window (query i sees keys i-w..i); FLOPs count in-window edges")
    ap.add_argument("--cross-prefix", type=int, default=None,
                    help="measure cross-attention: each segment's keys are a P-token prefix + the segment")
    ap.add_argument("--loss", action="store_true",
                    help="measure the packed loss (targets + token-weighted CE + gradient) instead")
    ap.add_argument("--vocab", type=int, default=32768, help="classes of the --loss logits")
    args = ap.parse_args()
    global WORKLOAD, WINDOW
    WORKLOAD = args.workload
    WINDOW = args.window
    PACKS_PER_STEP = args.packs
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.loss:
        res = run_loss(args, rank, world, local_rank)
    elif args.cross_prefix is not None:
        res = run_cross(args, rank, world, local_rank)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
