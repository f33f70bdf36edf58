#!/usr/bin/env python3
"""Benchmark of the hyper-connection low-rank mix block on GB300.

Default workload: the single decode block (rows = 1, C = 4, H = 2560, R = 320,
bf16, with prologue, the Qwen-shaped attributes), run as a chain over 96
distinct synthetic weight sets (1.27 GB of weights, far larger than the 129 MB
L2, so every block reads its weights from HBM). Block i + 1 takes block i's
pre_output and post_gate as its prologue and its streams_out as streams. One
step = one block. The timed steps replay CUDA graphs of 96 (and a remainder
of) chained blocks, captured from the public API; their kernels are linked by
programmatic dependent launch.

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle
instead, on a bounded sample of the same workload.
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

METRIC = "µs/block and rows/s, rows 1–8192, as % of HBM / bf16 tensor roofline"
C, H, R = 4, 2560, 320
NSETS = 96
QWEN = dict(epsilon=1e-6, reduction_scale=0.25, silu_alpha=0.25, gate_div=4.0, gate_mul=2.0)
WORKLOAD = ("decode block: rows=1, C=4, H=2560, R=320, bf16, with prologue, Qwen attributes; "
            "chain over 96 distinct weight sets (1.27 GB), graph replay")


def block_bytes(rows, C, H, R, es, prologue=True):
    """Algorithmic bytes of one block: weights and norm_scale once, and per row
    streams in, streams_out, prev_out, prev_gate, pre_output, post_gate."""
    CH = C * H
    weights = (2 * CH * R + CH * C + CH) * es
    per_row = (2 * CH + H + C + (H + C if prologue else 0)) * es
    return weights + rows * per_row


def block_flops(rows, C, H, R):
    CH = C * H
    return 2 * rows * (2 * CH * R + CH * C)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return dict(hbm=float(j["hbm_gbs"]), bf16=float(j["bf16_tflops"]),
                    bf16_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# Sources the decode kernel pair is compiled from: a recorded traffic figure is
# valid only while these are unchanged.
DECODE_SOURCES = ("hc_decode_um.cu", "hc_common.cuh", "hc_async.cuh", "hc_tc.cuh", "hc_vec.cuh", "hc_internal.h")


def kernel_source_hash(files=DECODE_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hyper_connection_rank_gb300", "csrc")
    for fn in sorted(files):
        h.update(fn.encode())
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(name):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    j = json.load(open(p)).get(name)
    if not j or j.get("source_hash") != kernel_source_hash(tuple(j.get("sources", DECODE_SOURCES))):
        return None
    return j.get("dram_bytes_per_unit")


# ------------------------------------------------------------ clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", "100", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ ranks --

def max_over_ranks(x, device):
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ our arm --

def run_ours(args, rank, world, local_rank):
    import torch

    import __graft_entry__
    import hyper_connection_rank_gb300 as hc
    from hyper_connection_rank_gb300 import inputs as I

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    __graft_entry__.build()
    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()

    if args.profile_case == "prefill":
        return profile_prefill(args, hc, I, dev)
    if args.profile_case == "rowops":
        return profile_rowops(args, hc, I, dev)
    rows = args.rows
    flags = hc.HC_FLAG_WEIGHTS_STATIC
    assert hc.path(rows, C, H, R, torch.bfloat16, flags) == hc.HC_PATH_DECODE
    if args.profile_case == "phases":
        return profile_phases(args, hc, I, dev, rows, flags)
    if args.profile_case == "sync":
        return {"profile_case": "synchronisation cost probe", "sync_costs": sync_costs(hc, dev)}
    if args.profile_case:
        return profile_case(args, hc, I, dev, rows, flags)
    weights = [I.make_weights(C, H, R, "bf16", seed=0, block=i, device=dev) for i in range(NSETS)]
    bufs = [I.make_activations(rows, C, H, "bf16", seed=0, block=0, prologue=True, device=dev)]
    bufs.append({k: torch.empty_like(v) for k, v in bufs[0].items()})
    ws = torch.empty(max(1, hc.workspace_size(rows, C, H, R, torch.bfloat16, flags)), dtype=torch.uint8, device=dev)

    def step(i):
        src, dst, w = bufs[i % 2], bufs[(i + 1) % 2], weights[i % NSETS]
        hc.lowrank_mix(src["streams"], w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"], src["prev_out"],
                       src["prev_gate"], num_branches=C, flags=flags,
                       out=(dst["prev_out"], dst["prev_gate"], dst["streams"]), workspace=ws, **QWEN)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    step(i)
        torch.cuda.current_stream(dev).wait_stream(s)
        return g

    K, W = args.steps, args.warmup
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    g_full = capture(NSETS)
    g_rem = capture(K % NSETS) if K % NSETS else None
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    # untimed lead-in: one 96-block replay enqueued ahead of the timed one, so
    # the timed blocks start right behind running work (steady state) and no
    # graph-launch gap enters the timed region, whatever K is
    g_full.replay()
    ev0.record(stream)
    for _ in range(K // NSETS):
        g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    t_ms = max_over_ranks(ev0.elapsed_time(ev1), dev) if dist else ev0.elapsed_time(ev1)
    for b in bufs:
        for v in b.values():
            assert torch.isfinite(v.float()).all(), "non-finite values in the chain"

    us_per_block = 1000.0 * t_ms / K
    value = world * rows * K / (t_ms / 1000.0)
    pk = peaks()
    bytes_blk = block_bytes(rows, C, H, R, 2)
    achieved = bytes_blk / (us_per_block * 1e-6) / 1e9
    traffic = recorded_traffic("decode_block_rows1_bf16")
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": t_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded splitmix64 + Box-Muller; Qwen-shaped, random weights)",
        "config": {"workload": WORKLOAD, "rows": rows, "C": C, "H": H, "R": R, "weight_sets": NSETS,
                   "l2": "inputs larger than L2: 96 weight sets of 13.2 MB rotated (1.27 GB)",
                   "timed_region": "K chained blocks (graph replays) enqueued right behind an untimed 96-block "
                                   "lead-in replay: steady state at any K, no graph-launch gap timed",
                   "parallelism": f"replicas x{world}"},
        "us_per_block": round(us_per_block, 4),
        "roofline": {"bound": "hbm", "kernel": "decode block (dec_down + dec_up, PDL-overlapped)",
                     "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm"], 4), "peak_source": pk["source"],
                     "bytes_per_launch": bytes_blk, "traffic": traffic},
        "gpu_launches": 2 * K,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_e2e:
        result["e2e"] = e2e_measure(args, hc, I, weights, dev, flags)
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0 and not args.no_sweep:
        del weights
        torch.cuda.empty_cache()
        result["isolated"] = isolated_latency(hc, I, dev, pk)
        result["sync_costs"] = sync_costs(hc, dev)
        result["sweep"] = sweep(hc, I, dev, pk)
    return result


def sync_costs(hc, dev, ctas=128, smem=100 * 1024, rounds=(500, 1000)):
    """What one all-to-all synchronisation of 128 CTAs costs (hc_debug_sync_probe),
    per round, as the slope between two round counts (so launch costs drop
    out): a kernel boundary with programmatic dependent launch (the chain of
    kernels captured in a CUDA graph, as the decode pair runs), a software
    grid barrier and an all-to-all flag exchange (one cooperative kernel
    each). Each CTA reserves 100 KB of shared memory, like a decode CTA (two
    fit on an SM, as the decode pair's two kernels do)."""
    import torch
    from hyper_connection_rank_gb300 import _binding as B
    L = B.lib()
    scratch = torch.zeros(32 + ctas, dtype=torch.int32, device=dev)
    nbytes = scratch.numel() * 4

    def call(mode, r, stream):
        st = L.hc_debug_sync_probe(mode, ctas, r, smem, scratch.data_ptr(), nbytes, stream.cuda_stream)
        if st != 0:
            B.check(st)

    out = {}
    for mode, name in ((0, "pdl_kernel_boundary"), (1, "grid_barrier"), (2, "flag_all_to_all")):
        t = {}
        for r in rounds:
            scratch.zero_()
            cur = torch.cuda.current_stream(dev)
            call(mode, 4, cur)
            torch.cuda.synchronize()
            if mode == 0:
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream(dev)
                side.wait_stream(cur)
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        call(0, r, side)
                cur.wait_stream(side)
                g.replay()
                torch.cuda.synchronize()
                run = g.replay
            else:
                def run(mode=mode, r=r):
                    scratch.zero_()
                    call(mode, r, torch.cuda.current_stream(dev))
            best = float("inf")
            for _ in range(5):
                if mode != 0:
                    scratch.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                if mode == 0:
                    run()
                else:
                    call(mode, r, torch.cuda.current_stream(dev))
                e1.record()
                e1.synchronize()
                best = min(best, 1000.0 * e0.elapsed_time(e1))
            errs = int(scratch[0].item())
            assert errs == 0, f"{errs} bounded polls gave up in mode {mode}"
            t[r] = best
        r0, r1 = rounds
        out[name] = {"us_per_round": round((t[r1] - t[r0]) / (r1 - r0), 3), "ctas": ctas, "smem_per_cta": smem}
    return out


def isolated_latency(hc, I, dev, pk, reps=200):
    """One decode block at a time with L2 cold: before each call a reduction
    reads a 512 MB buffer (four times L2; reading leaves no dirty lines to be
    written back during the call), then the call alone is timed with events on
    its stream. Min and median over `reps` calls, for rows 1/2/4/8 in bf16
    and fp16 (the single-block and row-sweep configurations, measured one
    call at a time rather than as a chain)."""
    import torch
    flags = hc.HC_FLAG_WEIGHTS_STATIC
    flush = torch.ones(256 << 20, dtype=torch.float16, device=dev)
    out = {}
    for dt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        w = I.make_weights(C, H, R, dt, seed=0, block=0, device=dev)
        for rows in (1, 2, 4, 8):
            a = I.make_activations(rows, C, H, dt, seed=0, block=0, prologue=True, device=dev)
            o = (torch.empty(rows, H, dtype=tdt, device=dev), torch.empty(rows, C, dtype=tdt, device=dev),
                 torch.empty(rows, C * H, dtype=tdt, device=dev))
            ws = torch.empty(max(1, hc.workspace_size(rows, C, H, R, tdt, flags)), dtype=torch.uint8, device=dev)

            def call():
                hc.lowrank_mix(a["streams"], w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"], a["prev_out"],
                               a["prev_gate"], num_branches=C, flags=flags, out=o, workspace=ws, **QWEN)

            for _ in range(5):
                call()
            torch.cuda.synchronize()
            s = torch.cuda.current_stream(dev)
            ts = []
            for _ in range(reps):
                flush.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                call()
                e1.record(s)
                e1.synchronize()
                ts.append(1000.0 * e0.elapsed_time(e1))
            b = block_bytes(rows, C, H, R, 2)
            t = min(ts)
            out[f"decode_rows{rows}_{dt}"] = {"us": round(t, 3), "us_median": round(statistics.median(ts), 3),
                                              "hbm_frac": round(b / (t * 1e-6) / 1e9 / pk["hbm"], 4)}
    del flush
    torch.cuda.empty_cache()
    return out


def profile_case(args, hc, I, dev, rows, flags):
    """Small case for profiler captures: the same decode block, 4 weight sets
    (53 MB), eager launches through the public API; prints a JSON line but is
    not a benchmark result (profiler captures flush caches per pass anyway)."""
    import torch
    weights = [I.make_weights(C, H, R, "bf16", seed=0, block=i, device=dev) for i in range(4)]
    bufs = [I.make_activations(rows, C, H, "bf16", seed=0, block=0, prologue=True, device=dev)]
    bufs.append({k: torch.empty_like(v) for k, v in bufs[0].items()})
    ws = torch.empty(max(1, hc.workspace_size(rows, C, H, R, torch.bfloat16, flags)), dtype=torch.uint8, device=dev)
    for i in range(args.warmup + args.steps):
        src, dst, w = bufs[i % 2], bufs[(i + 1) % 2], weights[i % 4]
        hc.lowrank_mix(src["streams"], w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"], src["prev_out"],
                       src["prev_gate"], num_branches=C, flags=flags,
                       out=(dst["prev_out"], dst["prev_gate"], dst["streams"]), workspace=ws, **QWEN)
    torch.cuda.synchronize()
    return {"profile_case": f"decode rows={rows} bf16, 4 weight sets, {args.warmup}+{args.steps} eager blocks"}


DOWN_POINTS = ("entry", "weights issued", "dependency wait returned", "S pass done", "inverse RMS stored",
               "weights landed", "MMA operands ready", "MMA done", "cluster exchange landed", "partial sums written")
UP_POINTS = ("entry", "prefetches issued", "dependency wait returned", "partial sums landed", "MMA operands ready",
             "MMA done", "pre-mix products landed", "pre_output written")


def phase_report(st, n_down, n_up, blocks):
    """Reduce phase stamps st[block][kernel][cta][point][gt, clock] (int64) to
    per-phase durations (ns: SM cycles converted with each CTA's own clock
    rate) and the hand-offs between the kernels (globaltimer)."""
    import numpy as np
    out = {}
    for kname, k, n, pts, last in (("down", 0, n_down, DOWN_POINTS, 9), ("up", 1, n_up, UP_POINTS, 7)):
        s = st[blocks, k, :n, :, :].astype(np.float64)          # (blocks, ctas, points, 2)
        ns_per_cycle = (s[:, :, last, 0] - s[:, :, 0, 0]) / np.maximum(1.0, s[:, :, last, 1] - s[:, :, 0, 1])
        rows = {}
        for p in range(1, last + 1):
            d = (s[:, :, p, 1] - s[:, :, p - 1, 1]) * ns_per_cycle
            rows[f"{p - 1}->{p} {pts[p]}"] = {"mean_ns": round(float(d.mean()), 1),
                                              "mean_of_block_max_ns": round(float(d.max(1).mean()), 1)}
        out[kname] = rows
        out[f"{kname}_mhz"] = round(float(1e3 / np.median(ns_per_cycle)), 1)
    gt = st[:, :, :, :, 0].astype(np.float64)
    down_end = gt[:, 0, :n_down, 9].max(1)
    down_wait = gt[:, 0, :n_down, 2]
    up_wait = gt[:, 1, :n_up, 2]
    up_end = gt[:, 1, :n_up, 7].max(1)
    b = np.array(blocks)
    bp = b[b > 0]
    out["handoff_ns"] = {
        "down wait returned (first CTA) after the previous block's last up CTA ended":
            round(float((down_wait[bp].min(1) - up_end[bp - 1]).mean()), 1),
        "down wait returned (last CTA) after the previous block's last up CTA ended":
            round(float((down_wait[bp].max(1) - up_end[bp - 1]).mean()), 1),
        "up wait returned (first CTA) after the last down CTA ended":
            round(float((up_wait[b].min(1) - down_end[b]).mean()), 1),
        "up wait returned (last CTA) after the last down CTA ended":
            round(float((up_wait[b].max(1) - down_end[b]).mean()), 1),
        "block period (last up CTA end to the next)": round(float((up_end[bp] - up_end[bp - 1]).mean()), 1),
        "down critical path (last wait return to last end)":
            round(float((down_end[b] - down_wait[b].max(1)).mean()), 1),
        "up critical path (last wait return to last end)": round(float((up_end[b] - up_wait[b].max(1)).mean()), 1)}
    steps = np.diff(np.unique(gt[b, 0, :n_down, :10].ravel()))
    out["globaltimer_step_ns"] = float(steps[steps > 0].min()) if (steps > 0).any() else None
    return out


def profile_phases(args, hc, I, dev, rows, flags):
    """Phase clocks of the decode pair (hc_debug_phase_clocks): a 96-block
    chain over 96 weight sets captured as one CUDA graph with the timed
    kernels, replayed 5 times; the last replay's stamps are reduced over the
    steady-state blocks 8..87. The timed kernels compute the same results and
    add only the stamps; this is a diagnostic, not a benchmark result."""
    import numpy as np
    import torch
    from hyper_connection_rank_gb300 import _binding as B
    L = B.lib()
    weights = [I.make_weights(C, H, R, "bf16", seed=0, block=i, device=dev) for i in range(NSETS)]
    bufs = [I.make_activations(rows, C, H, "bf16", seed=0, block=0, prologue=True, device=dev)]
    bufs.append({k: torch.empty_like(v) for k, v in bufs[0].items()})
    ws = torch.empty(max(1, hc.workspace_size(rows, C, H, R, torch.bfloat16, flags)), dtype=torch.uint8, device=dev)

    def step(i):
        src, dst, w = bufs[i % 2], bufs[(i + 1) % 2], weights[i % NSETS]
        hc.lowrank_mix(src["streams"], w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"], src["prev_out"],
                       src["prev_gate"], num_branches=C, flags=flags,
                       out=(dst["prev_out"], dst["prev_gate"], dst["streams"]), workspace=ws, **QWEN)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    slot = L.hc_debug_phase_clocks(None, 0)
    stamps = torch.zeros(NSETS * slot // 8, dtype=torch.int64, device=dev)
    L.hc_debug_phase_clocks(stamps.data_ptr(), NSETS * slot)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    try:
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(NSETS):
                    step(i)
    finally:
        L.hc_debug_phase_clocks(None, 0)
    torch.cuda.current_stream(dev).wait_stream(s)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    st = stamps.view(NSETS, 2, 256, 10, 2).cpu().numpy()
    n_down = int((st[0, 0, :, 0, 0] != 0).sum())
    n_up = int((st[0, 1, :, 0, 0] != 0).sum())
    rep = phase_report(st, n_down, n_up, list(range(8, 88)))
    return {"profile_case": f"decode phase clocks, rows={rows} bf16, 96-block graph, blocks 8..87 of the last of "
                            f"5 replays", "ctas": {"down": n_down, "up": n_up}, "phases": rep}


PREFILL_CONFIGS = {"bf16_c4": ("bf16", 4, 2560), "f16_c8": ("f16", 8, 1280)}


def profile_prefill(args, hc, I, dev):
    """Profiler case for the prefill path: one of the two prefill blocks
    (--prefill-config: bf16 C=4 H=2560, or fp16 C=8 H=1280; R=320) at
    --prefill-rows rows (8192 by default), warmup + steps eager calls through
    the public API."""
    import torch
    dt, Cp, Hp = PREFILL_CONFIGS[args.prefill_config]
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dt]
    rows = args.prefill_rows
    d = I.make_block(rows, Cp, Hp, R, dt, seed=0, prologue=True, device=dev)
    ws = torch.empty(hc.workspace_size(rows, Cp, Hp, R, tdt), dtype=torch.uint8, device=dev)
    out = (torch.empty(rows, Hp, dtype=tdt, device=dev), torch.empty(rows, Cp, dtype=tdt, device=dev),
           torch.empty(rows, Cp * Hp, dtype=tdt, device=dev))
    for _ in range(args.warmup + args.steps):
        hc.lowrank_mix(d["streams"], d["norm_scale"], d["down_w"], d["up_w"], d["inject_w"], d["prev_out"],
                       d["prev_gate"], num_branches=Cp, out=out, workspace=ws, **QWEN)
    torch.cuda.synchronize()
    return {"profile_case": f"prefill rows={rows} {dt} C={Cp} H={Hp}, {args.warmup}+{args.steps} eager blocks"}


def profile_rowops(args, hc, I, dev):
    """Profiler case for the two row operations: the row inverse RMS on 8192 x
    16384 bf16 (268 MB) and the Engram gate on 8192 x 4 x 4096 fp16 (872 MB),
    warmup + steps eager calls each, alternating."""
    import torch
    x = I.make_inv_rms_input(8192, 16384, "bf16", seed=0, device=dev)
    o = torch.empty(8192, dtype=torch.float32, device=dev)
    d = I.make_engram_inputs(8192, 4, 4096, "f16", seed=0, device=dev)
    eo = torch.empty_like(d["key"])
    for _ in range(args.warmup + args.steps):
        hc.inv_rms(x, 1e-6, out=o)
        hc.engram_gate(d["key"], d["query"], d["value"], d["key_scale"], d["query_scale"], 1e-5, out=eo)
    torch.cuda.synchronize()
    return {"profile_case": f"row ops (inv_rms 8192x16384 bf16, engram 8192x4x4096 f16), "
                            f"{args.warmup}+{args.steps} eager calls each"}


def e2e_measure(args, hc, I, weights, dev, flags):
    """Same metric through the C ABI with host buffers: every step copies its
    inputs host->device from pinned memory, calls hc_lowrank_mix, and reads its
    outputs back device->host."""
    import torch
    rows = 1
    src = I.make_activations(rows, C, H, "bf16", seed=1, block=0, prologue=True, device="cpu")
    # The step's inputs live in one pinned host buffer and one device buffer
    # (streams | prev_out | prev_gate, each 16-byte aligned), its outputs
    # likewise (pre_output | post_gate | streams_out): one copy each way.
    def packed(shapes, device, pin):
        sizes = [int(torch.Size(s).numel()) for s in shapes]
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += (n + 7) // 8 * 8
        buf = torch.empty(o, dtype=torch.bfloat16, device=device)
        if pin:
            buf = buf.pin_memory()
        return buf, [buf[a:a + n].view(*s) for a, n, s in zip(offs, sizes, shapes)]
    in_shapes = [src[k].shape for k in ("streams", "prev_out", "prev_gate")]
    out_shapes = [(rows, H), (rows, C), (rows, C * H)]
    host_in_buf, host_in = packed(in_shapes, "cpu", True)
    for t, k in zip(host_in, ("streams", "prev_out", "prev_gate")):
        t.copy_(src[k])
    dev_in_buf, dev_in = packed(in_shapes, dev, False)
    host_out_buf, host_out = packed(out_shapes, "cpu", True)
    dev_out_buf, dev_out = packed(out_shapes, dev, False)
    ws = torch.empty(max(1, hc.workspace_size(rows, C, H, R, torch.bfloat16, flags)), dtype=torch.uint8, device=dev)
    n = max(1, min(args.steps, args.e2e_steps))
    # the C-ABI call itself (hc_lowrank_mix through ctypes), its attribute
    # struct and device addresses prepared once: what a host program calling
    # the library pays per block, plus the two copies
    from hyper_connection_rank_gb300 import _binding as B
    attrs = B.make_attrs(flags=flags, **QWEN)
    stream = torch.cuda.current_stream(dev).cuda_stream
    act = [t.data_ptr() for t in dev_in]
    outs = [t.data_ptr() for t in dev_out]
    wps = [[w[k].data_ptr() for k in ("norm_scale", "down_w", "up_w", "inject_w")] for w in weights]
    call = B.raw_call
    wsp, wsn = ws.data_ptr(), ws.numel()

    def one(i):
        dev_in_buf.copy_(host_in_buf, non_blocking=True)
        ns, dw, uw, iw = wps[i % NSETS]
        st = call(act[0], ns, dw, uw, iw, act[1], act[2], rows, C, H, R, attrs, B.HC_BF16, outs[0], outs[1], outs[2],
                  wsp, wsn, stream)
        if st != 0:
            B.check(st)
        host_out_buf.copy_(dev_out_buf, non_blocking=True)

    for i in range(max(3, args.warmup)):
        one(i)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(s)
    for i in range(n):
        one(i)
    e1.record(s)
    e1.synchronize()
    wall = time.perf_counter() - t0
    t = e0.elapsed_time(e1) / 1000.0
    bi = host_in_buf.numel() * host_in_buf.element_size()
    bo = host_out_buf.numel() * host_out_buf.element_size()
    return {"value": round(rows * n / t, 1), "unit": "rows/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": n, "us_per_step": round(1e6 * t / n, 3), "wall_us_per_step": round(1e6 * wall / n, 3),
            "api": "hc_lowrank_mix (C ABI, through ctypes) with host buffers: one pinned H2D copy, the block, one D2H copy per step; eager launches"}


def host_cpu():
    """Host processor as the benchmark saw it: logical cores, architecture
    and model name (from lscpu, else /proc/cpuinfo)."""
    import platform
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                model = line.split(":", 1)[1].strip()
                if line.startswith("Model name"):
                    break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model and os.path.exists("/proc/cpuinfo"):
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                model = line.split(":", 1)[1].strip()
                break
    return {"nproc": os.cpu_count(), "machine": platform.machine(), "model": model}


def _oracle_rate(run, seconds, min_calls=2):
    """Calls of run() until about `seconds` have passed: (calls, elapsed)."""
    n, t0 = 0, time.perf_counter()
    while True:
        run(n)
        n += 1
        el = time.perf_counter() - t0
        if (el >= seconds and n >= min_calls) or n >= 100000:
            return n, el


def cpu_baseline(seconds):
    """The oracle, as it stands, on bounded samples of the benchmark's
    configurations, on the host cores of this machine.

    Headline (the line's own workload, single-threaded: the oracle splits a
    call across threads by rows, and a chain of one-row blocks has one row per
    call): chained rows=1 bf16 decode blocks over 2 weight sets for about
    `seconds`. Then on all host cores: nproc independent one-row chains as one
    nproc-row call per block (the oracle's row threads), and a sample of rows
    of each 8192-row prefill block (C=4, H=2560 bf16; C=8, H=1280 fp16), one
    thread and all threads. Rates are rows/s."""
    import numpy as np
    import torch

    import oracle
    from hyper_connection_rank_gb300 import inputs as I
    oracle.build()
    info = host_cpu()
    ncores = max(1, int(info["nproc"] or 1))
    codes = lambda t: None if t is None else t.contiguous().view(torch.int16).numpy().view(np.uint16)

    def chain(rows, nthreads, secs):
        ws = [{k: codes(v) for k, v in I.make_weights(C, H, R, "bf16", seed=0, block=i).items()} for i in range(2)]
        act = [{k: codes(v) for k, v in I.make_activations(rows, C, H, "bf16", seed=0, block=0,
                                                          prologue=True).items()}]

        def one(n):
            w, a = ws[n % 2], act[0]
            pre, post, sout = oracle.lowrank_mix(a["streams"], w["norm_scale"], w["down_w"], w["up_w"],
                                                 w["inject_w"], a["prev_out"], a["prev_gate"], num_branches=C,
                                                 dtype=oracle.DT_BF16, nthreads=nthreads, **QWEN)
            act[0] = {"streams": sout, "prev_out": pre, "prev_gate": post}
        return _oracle_rate(one, secs, min_calls=3)

    n, el = chain(1, 1, seconds)
    res = {"value": round(n / el, 2), "unit": "rows/s", "cores": 1, "kind": "oracle",
           "sample": f"{n} chained decode blocks (rows=1, bf16, C=4, H=2560, R=320) over 2 weight sets, "
                     f"{el:.1f} s on 1 host thread", "us_per_block": round(1e6 * el / n, 1), "host": info}
    lines = {}
    n, el = chain(ncores, ncores, seconds / 2)
    lines["decode_rows1_chain_bf16"] = {
        "rows_per_s": round(n * ncores / el, 2), "threads": ncores,
        "sample": f"{ncores} independent one-row chains as {n} calls of {ncores} rows ({el:.1f} s)"}
    for dt, Cp, Hp in (("bf16", 4, 2560), ("f16", 8, 1280)):
        code = {"bf16": oracle.DT_BF16, "f16": oracle.DT_F16}[dt]
        w = {k: codes(v) for k, v in I.make_weights(Cp, Hp, R, dt, seed=0, block=0).items()}
        full = I.make_block(max(4 * ncores, 8), Cp, Hp, R, dt, seed=0, prologue=True)
        for threads, rows in ((1, 4), (ncores, 4 * ncores)):
            a = {k: codes(full[k][:rows]) for k in ("streams", "prev_out", "prev_gate")}

            def one(_n, a=a, threads=threads):
                oracle.lowrank_mix(a["streams"], w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"],
                                   a["prev_out"], a["prev_gate"], num_branches=Cp, dtype=code, nthreads=threads,
                                   **QWEN)
            n, el = _oracle_rate(one, seconds / 4, min_calls=1)
            lines[f"prefill_rows8192_C{Cp}_H{Hp}_{dt}_{'1thread' if threads == 1 else 'all_cores'}"] = {
                "rows_per_s": round(n * rows / el, 2), "threads": threads,
                "us_per_8192_row_block": round(1e6 * el / (n * rows) * 8192, 1),
                "sample": f"{n} calls of {rows} rows of the 8192-row block ({el:.1f} s)"}
    res["other_configs"] = lines
    return res


def sweep(hc, I, dev, pk):
    """Other configurations of the metric (context lines, not the headline):
    decode rows 1/2/4/8 in bf16 and fp16 (96-block graphs; us/block also as the
    slope between 96- and 48-block graphs, min over 15 x 10 replays), the
    8192-row prefill blocks, and the two companion row operations."""
    import torch
    out = {}
    flags = hc.HC_FLAG_WEIGHTS_STATIC
    for dt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        weights = [I.make_weights(C, H, R, dt, seed=0, block=i, device=dev) for i in range(NSETS)]
        # rows 1-8 take the decode path; 16 / 64 / 256 (bf16) the prefill path's
        # small-batch regime, measured the same way (weights rotate past L2)
        for rows in ((1, 2, 4, 8, 16, 64, 256) if dt == "bf16" else (1, 2, 4, 8)):
            bufs = [I.make_activations(rows, C, H, dt, seed=0, block=0, prologue=True, device=dev)]
            bufs.append({k: torch.empty_like(v) for k, v in bufs[0].items()})
            ws = torch.empty(max(1, hc.workspace_size(rows, C, H, R, tdt, flags)), dtype=torch.uint8, device=dev)

            def step(i):
                src, dst, w = bufs[i % 2], bufs[(i + 1) % 2], weights[i % NSETS]
                hc.lowrank_mix(src["streams"], w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"],
                               src["prev_out"], src["prev_gate"], num_branches=C, flags=flags,
                               out=(dst["prev_out"], dst["prev_gate"], dst["streams"]), workspace=ws, **QWEN)

            graphs = {}
            for n in (96, 48):
                step(0)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                s = torch.cuda.Stream(dev)
                s.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        for i in range(n):
                            step(i)
                torch.cuda.current_stream(dev).wait_stream(s)
                graphs[n] = g
            best = {}
            for n, g in graphs.items():
                g.replay()
                torch.cuda.synchronize()
                ts = []
                for _ in range(15):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for _ in range(10):
                        g.replay()
                    e1.record()
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1) / 10)
                best[n] = min(ts)
            us96 = 1000 * best[96] / 96
            slope = 1000 * (best[96] - best[48]) / 48
            b = block_bytes(rows, C, H, R, 2)
            name = f"decode_rows{rows}_{dt}" if rows <= 8 else f"rows{rows}_{dt}"
            out[name] = {
                "path": hc.PATH_NAMES[hc.path(rows, C, H, R, tdt, flags)],
                "us_per_block": round(us96, 3), "us_per_block_slope": round(slope, 3),
                "rows_per_s": round(rows / (us96 * 1e-6), 1),
                "hbm_frac": round(b / (us96 * 1e-6) / 1e9 / pk["hbm"], 4),
                "hbm_frac_slope": round(b / (slope * 1e-6) / 1e9 / pk["hbm"], 4) if slope > 0 else None}
            del graphs
        del weights
        torch.cuda.empty_cache()
    for dt, tdt, Cp, Hp in (("bf16", torch.bfloat16, 4, 2560), ("f16", torch.float16, 8, 1280)):
        rows = 8192
        d = I.make_block(rows, Cp, Hp, R, dt, seed=0, prologue=True, device=dev)
        pre = torch.empty(rows, Hp, dtype=tdt, device=dev)
        post = torch.empty(rows, Cp, dtype=tdt, device=dev)
        sout = torch.empty(rows, Cp * Hp, dtype=tdt, device=dev)
        ws = torch.empty(max(1, hc.workspace_size(rows, Cp, Hp, R, tdt)), dtype=torch.uint8, device=dev)

        def call():
            hc.lowrank_mix(d["streams"], d["norm_scale"], d["down_w"], d["up_w"], d["inject_w"], d["prev_out"],
                           d["prev_gate"], num_branches=Cp, out=(pre, post, sout), workspace=ws, **QWEN)

        # four back-to-back blocks per graph replay (inputs far larger than L2)
        tmin, tmed = graph_time([call] * 4, reps=10)
        t = tmin * 1e-6
        b, f = block_bytes(rows, Cp, Hp, R, 2), block_flops(rows, Cp, Hp, R)
        t_roof = max(b / (pk["hbm"] * 1e9), f / (pk["bf16"] * 1e12))
        out[f"prefill_rows{rows}_C{Cp}_H{Hp}_{dt}"] = {
            "path": hc.PATH_NAMES[hc.path(rows, Cp, Hp, R, tdt)],
            "us_per_block": round(1e6 * t, 2), "us_per_block_median": round(tmed, 2),
            "rows_per_s": round(rows / t, 1), "hbm_frac": round(b / t / 1e9 / pk["hbm"], 4),
            "tensor_frac": round(f / t / 1e12 / pk["bf16"], 4), "roofline_frac": round(t_roof / t, 4)}
        del d
        torch.cuda.empty_cache()
    out.update(sweep_row_ops(hc, I, dev, pk))
    return out


def graph_time(calls, reps=15):
    """Device time (us) per call of the list `calls`, captured once into a CUDA
    graph and replayed: min and median over `reps` replays, so no host-side
    launch overhead enters the figure."""
    import torch
    dev = torch.cuda.current_device()
    for c in calls[:3]:
        c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for c in calls:
                c()
    torch.cuda.current_stream(dev).wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ts.append(1000 * e0.elapsed_time(e1) / len(calls))
    del g
    return min(ts), statistics.median(ts)


def timed_rotating(make, call, bytes_each, target=400 << 20, max_calls=64):
    """Device time (us) per call of call(inputs), the calls cycling through
    enough copies of the inputs (made by `make`) to span `target` bytes (about
    three L2s): each call reads data the previous ones evicted, and no flush
    leaves dirty lines to be written back during a timed call. Timed as one
    CUDA graph of the calls (graph_time)."""
    ncopy = max(1, -(-target // bytes_each))
    copies = [make(i) for i in range(ncopy)]
    n = max(ncopy, min(max_calls, 4 * ncopy))
    tmin, tmed = graph_time([(lambda a=copies[i % ncopy]: call(a)) for i in range(n)])
    del copies
    return tmin, tmed


def sweep_row_ops(hc, I, dev, pk):
    """The two companion row operations, each call on inputs not in L2 (the
    calls cycle through copies spanning about three L2s): the row inverse RMS
    at the shapes FreeToken PR #101 measures (hc_dim 16384, 64 to 8192 rows,
    bf16) and the Engram gate at 8192 tokens x hc_mult 4 x hidden 4096 (fp16).
    Bytes = what each must read and write once."""
    import torch
    out = {}
    for rows in (64, 512, 4096, 8192):
        dim = 16384
        b = rows * dim * 2 + rows * 4

        def make(i, rows=rows, dim=dim):
            return (I.make_inv_rms_input(rows, dim, "bf16", seed=i, device=dev),
                    torch.empty(rows, dtype=torch.float32, device=dev))

        tmin, tmed = timed_rotating(make, lambda a: hc.inv_rms(a[0], 1e-6, out=a[1]), b)
        out[f"inv_rms_rows{rows}_dim{dim}_bf16"] = {
            "us": round(tmin, 2), "us_median": round(tmed, 2), "bytes": b,
            "GB_s": round(b / (tmin * 1e-6) / 1e9, 1), "hbm_frac": round(b / (tmin * 1e-6) / 1e9 / pk["hbm"], 4)}
        torch.cuda.empty_cache()
    rows, M, D = 8192, 4, 4096
    b = (3 * rows * M * D + rows * D + 2 * M * D) * 2

    def make_e(i):
        d = I.make_engram_inputs(rows, M, D, "f16", seed=i, device=dev)
        d["out"] = torch.empty_like(d["key"])
        return d

    tmin, tmed = timed_rotating(make_e, lambda d: hc.engram_gate(d["key"], d["query"], d["value"], d["key_scale"],
                                                                 d["query_scale"], 1e-5, out=d["out"]), b)
    out[f"engram_gate_rows{rows}_M{M}_D{D}_f16"] = {
        "us": round(tmin, 2), "us_median": round(tmed, 2), "bytes": b,
        "GB_s": round(b / (tmin * 1e-6) / 1e9, 1), "hbm_frac": round(b / (tmin * 1e-6) / 1e9 / pk["hbm"], 4)}
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------- reference arm --

def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the same workload, metric and
    unit: chained rows=1 bf16 blocks, timed on the host cores. Steps are capped
    so the run ends within a few minutes; the metric is a rate."""
    if rank != 0:
        return None
    cap_s = args.ref_seconds
    import numpy as np
    import torch

    import oracle
    from hyper_connection_rank_gb300 import inputs as I
    oracle.build()
    codes = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    ws = [{k: codes(v) for k, v in I.make_weights(C, H, R, "bf16", seed=0, block=i).items()} for i in range(2)]
    act = {k: codes(v) for k, v in I.make_activations(1, C, H, "bf16", seed=0, block=0, prologue=True).items()}

    def one(i, act):
        w = ws[i % 2]
        pre, post, sout = oracle.lowrank_mix(act["streams"], w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"],
                                             act["prev_out"], act["prev_gate"], num_branches=C,
                                             dtype=oracle.DT_BF16, nthreads=1, **QWEN)
        return {"streams": sout, "prev_out": pre, "prev_gate": post}

    for i in range(args.warmup):
        act = one(i, act)
    n, t0 = 0, time.perf_counter()
    while n < args.steps:
        act = one(n, act)
        n += 1
        if time.perf_counter() - t0 > cap_s:
            break
    el = time.perf_counter() - t0
    v = n / el
    return {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "steps_timed": n, "warmup": args.warmup, "ms_per_step": 1000 * el / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": WORKLOAD.replace("graph replay", "CPU oracle, 2 weight sets"),
                                            "rows": 1, "C": C, "H": H, "R": R},
            "cpu_baseline": {"value": round(v, 2), "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n} chained decode blocks on 1 host thread ({el:.1f} s)",
                             "host": host_cpu()},
            "e2e": {"value": round(v, 2), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=96 * 2000)
    ap.add_argument("--warmup", type=int, default=96)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--rows", type=int, default=1, help="decode rows per block (1..8)")
    ap.add_argument("--prefill-config", choices=("bf16_c4", "f16_c8"), default="bf16_c4",
                    help="block of the prefill profile case")
    ap.add_argument("--prefill-rows", type=int, default=8192, help="rows of the prefill profile case")
    ap.add_argument("--profile-case", nargs="?", const="decode", choices=("decode", "phases", "sync", "prefill", "rowops"),
                    help="small eager case for profiler captures (not a benchmark result)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
