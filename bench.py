"""Benchmark of the ring-attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload striped-128k] [--no-e2e] [--no-cpu-baseline]

One step = one ring_attn_fwd over the whole workload: pack K/V, P ring steps
(one block-partial kernel each, K/V rotated by device-to-device copies on a
side stream), finalize fused into the last step.  Default workload: B=1,
H=16, N=131072, d=128, P=16 striped shards, causal, Q/K/V ~ N(0,1) bf16 with
1% of key rows scaled by 8 (synthetic, seeded).  Inputs (3 x 0.5 GB) are
larger than the 129 MB L2, so no flush is needed between steps.

Metric: causal-adjusted attention TFLOP/s = 4 d B H N(N+1)/2 / t (also
tokens/s and % of bf16 peak).  With --gpus N (torchrun) every rank runs an
independent replica of the workload (the ring is simulated on one device;
no data-path collective); the value is the sum over ranks of the work
divided by the slowest rank's time.

--impl reference times the float64 CPU oracle (dense attention by
definition) on a bounded sample of query rows of the same workload, on the
host cores, in the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal-adjusted attention TFLOP/s and % of GB300 bf16 peak; tokens/s (1 GPU)"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
KERNEL_SOURCE = os.path.join(ROOT, "ring_sequence_parallelism_gb300", "csrc", "block_partial.cu")
BWD_SOURCE = os.path.join(ROOT, "ring_sequence_parallelism_gb300", "csrc", "block_backward.cu")
LAP_SOURCE = os.path.join(ROOT, "ring_sequence_parallelism_gb300", "csrc", "block_lap.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="striped-128k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--bwd", action="store_true", help="time the ring backward (ring_attn_bwd) instead")
    ap.add_argument("--bwd-per-step", action="store_true",
                    help="with --bwd: one dK/dV and one dQ launch per ring step (RING_OPT_BWD_LAP 0) instead "
                         "of one launch per kernel for the whole ring")
    ap.add_argument("--merge", action="store_true",
                    help="time the standalone merge of two fp32 states (ring_attn_merge) of one shard instead")
    ap.add_argument("--decode", type=int, default=0, metavar="LQ",
                    help="measure split-K/V decode of LQ new queries over the workload's K/V cache instead")
    ap.add_argument("--imbalance", action="store_true",
                    help="print only the per-shard work and time of the 8K causal workloads (contiguous, "
                         "striped, zigzag)")
    ap.add_argument("--fwd-lap", action="store_true",
                    help="run the forward as one launch for the whole ring (RING_OPT_FWD_LAP 1) instead of one "
                         "step kernel per ring step")
    ap.add_argument("--no-extra", action="store_true",
                    help="leave out the sub-records of the default line (side-stream rotation, per-shard "
                         "imbalance, the other workloads)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, world: int) -> float:
    """Max of a per-rank float over all ranks (the slowest rank's time).
    Uses the process group's backend: a CUDA tensor for nccl, CPU for gloo."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank_step: float, ms_max: float) -> float:
    """Work of all ranks (each runs one replica of the step) over the slowest rank's time."""
    return world * flops_per_rank_step / (ms_max * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(path=KERNEL_SOURCE):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(key: str, source=KERNEL_SOURCE):
    """ncu DRAM bytes per launch of a kernel (entry `key` of the traffic
    record), if taken on this exact kernel source (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(key)
    if not e or e.get("kernel_sha256_16") != source_hash(source):
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------- clocks
def host_link_rates(torch, mib=256, reps=3):
    """Pinned host-to-device and device-to-host copy rates (GB/s, median of
    `reps` copies of `mib` MiB), to read the end-to-end figure against."""
    n = mib << 20
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    rates = {}
    for name, fn in (("h2d", lambda: d.copy_(h, non_blocking=True)), ("d2h", lambda: h.copy_(d, non_blocking=True))):
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        rates[name] = round(n / sorted(ts)[len(ts) // 2] / 1e6, 1)
    del h, d
    return rates


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- oracle leg
def allowed_keys(w, rows) -> int:
    """Allowed keys summed over the sampled query rows (causal mask, window
    and documents of the workload)."""
    import numpy as np

    rows = np.asarray(rows, dtype=np.int64)
    lo = np.zeros_like(rows)
    hi = np.full_like(rows, w.N - 1)
    if w.causal:
        hi = rows.copy()
        if w.window:
            lo = np.maximum(lo, rows - w.window + 1)
    if w.doc_len:
        b = np.asarray(w.segments(), dtype=np.int64)
        x = np.searchsorted(b, rows, side="right") - 1
        lo = np.maximum(lo, b[x])
        hi = np.minimum(hi, b[x + 1] - 1)
    return int(np.maximum(0, hi - lo + 1).sum())


def oracle_sample(w, q, k, v, seconds: float, seed: int = 4242):
    """Time the float64 oracle on a bounded sample of query rows.  Returns
    (TFLOP/s, rows per second, threads, description, wall seconds)."""
    import oracle
    from ring_sequence_parallelism_gb300.inputs import sample_rows

    from ring_sequence_parallelism_gb300.inputs import expand_kv

    orc = oracle.default()
    BH = w.B * w.H
    k, v = expand_kv(k, w.H), expand_kv(v, w.H)  # grouped K/V heads written out per query head
    qf, kf, vf = (oracle.bf16_bits(x.reshape(BH, w.N, w.d)) for x in (q, k, v))
    rows_per_head = 2
    t_used = 0.0
    flops = 0
    while True:
        rows = sample_rows(w.N, rows_per_head, seed=seed).numpy()
        t0 = time.perf_counter()
        orc.dense(qf, kf, vf, w.causal, rows=rows, window=w.window, segments=w.segments())
        t_used = time.perf_counter() - t0
        keys = allowed_keys(w, rows)
        flops = 4 * w.d * BH * int(keys)
        if t_used >= seconds / 4 or rows_per_head >= w.N:
            break
        rows_per_head = min(w.N, max(rows_per_head * 2, int(rows_per_head * seconds / max(t_used, 1e-3) / 2)))
    desc = (f"{rows_per_head} seeded query rows per head x {BH} heads of {w.name} "
            f"({rows_per_head * BH} rows, {flops / 1e9:.1f} GFLOP, dense oracle, float64)")
    return flops / t_used / 1e12, rows_per_head * BH / t_used, orc.threads(), desc, t_used, rows_per_head


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch

    from ring_sequence_parallelism_gb300.inputs import make_workload

    q, k, v = make_workload(w)
    per_step_seconds = max(1.0, min(20.0, 90.0 / max(1, args.steps + args.warmup)))
    # calibrate the sample once, then time W + K steps of that sample
    _, _, threads, desc, _, rph = oracle_sample(w, q, k, v, per_step_seconds)
    import oracle
    from ring_sequence_parallelism_gb300.inputs import sample_rows

    from ring_sequence_parallelism_gb300.inputs import expand_kv

    orc = oracle.default()
    BH = w.B * w.H
    k, v = expand_kv(k, w.H), expand_kv(v, w.H)
    qf, kf, vf = (oracle.bf16_bits(x.reshape(BH, w.N, w.d)) for x in (q, k, v))
    times, flops = [], 0
    for i in range(args.warmup + args.steps):
        rows = sample_rows(w.N, rph, seed=5000 + i).numpy()
        keys = allowed_keys(w, rows)
        t0 = time.perf_counter()
        orc.dense(qf, kf, vf, w.causal, rows=rows, window=w.window, segments=w.segments())
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            flops += 4 * w.d * BH * int(keys)
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc + "; each step a fresh row sample of that size"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    del torch


def config_of(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.kv_heads, "N": w.N, "d": w.d, "P": w.P,
            "layout": w.layout, "causal": w.causal, "window": w.window,
            "documents": len(w.segments()) - 1 if w.doc_len else 1, "global_batch": w.B, "seq_len": w.N,
            "inputs": "Q,K,V ~ N(0,1) rounded to bf16" + (", 1% of key rows x8" if w.key_boost_frac else ""),
            "l2": l2_note(w)}


def l2_note(w):
    gb = w.B * w.H * w.N * w.d * 2 / 1e9
    if gb * 1e3 > 129:
        return "inputs (3 x %.2f GB bf16) larger than the 129 MB L2; no flush" % gb
    return "inputs (3 x %.1f MB bf16) fit in L2: small case, not a timed workload" % (gb * 1e3)


class L2Flush:
    """Evicts the inputs from the 129 MB L2 between timed calls: writes a
    256 MB buffer, then reads another, so L2 ends up holding clean lines (a
    write alone would leave 129 MB of dirty lines, written back to HBM
    during the next timed kernel)."""

    def __init__(self):
        import torch

        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.fill_(1)
        return self.r.sum()


# ------------------------------------------------------------- sub-records
def measure_imbalance(names=("contiguous-8k", "striped-8k", "zigzag-8k"), reps=5):
    """Per-shard causal work and time ([GRA] "The causal mask wrecks the load
    balance"; [RA-CN] "Causal Attention 让环不再完全对称" and
    "如何判断通信是否真的被覆盖", which lists the spread of step times across
    ranks).  Every (shard r, step s) block partial is one
    ring_attn_block_partial launch on shard-major copies of the inputs,
    timed alone with CUDA events after an L2 flush, the stream backed up so
    the host's launch cost stays outside the events; the median over `reps`
    rounds.  A shard's time is the sum of its P launches (skipped blocks
    launch nothing); a synchronous ring step lasts as long as its slowest
    shard."""
    import statistics as st

    import torch

    import ring_sequence_parallelism_gb300 as ra
    from ring_sequence_parallelism_gb300 import report
    from ring_sequence_parallelism_gb300.inputs import WORKLOADS, make_workload

    flush = L2Flush()
    stream = torch.cuda.current_stream()
    res = []
    for name in names:
        w = WORKLOADS[name]
        q, k, v = make_workload(w)
        att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout, kv_heads=w.kv_heads)
        pos = [torch.tensor(report.shard_positions(w.layout, w.n, w.P, r)) for r in range(w.P)]
        Qs = [q[:, :, p].contiguous().cuda() for p in pos]
        Ks = [k[:, :, p].contiguous().cuda() for p in pos]
        Vs = [v[:, :, p].contiguous().cuda() for p in pos]
        states = [att.new_state() for _ in range(w.P)]
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(w.P)]
              for _ in range(w.P)]
        samples = [[[] for _ in range(w.P)] for _ in range(w.P)]  # [s][r]
        for rep in range(reps + 1):  # repetition 0 warms up
            for s in range(w.P):
                for r in range(w.P):
                    j = (r - s) % w.P
                    flush()
                    torch.cuda._sleep(100000)
                    e0, e1 = ev[s][r]
                    e0.record(stream)
                    att.block_partial(r, s, Qs[r], Ks[j], Vs[j], states[r], 1 if s > 0 else 0)
                    e1.record(stream)
            torch.cuda.synchronize()
            if rep:
                for s in range(w.P):
                    for r in range(w.P):
                        samples[s][r].append(ev[s][r][0].elapsed_time(ev[s][r][1]))
        att.check()
        t = [[st.median(samples[s][r]) for r in range(w.P)] for s in range(w.P)]
        shard_ms = [sum(t[s][r] for s in range(w.P)) for r in range(w.P)]
        pairs, tiles = att.shard_work()
        ring_ms = report.synchronous_ring_ms(t)
        balanced = sum(shard_ms) / w.P
        res.append({
            "workload": name, "layout": w.layout, "P": w.P, "n": w.n, "heads": w.B * w.H,
            "shard_pairs": pairs,
            "shard_pairs_closed_form": [w.B * w.H * x for x in report.shard_pairs_closed_form(w.layout, w.n, w.P)],
            "shard_tiles": tiles, "shard_ms": shard_ms,
            "pairs_max_over_min": report.imbalance(pairs), "ms_max_over_min": report.imbalance(shard_ms),
            "step_max_ms": [max(row) for row in t], "synchronous_ring_ms": ring_ms, "balanced_ms": balanced,
            "ring_over_balanced": ring_ms / balanced,
        })
        att.close()
        del Qs, Ks, Vs, states
    return {"method": "one ring_attn_block_partial launch per (shard, step), CUDA events, L2 flushed before "
                      f"each, median of {reps} rounds; shard time = sum of its launches; synchronous ring = sum "
                      "over steps of the slowest shard",
            "workloads": res}


def measure_side_stream_rotation(att, q, k, v, out, lse, w, warmup=3, steps=3):
    """RING_OPT_ROTATION = 1, the pages' double-buffered rotation as written
    ([RA-CN] "双缓冲是重叠成立的基础"; "如何判断通信是否真的被覆盖": compute
    waiting for the communication, communication waiting for the buffer's
    release): every step's K/V move is two cudaMemcpyAsync device-to-device
    copies per tensor on the side stream, ordered by events.  Reports the
    copy time and rate, the compute stream's exposed wait for each copy, and
    the side stream's wait for the buffer it fills."""
    import torch

    import ring_sequence_parallelism_gb300 as ra

    att.set_option(ra.RING_OPT_ROTATION, 1)
    att.set_option(ra.RING_OPT_TIMING, 1)
    try:
        for _ in range(warmup):
            att.fwd(q, k, v, out, lse)
        if warmup:
            att.timing()  # the timed calls below start a new record
        stream = torch.cuda.current_stream()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            att.fwd(q, k, v, out, lse)
        e1.record(stream)
        torch.cuda.synchronize()
        t = att.timing()
        att.check()
    finally:
        att.set_option(ra.RING_OPT_ROTATION, 2)
    ms = e0.elapsed_time(e1) / steps
    copy_bytes = 2 * 2 * w.B * w.kv_heads * w.N * w.d * 2  # K and V, every slot, read + written
    copies = [c for c in t["copy_ms"] if c > 0]
    return {
        "rotation": "side-stream cudaMemcpyAsync D2D, 2 per tensor per step, events landed/released",
        "ms_per_step": ms, "tflops": w.flops() / (ms * 1e-3) / 1e12,
        "step_kernel_ms": t["kernel_ms"], "copy_ms": t["copy_ms"], "copy_total_ms": sum(t["copy_ms"]),
        "copy_gbs_mean": (copy_bytes / (sum(copies) / len(copies) * 1e-3) / 1e9) if copies else None,
        "copy_bytes_each": copy_bytes,
        "exposed_wait_ms": t["wait_ms"], "exposed_wait_total_ms": sum(t["wait_ms"]),
        "release_wait_ms": t["release_wait_ms"], "release_wait_total_ms": sum(t["release_wait_ms"]),
    }


def measure_schedules(q, k, v, base, names=("striped-128k", "swa-128k", "packed-128k"), warmup=3, steps=5):
    """The step schedule (one kernel per ring step, state through HBM) and the
    lap (RING_OPT_FWD_LAP 1: one launch, state on chip) on workloads whose
    inputs are the given ones (the 128K workloads share their seed and
    recipe; they differ in the mask).  Inputs are larger than L2."""
    import torch

    import ring_sequence_parallelism_gb300 as ra
    from ring_sequence_parallelism_gb300.inputs import WORKLOADS

    stream = torch.cuda.current_stream()
    res = []
    for name in names:
        w = WORKLOADS[name]
        if (w.B, w.H, w.kv_heads, w.N, w.d, w.seed, w.key_boost_frac) != \
                (base.B, base.H, base.kv_heads, base.N, base.d, base.seed, base.key_boost_frac):
            continue
        att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout, kv_heads=w.kv_heads)
        if w.window:
            att.set_option(ra.RING_OPT_WINDOW, w.window)
        if w.doc_len:
            att.set_segments(w.segments())
        out = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
        rec = {"workload": name}
        for lap in (0, 1):
            att.set_option(ra.RING_OPT_FWD_LAP, lap)
            for _ in range(warmup):
                att.fwd(q, k, v, out, lse)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                att.fwd(q, k, v, out, lse)
            e1.record(stream)
            torch.cuda.synchronize()
            att.check()
            ms = e0.elapsed_time(e1) / steps
            rec["lap" if lap else "step"] = {"ms_per_step": ms, "tflops": w.flops() / (ms * 1e-3) / 1e12}
        rec["lap_speedup"] = rec["step"]["ms_per_step"] / rec["lap"]["ms_per_step"]
        res.append(rec)
        att.close()
        del out, lse
    return res


def measure_workloads(names, peak_burst, warmup=3):
    """Whole forwards of other workloads, inputs resident; inputs that fit in
    L2 are flushed (L2Flush) before each timed forward."""
    import torch

    import ring_sequence_parallelism_gb300 as ra
    from ring_sequence_parallelism_gb300.inputs import WORKLOADS, make_workload

    flush = L2Flush()
    stream = torch.cuda.current_stream()
    res = []
    for name in names:
        w = WORKLOADS[name]
        q, k, v = (x.to("cuda") for x in make_workload(w))
        att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout, kv_heads=w.kv_heads)
        out = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
        for _ in range(warmup):
            att.fwd(q, k, v, out, lse)
        att.check()
        small = 3 * w.B * w.H * w.N * w.d * 2 < (129 << 20)
        steps = 3 if w.N >= (1 << 20) else 10
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            if small:
                flush()
            e0.record(stream)
            att.fwd(q, k, v, out, lse)
            e1.record(stream)
        torch.cuda.synchronize()
        att.check()
        ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
        tf = w.flops() / (ms * 1e-3) / 1e12
        res.append({"workload": name, "config": config_of(w), "ms_per_step": ms, "steps": steps, "warmup": warmup,
                    "tflops": tf, "tokens_per_s": w.B * w.N / (ms * 1e-3), "frac_of_burst": tf / peak_burst,
                    "l2": "flushed before each forward" if small else "inputs larger than L2"})
        att.close()
        del q, k, v, out, lse
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------- our arm
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import ring_sequence_parallelism_gb300 as ra

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from ring_sequence_parallelism_gb300.inputs import make_workload

    q_h, k_h, v_h = make_workload(w, pin=True)
    q, k, v = (x.to("cuda", non_blocking=True) for x in (q_h, k_h, v_h))
    torch.cuda.synchronize()
    att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout, kv_heads=w.kv_heads)
    if w.window:
        att.set_option(ra.RING_OPT_WINDOW, w.window)
    if w.doc_len:
        att.set_segments(w.segments())
    if args.fwd_lap:
        att.set_option(ra.RING_OPT_FWD_LAP, 1)
    out = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    att.set_option(ra.RING_OPT_TIMING, 1)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        att.fwd(q, k, v, out, lse)
    att.check()
    if args.warmup:
        att.timing()  # a read: the record of the timed region starts with its first forward

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region: K forwards, inputs resident in HBM
    kernel_ms, copy_ms, wait_ms, pack_ms = [], [], [], []
    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            att.fwd(q, k, v, out, lse)
        e1.record(stream)
        barrier()
    t = att.timing()  # per-launch means over every forward of the timed region (launch stream)
    kernel_ms, copy_ms, wait_ms, pack_ms = t["kernel_ms"], t["copy_ms"], t["wait_ms"], t["pack_ms"]
    att.check()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world)

    flops = w.flops()
    value = whole_job_tflops(world, flops, ms_max)
    tokens_s = world * w.B * w.N / (ms_max * 1e-3)
    pk, pk_kind = peaks()

    # ---- roofline of the dominant kernel (the block-partial step kernel)
    step_flops = [4 * w.d * att.step_work(s)[0] for s in range(w.P)]
    k_total_ms = sum(kernel_ms)  # (lap: the one launch, in entry 0)
    achieved = sum(step_flops) / (k_total_ms * 1e-3) / 1e12
    peak_sus = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    traffic = traffic_for(f"{w.name}:fwd_lap", LAP_SOURCE) if args.fwd_lap else traffic_for(w.name)

    # ---- end to end through the public API, host buffers, copies in the timed region
    e2e = None
    if not args.no_e2e:
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        lse_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        link = host_link_rates(torch)
        att.set_option(ra.RING_OPT_TIMING, 0)
        att.fwd_host(q_h, k_h, v_h, out_h, lse_h)
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cpu_ms = []
        with ClockSampler(torch.cuda.current_device()) as e2e_clocks:
            f0.record(stream)
            for _ in range(args.steps):
                c0 = time.perf_counter()
                att.fwd_host(q_h, k_h, v_h, out_h, lse_h)
                cpu_ms.append((time.perf_counter() - c0) * 1e3)
            f1.record(stream)
            barrier()
            torch.cuda.synchronize()
        e2e_ms = max_over_ranks(f0.elapsed_time(f1) / args.steps, world)
        e2e = {"value": whole_job_tflops(world, flops, e2e_ms), "unit": "TFLOP/s",
               "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (q_h, k_h, v_h)),
               "d2h_bytes_per_step": out_h.numel() * 4 + lse_h.numel() * 4,
               "clocks": e2e_clocks.summary(),
               # pinned copy rates measured just before this leg (the host link is shared
               # with the machine's other jobs and varies between runs)
               "host_link_gbs": link,
               # host time to enqueue one call (all its copies, events and launches): the first
               # call of the loop (queues empty) and the median
               "enqueue_ms": {"first": round(cpu_ms[0], 3), "median": round(sorted(cpu_ms)[len(cpu_ms) // 2], 3)}}

    extra = {}
    if world == 1 and not args.no_extra:
        if not args.fwd_lap:
            extra["ring_mode1"] = measure_side_stream_rotation(att, q, k, v, out, lse, w)
        extra["schedules"] = measure_schedules(q, k, v, w)
        extra["imbalance"] = measure_imbalance()
        extra["workloads"] = measure_workloads(
            [x for x in ("noncausal-512", "contiguous-8k", "striped-8k", "zigzag-8k", "striped-1m") if x != w.name],
            peak_burst)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, rows_s, threads, desc, secs, _ = oracle_sample(w, q_h, k_h, v_h, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc,
               "rows_per_s": rows_s, "seconds": secs}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(w),
            "tokens_per_s": tokens_s,
            "pct_of_bf16_peak": {"sustained": 100 * value / world / peak_sus, "burst": 100 * value / world / peak_burst,
                                 "nominal_2250": 100 * value / world / 2250.0, "source": pk_kind},
            "schedule": "lap (one launch for the ring, state on chip, blocks read in place)" if args.fwd_lap else
                        "step (one kernel per ring step, blocks sent along the ring)",
            "roofline": {"bound": "tensor", "kernel": ("fwd_lap_kernel<128> (one launch for the ring)" if args.fwd_lap
                                                       else "block_partial_kernel<128> (one launch per ring step)"),
                         "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                         "frac": achieved / peak_burst, "peak_kind": f"bf16_tflops burst ({pk_kind})",
                         "frac_of_sustained": achieved / peak_sus, "traffic": traffic,
                         "launches_per_step": 1 if args.fwd_lap else w.P,
                         "avg_launch_ms": k_total_ms / (1 if args.fwd_lap else w.P)},
            "ring": {"step_kernel_ms": kernel_ms, "rotation_copy_ms": copy_ms, "exposed_wait_ms": wait_ms,
                     "pack_ms": pack_ms, "exposed_wait_total_ms": sum(wait_ms),
                     "rotation": "each step kernel sends its K/V blocks to the next shard's slot "
                                 "(TMA stores from shared memory); side-stream copies only for shards "
                                 "with no work in a step",
                     "rotation_bytes_per_step": 2 * w.B * w.H * w.N * w.d * 2},
            "clocks": clocks.summary(),
            # pack + P step kernels; the lap reads its blocks in place (packs only for zigzag)
            "gpu_launches": args.steps * ((1 + (1 if w.layout == "zigzag" else 0)) if args.fwd_lap else 1 + w.P),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    att.close()
    if world > 1:
        dist.destroy_process_group()


def run_decode(args, w):
    """Split-K/V decode / short-query prefill (ring_attn_decode): LQ queries
    at the end of the workload's sequence over its K/V cache, inputs resident,
    K calls timed with CUDA events.  The roofline is HBM for short queries:
    algorithmic bytes per call = the K/V cache read once + q read + out and
    lse written (the key pieces' partial states, a few hundred KB, are the
    implementation's and not counted)."""
    import torch

    import ring_sequence_parallelism_gb300 as ra
    from ring_sequence_parallelism_gb300.inputs import make_workload

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    Lq = args.decode
    q_all, k, v = (x.to("cuda") for x in make_workload(w))
    q = q_all[:, :, :Lq].contiguous()
    att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout, kv_heads=w.kv_heads)
    for _ in range(args.warmup):
        out, lse = att.decode(q, k, v)
    att.check()
    stream = torch.cuda.current_stream()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            att.decode(q, k, v, out, lse)
        e1.record(stream)
        torch.cuda.synchronize()
    att.check()
    ms = e0.elapsed_time(e1) / args.steps
    BH = w.B * w.H
    pairs = sum(min(w.N, w.N - Lq + i + 1) for i in range(Lq)) if w.causal else Lq * w.N
    flops = 4 * w.d * BH * pairs
    bytes_ = 2 * w.B * w.kv_heads * w.N * w.d * 2 + BH * Lq * w.d * 2 + BH * Lq * (w.d + 1) * 4
    pk, pk_kind = peaks()
    hbm = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    gbs = bytes_ / (ms * 1e-3) / 1e9
    line = {
        "metric": f"split-K/V decode of {Lq} queries over the {w.N}-token cache, causal-adjusted TFLOP/s",
        "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": dict(config_of(w), Lq=Lq),
        "tokens_per_s": w.B * Lq / (ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_kind": f"hbm_gbs ({pk_kind})", "algorithmic_bytes": bytes_,
                     "kernels": "block_partial_kernel (one state per key piece) + merge_shards_kernel"},
        "clocks": clocks.summary(),
        "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)
    att.close()


def run_bwd(args, w):
    """The ring backward (ring_attn_bwd) on the workload: q, k, v, the
    forward's out and lse and a seeded dO resident in HBM; K backward calls
    timed with CUDA events.  The metric counts 10*d FLOPs per allowed pair
    (the five distinct matmuls S, dP, dV, dK, dQ; 2.5x the forward); the
    kernels execute seven (S and dP in both kernels).  The roofline is the
    dK/dV kernel's: 8*d FLOPs per allowed pair of a step (S^T, dP^T, dV, dK)."""
    import torch

    import ring_sequence_parallelism_gb300 as ra
    from ring_sequence_parallelism_gb300.inputs import make_dout, make_workload

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    q, k, v = (x.to("cuda") for x in make_workload(w))
    do = make_dout(w.B, w.H, w.N, w.d, w.seed, device="cuda")
    att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout, kv_heads=w.kv_heads)
    if w.window:
        att.set_option(ra.RING_OPT_WINDOW, w.window)
    if w.doc_len:
        att.set_segments(w.segments())
    out, lse = att.fwd(q, k, v)
    lap = not args.bwd_per_step and w.P > 1
    att.set_option(ra.RING_OPT_BWD_LAP, 0 if args.bwd_per_step else 1)
    shape = (w.B, w.H, w.N, w.d)
    dq = torch.empty(shape, dtype=torch.float32, device="cuda")
    dk, dv = (torch.empty((w.B, att.Hkv, w.N, w.d), dtype=torch.float32, device="cuda") for _ in range(2))
    att.set_option(ra.RING_OPT_TIMING, 1)
    for _ in range(args.warmup):
        att.bwd(q, k, v, out, lse, do, dq, dk, dv)
    att.check()
    stream = torch.cuda.current_stream()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            att.bwd(q, k, v, out, lse, do, dq, dk, dv)
        e1.record(stream)
        torch.cuda.synchronize()
    t = att.bwd_timing()
    att.check()
    ms = e0.elapsed_time(e1) / args.steps
    pairs = [att.step_work(s)[0] for s in range(w.P)]
    BH = w.B * w.H
    flops = 10 * w.d * sum(pairs)
    pk, pk_kind = peaks()
    peak_sus = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    dkdv_ms, dq_ms = sum(t["dkdv_ms"]), sum(t["dq_ms"])
    ach_dkdv = 8 * w.d * sum(pairs) / (dkdv_ms * 1e-3) / 1e12
    ach_dq = 6 * w.d * sum(pairs) / (dq_ms * 1e-3) / 1e12
    line = {
        "metric": "causal-adjusted attention backward TFLOP/s (10*d FLOPs per allowed pair)",
        "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": dict(config_of(w), dout="N(0,1) bf16, seed + 7"),
        "tokens_per_s": w.B * w.N / (ms * 1e-3),
        "schedule": "lap (one launch per kernel)" if lap else "per step",
        "roofline": {"bound": "tensor",
                     "kernel": "bwd_dkdv_kernel<128> " + ("(one launch for the ring)" if lap else
                                                          "(one launch per ring step)"),
                     "achieved": ach_dkdv, "peak": peak_sus, "unit": "TFLOP/s", "frac": ach_dkdv / peak_sus,
                     "peak_kind": f"bf16_tflops_sustained ({pk_kind})",
                     "traffic": traffic_for(f"{w.name}:bwd_dkdv" + (":lap" if lap else ""), BWD_SOURCE),
                     "algorithmic": "8*d FLOPs per allowed pair (S^T, dP^T, dV, dK)"},
        "dq_kernel": {"achieved": ach_dq, "frac": ach_dq / peak_sus,
                      "algorithmic": "6*d FLOPs per allowed pair (S, dP, dQ)"},
        "bwd": {"dkdv_ms": t["dkdv_ms"], "dq_ms": t["dq_ms"], "prep_ms": t["prep_ms"],
                "kernel_ms_total": dkdv_ms + dq_ms + t["prep_ms"]},
        "clocks": clocks.summary(),
        "gpu_launches": args.steps * (1 + (2 if lap else 2 * w.P)),
    }
    print(json.dumps(line), flush=True)
    att.close()


def run_merge(args, w):
    """ring_attn_merge of two fp32 states of one shard of the workload
    (B*H*n rows; 3*(d+2)*4 algorithmic bytes a row: a and b read, a
    written), in place into a, K times.  Each merge is timed alone with
    CUDA events after an L2 flush (L2Flush; the two states, 68 MB each at
    the 128K workload, would otherwise partly stay in L2)."""
    import torch

    import ring_sequence_parallelism_gb300 as ra

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout, kv_heads=w.kv_heads)
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    rows = (w.B, w.H, w.n)

    def state():
        m = torch.randn(rows, device="cuda", generator=g)
        l = torch.rand(rows, device="cuda", generator=g) + 0.5
        o = torch.randn(rows + (w.d,), device="cuda", generator=g)
        return m, l, o

    a, b = state(), state()
    flush = L2Flush()
    for _ in range(args.warmup):
        att.merge(a, b)
    att.check()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device()) as clocks:
        torch.cuda.synchronize()
        for e0, e1 in ev:
            flush()
            e0.record(stream)
            att.merge(a, b)
            e1.record(stream)
        torch.cuda.synchronize()
    att.check()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / args.steps
    n_rows = w.B * w.H * w.n
    bytes_ = n_rows * 3 * (w.d + 2) * 4
    gbs = bytes_ / (ms * 1e-3) / 1e9
    pk, pk_kind = peaks()
    hbm = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    line = {
        "metric": "merge of two fp32 online-softmax states (ring_attn_merge), algorithmic HBM GB/s",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "config": dict(config_of(w), rows=n_rows,
                       l2="L2 flushed before each timed merge (256 MB written, then 256 MB read)"),
        "roofline": {"bound": "hbm", "kernel": "merge_kernel", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "peak_kind": f"hbm_gbs ({pk_kind})", "traffic": None,
                     "algorithmic": "3*(d+2)*4 bytes per row"},
        "clocks": clocks.summary(),
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    att.close()


def main():
    args = parse()
    from ring_sequence_parallelism_gb300.inputs import WORKLOADS

    w = WORKLOADS[args.workload]
    if args.imbalance:
        import torch

        torch.cuda.set_device(dist_env()[2])
        print(json.dumps({"metric": "per-shard causal work and time", "imbalance": measure_imbalance()}), flush=True)
    elif args.merge:
        run_merge(args, w)
    elif args.decode > 0:
        run_decode(args, w)
    elif args.bwd:
        run_bwd(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
