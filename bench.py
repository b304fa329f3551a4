#!/usr/bin/env python
"""Benchmark of the exact sequential fp64 sum on GB300.

One step = one call of the hot path (seqsum_f64) over a 3840x2160 plane of
synthetic fp64 terms (the c3 workload: 64 zero rows, then 2^U * mantissa with
U in [-40, 0], 1% zeros), result bit-checked against the oracle before timing.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is Gterms/s (terms / device time), timed with
CUDA events on the launching stream around each call, the L2 flushed before
every step by writing one 256 MB buffer and then reading another (so the L2
holds clean lines of the second buffer and the timed call writes nothing
back; the plane itself is 66 MB, under the 129 MB L2).  Multi-GPU runs (torchrun) are independent replicas, one per rank:
a single sequential sum has no data-parallel split without an exchange step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "bit-exact sequential fp64 sum: Gterms/s and HBM GB/s vs roofline at 3840x2160"
UNIT = "Gterms/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c3", choices=["c1", "c2", "c3", "c5"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary configs")
    ap.add_argument("--quick", action="store_true", help="few steps, no CPU baseline (profiling runs)")
    ap.add_argument("--height-mult", type=int, default=1,
                    help="plane this many times taller (profiling captures larger than L2)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_traffic(config: str, height_mult: int):
    """DRAM bytes per launch of the kernel from a committed ncu capture
    (profiles/), or None when the kernel's sources changed since it was taken
    or the workload differs."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", f"seqsum_kernel_{config}_traffic.json")) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["kernel_sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["kernel_sources_sha256"] or height_mult != 1:
            return None
        return int(rec["dram_bytes_read_per_launch"]) + int(rec["dram_bytes_write_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def job_rate(ms_local: float, terms_local: int, ws: int, device="cpu"):
    """Whole-job rate of the replicas: the terms of every rank over the
    slowest rank's time per step (the maximum over ranks).  Returns
    (Gterms/s, ms).  With ws > 1 the process group must be initialised."""
    ms, terms = float(ms_local), float(terms_local)
    if ws > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        u = torch.tensor([terms], device=device, dtype=torch.float64)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
        ms, terms = t.item(), u.item()
    return terms / (ms * 1e-3) / 1e9, ms


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(x, s0, budget_s):
    """The oracle as it stands, on one host core, over whole sums of the
    workload until the time budget is used."""
    import oracle
    oracle.lib()
    n = len(x)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.seqsum(x, s0)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    return {"value": reps * n / el / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} whole sums of the {n}-term plane, {el:.1f} s on 1 host core "
                      f"(the sequential loop cannot use more cores without changing its bits)"}


def cpu_batched_all_cores(x, offsets, s0s, reps=3):
    """The oracle's loop for every sum of a batched workload, the sums spread
    over all host cores (one sum per thread, largest first; each sum is still
    one sequential loop, so its bits do not change).  Returns the baseline
    record and the sums of the last pass."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.lib()
    n = len(offsets) - 1
    order = sorted(range(n), key=lambda k: -(int(offsets[k + 1]) - int(offsets[k])))
    cores = os.cpu_count() or 1
    outs = np.empty(n)

    def one(k):
        outs[k] = oracle.seqsum(x[int(offsets[k]):int(offsets[k + 1])], float(s0s[k]))

    times = []
    with ThreadPoolExecutor(cores) as ex:
        for _ in range(reps):
            t0 = time.perf_counter()
            list(ex.map(one, order))
            times.append(time.perf_counter() - t0)
    best = min(times)
    return {"value": len(x) / best / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"all {n} sums ({len(x)} terms), best of {reps} passes, one sum per thread "
                      f"on {cores} host threads"}, outs


def reference_arm(args, ws, rank):
    """The oracle as the reference arm: same metric, config and unit."""
    if rank != 0:
        return
    import workloads as W
    wl = W.config(args.config)
    x, s0 = wl.x, float(wl.s0[0])
    import oracle
    oracle.lib()
    for _ in range(max(args.warmup, 1)):
        oracle.seqsum(x, s0)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.seqsum(x, s0)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = len(x) / (ms * 1e-3) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.config} 3840x2160 single sum ({len(x)} terms)",
                       "n_terms": len(x), "l2": "n/a (host)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} whole sums of the {len(x)}-term plane"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class Flush:
    """Leaves the L2 holding clean lines that the timed call does not use: a
    256 MB write, then a read of another 256 MB buffer (twice the 129 MB L2)."""

    def __init__(self, torch, dev):
        self.a = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.b = torch.ones(32 << 20, dtype=torch.int64, device=dev)

    def __call__(self):
        self.a.fill_(1)
        self.b.sum()


def time_kernel(sq, torch, xd, s0, out, steps, warmup, flush, stream):
    """Per-step CUDA events on the launching stream around one call; the L2
    is flushed before each step, outside the events."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            sq.seqsum_f64(xd, s0, out=out, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush()
            a.record(stream)
            sq.seqsum_f64(xd, s0, out=out, stream=stream)
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def main():
    args = parse()
    ws, rank, local = dist_init()
    if args.impl == "reference":
        reference_arm(args, ws, rank)
        return
    import torch
    import parity_binade_chunked_gb300 as sq
    import workloads as W
    import oracle

    if args.quick:
        args.steps = min(args.steps, 20)
        args.warmup = min(args.warmup, 3)
    args.warmup = max(args.warmup, 3)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    wl = W.config(args.config, height_mult=args.height_mult)
    x = wl.x
    n = len(x)
    s0 = float(wl.s0[0])
    xd = torch.from_numpy(x).to(dev)
    out = torch.empty(1, dtype=torch.float64, device=dev)
    flush = Flush(torch, dev)

    # parity before timing (0 ULP)
    want = oracle.seqsum(x, s0)
    sq.seqsum_f64(xd, s0, out=out, stream=stream)
    stream.synchronize()
    got = out.item()
    parity = bool(np.float64(got).view(np.uint64) == np.float64(want).view(np.uint64))
    sq.get_stats()

    # ---- the timed region (device time per step)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        times = time_kernel(sq, torch, xd, s0, out, args.steps, args.warmup, flush, stream)
        t_wall = time.perf_counter() - t_wall0
    torch.cuda.synchronize()
    stats = sq.get_stats()
    value, ms = job_rate(sum(times) / len(times), n, ws, dev)
    peak, peak_src = peaks()
    achieved = 8.0 * n / (ms * 1e-3) / 1e9          # GB/s, algorithmic bytes (8 per term read once)

    # ---- end to end through the C ABI with host buffers
    e2e_steps = max(5, min(50, args.steps))
    hx = torch.from_numpy(x).pin_memory()
    hout = torch.empty(1, dtype=torch.float64).pin_memory()
    xe = torch.empty(n, dtype=torch.float64, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            xe.copy_(hx, non_blocking=True)
            sq.seqsum_f64(xe, s0, out=out, stream=stream)
            hout.copy_(out, non_blocking=True)
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            xe.copy_(hx, non_blocking=True)
            sq.seqsum_f64(xe, s0, out=out, stream=stream)
            hout.copy_(out, non_blocking=True)
        b.record(stream)
    stream.synchronize()
    e2e_ms = a.elapsed_time(b) / e2e_steps
    e2e_ok = bool(np.float64(hout.item()).view(np.uint64) == np.float64(want).view(np.uint64))

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.config} {wl.shape[0][0]}x{wl.shape[0][1]} single sum ({n} terms)", "n_terms": n,
                   "recipe": wl.recipe, "l2": "flushed before every step (256 MB write, then a 256 MB read of another buffer)",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "parity_0ulp": parity and e2e_ok,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": measured_traffic(args.config, args.height_mult),
                     "peak_source": peak_src, "algorithmic_bytes_per_launch": 8 * n,
                     "traffic_source": "profiles/seqsum_kernel_%s_traffic.json (null if the kernel changed)" % args.config},
        "e2e": {"value": n / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": 8 * n,
                "d2h_bytes_per_step": 8},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "kernel_ms": {"median": statistics.median(times), "min": min(times), "max": max(times)},
        # counters and ns_* (summed over CTAs) per call; t_* are the last call's own
        "device_stats_per_call": {k: (v if k.startswith("t_") else v / (args.steps + args.warmup))
                                  for k, v in stats.items()
                                  if k not in ("device_status", "device_error_bits", "check_site", "check_pad",
                                               "check_value")},
        "device_status": stats["device_status"],
        "wall_s": t_wall,
    }

    # ---- secondary configs (same timing method), context only
    if not args.no_extra and not args.quick and rank == 0:
        extra = {}
        for name in ["c5", "c1", "c2"]:
            if name == args.config:
                continue
            w2 = W.config(name)
            x2 = torch.from_numpy(w2.x).to(dev)
            o2 = torch.empty(1, dtype=torch.float64, device=dev)
            t2 = time_kernel(sq, torch, x2, float(w2.s0[0]), o2, 200, 5, flush, stream)
            ok = np.float64(o2.item()).view(np.uint64) == np.float64(oracle.seqsum(w2.x, float(w2.s0[0]))).view(
                np.uint64)
            m2 = sum(t2) / len(t2)
            extra[name] = {"n_terms": len(w2.x), "ms_per_step": m2, "Gterms/s": len(w2.x) / (m2 * 1e-3) / 1e9,
                           "frac_hbm": 8 * len(w2.x) / (m2 * 1e-3) / 1e9 / peak, "parity_0ulp": bool(ok)}
        # c4: the 108-sum pyramid, batched
        w4 = W.config("c4")
        x4 = torch.from_numpy(w4.x).to(dev)
        o4 = torch.from_numpy(w4.offsets).to(dev)
        s4 = torch.from_numpy(w4.s0).to(dev)
        outs = sq.seqsum_f64_batched_sized(x4, o4, s4, stream=stream)
        stream.synchronize()
        ok4 = np.array_equal(outs.cpu().numpy().view(np.uint64),
                             oracle.seqsum_batched(w4.x, w4.offsets, w4.s0).view(np.uint64))
        ts = []
        for i in range(30):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                flush()   # (on the timed stream: it must not overlap the call)
                a.record(stream)
                sq.seqsum_f64_batched_sized(x4, o4, s4, outs=outs, stream=stream)
                b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        t4 = [a.elapsed_time(b) for a, b in ts[3:]]
        m4 = sum(t4) / len(t4)
        extra["c4"] = {"n_terms": len(w4.x), "nsums": w4.nsums, "ms_per_step": m4,
                       "Gterms/s": len(w4.x) / (m4 * 1e-3) / 1e9,
                       "frac_hbm": 8 * len(w4.x) / (m4 * 1e-3) / 1e9 / peak, "parity_0ulp": bool(ok4)}
        if not args.quick:
            cpu4, cpu_outs = cpu_batched_all_cores(w4.x, w4.offsets, w4.s0)
            cpu4["bits_match_oracle"] = bool(np.array_equal(
                cpu_outs.view(np.uint64), oracle.seqsum_batched(w4.x, w4.offsets, w4.s0).view(np.uint64)))
            extra["c4"]["cpu_baseline_all_cores"] = cpu4
        # the lcs variant: four interleaved sums per 1920x1080 window plane, with their float means
        nl = 1920 * 1080
        xl = np.empty(4 * nl)
        xl[0::4] = W.plane_c2(1920, 1080, seed=41)
        xl[1::4] = W.plane_pow2(nl, 42, -30, 2, stream=5)
        xl[2::4] = W.plane_pow2(nl, 43, -20, 0, stream=5)
        xl[3::4] = -W.plane_pow2(nl, 44, -40, 0, stream=5)
        s0l = np.array([0.0, 1.0, 0.0, -0.5])
        xld, s0ld = torch.from_numpy(xl).to(dev), torch.from_numpy(s0l).to(dev)
        outl = torch.empty(4, dtype=torch.float64, device=dev)
        meanl = torch.empty(4, dtype=torch.float32, device=dev)
        sq.seqsum_f64_strided(xld, 4, s0ld, outs=outl, means=meanl, stream=stream)
        stream.synchronize()
        wl_sums, wl_means = oracle.seqsum_strided(xl, 4, s0l)
        okl = (np.array_equal(outl.cpu().numpy().view(np.uint64), wl_sums.view(np.uint64)) and
               np.array_equal(meanl.cpu().numpy().view(np.uint32), wl_means.view(np.uint32)))
        ts = []
        for i in range(30):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                flush()   # (on the timed stream: it must not overlap the call)
                a.record(stream)
                sq.seqsum_f64_strided(xld, 4, s0ld, outs=outl, means=meanl, stream=stream)
                b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        tl = [a.elapsed_time(b) for a, b in ts[3:]]
        ml = sum(tl) / len(tl)
        extra["lcs_4x1920x1080"] = {"n_terms": len(xl), "nsums": 4, "ms_per_step": ml,
                                    "Gterms/s": len(xl) / (ml * 1e-3) / 1e9,
                                    "frac_hbm": 8 * len(xl) / (ml * 1e-3) / 1e9 / peak,
                                    "parity_0ulp": bool(okl),
                                    "note": "interleaved plane copied apart, then summed batched; float means"}
        # plan reuse: a sequence of frames close to one another (the workload's
        # plane, each term scaled by its own factor in [1 - 2^-7, 1 + 2^-7]),
        # one plan kept from frame to frame
        u = [W.uniform53(W.draws_u64(100 + k, 7, n)) for k in range(4)]
        frames = [x * (1.0 + 2.0 ** -7 * (2.0 * uk - 1.0)) for uk in u]
        fd = [torch.from_numpy(f).to(dev) for f in frames]
        outs_p = torch.empty(4, dtype=torch.float64, device=dev)
        plan = sq.SeqsumPlan()
        with torch.cuda.stream(stream):
            for k in range(4):
                plan(fd[k], s0, out=outs_p[k:k + 1], stream=stream)
        stream.synchronize()
        sq.get_stats()
        ts = []
        for i in range(40):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                flush()
                a.record(stream)
                plan(fd[i % 4], s0, out=outs_p[i % 4:i % 4 + 1], stream=stream)
                b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        stp = sq.get_stats()
        okp = all(np.float64(outs_p[k].item()).view(np.uint64) == np.float64(oracle.seqsum(frames[k], s0)).view(np.uint64)
                  for k in range(4))
        plan.close()
        tp = [a.elapsed_time(b) for a, b in ts[4:]]
        mp = sum(tp) / len(tp)
        extra["planned_frames"] = {"workload": args.config, "n_terms": n, "ms_per_step": mp,
                                   "Gterms/s": n / (mp * 1e-3) / 1e9,
                                   "frac_hbm": 8 * n / (mp * 1e-3) / 1e9 / peak, "parity_0ulp": bool(okp),
                                   "tiles_redone_per_call": stp["tiles_redone"] / 40.0,
                                   "note": "seqsum_f64_planned over 4 frames in turn, the plan of each call "
                                           "from the call before"}
        line["other_configs"] = extra

    if rank == 0:
        if not args.quick:
            line["cpu_baseline"] = cpu_baseline(x, s0, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
