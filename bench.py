"""Benchmark of exact row-wise FP32 Top-K on GB300.

Metric: rows/s and score-row HBM GB/s (fraction of the measured GB300 HBM
peak) per workload, 1 GPU.  The headline line is the largest workload, the
causal prefill batch (M=4096, N=131072, ke[r] = N - M + r + 1, K=2048,
indexer-like scores with a positional trend); "per_config" repeats the
measurement, with its own end-to-end and CPU-oracle numbers, for all five
workloads.

A step is one exact Top-K call (one kernel launch) over one batch whose
inputs are already resident in HBM.  Inputs smaller than L2 are rotated over
copies whose total footprint is at least 4x the L2 size, so every call reads
its scores from HBM.  Calls are captured in CUDA graphs and timed with CUDA
events on the launching stream.

Algorithmic bytes per call: sum_r clamp(ke[r], 0, N) * 4 (valid scores read
once) + M * K * 4 (indices written).  Sampling, band and recovery rereads,
frontier gathers and padding are not credited.

``--impl reference`` times the CPU oracle (per-row std::nth_element, all host
cores) on the same workload instead: the pages' own kernels are Hopper code
that is not available here.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "prefill_causal"
MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_SOURCE = os.path.join(ROOT, "exact_top_selection_gb300", "csrc", "topk_kernels.cu")
KERNEL_NAMES = {1: "persistent_sampled_kernel", 2: "kv_split_kernel", 3: "row_local_exact_kernel",
                4: "cluster_split_kernel"}


# ---------------------------------------------------------------- distributed helpers


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def aggregate_over_ranks(elapsed_s: float, rows: int, group=None):
    """Whole-job numbers: the slowest rank's time and the rows of all ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return elapsed_s, rows
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    n = torch.tensor([rows], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), int(n.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- peaks, profiles, clocks


def hbm_peak():
    try:
        with open(MEASURED_PEAKS) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


def kernel_source_hash():
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, or None if there is
    none or the kernel source changed since it was taken."""
    path = os.path.join(PROFILES, f"{kernel}__{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU is under load."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 100):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.interval}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        rows = [p for (t, p) in self.samples if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        if not rows:
            rows = [p for (_, p) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = sorted(v for v in (num(p[1]) for p in rows) if v is not None)
        smax = max((v for v in (num(p[2]) for p in rows) if v is not None), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in rows for i in range(4) if p[5 + i] == "Active"})
        power = [v for v in (num(p[3]) for p in rows) if v is not None]
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- workload setup


def algorithmic_bytes(ke, N, M, K):
    import torch
    L = ke.to(torch.int64).clamp(0, N)
    return int(L.sum().item()) * 4 + M * K * 4


class Case:
    """One workload resident on the device, rotated over enough copies to
    defeat L2, with its runner (plan + counters + workspace)."""

    def __init__(self, name, device, seed_offset=0, min_footprint_factor=4.0, rows=None):
        import torch

        import exact_top_selection_gb300 as etk
        import workloads

        self.name = name
        self.w = workloads.WORKLOADS[name]
        self.device = device
        X, ke, K = workloads.generate(name, M=rows, device=str(device),
                                      seed=self.w.seed + seed_offset)
        self.M, self.N = X.shape
        self.K = K
        self.ke = ke.to(device)
        self.alg_bytes = algorithmic_bytes(self.ke, self.N, self.M, K)
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        per = X.numel() * 4
        self.copies = max(1, math.ceil(min_footprint_factor * l2 / per)) if per < 2 * l2 else 1
        self.X = [X] + [X.clone() for _ in range(self.copies - 1)]
        self.runner = etk.ExactTopK(self.M, self.N, K, device=device)
        self.plan = self.runner.plan
        self.outs = [torch.empty(self.M, K, dtype=torch.int32, device=device)
                     for _ in range(min(self.copies, 4))]
        self.nv = torch.tensor([self.M], dtype=torch.int32, device=device)
        self.l2_bytes = l2
        # inputs are made on the default stream; calls run on other streams
        torch.cuda.synchronize(device)

    def call(self, i, stream=None):
        return self.runner(self.X[i % self.copies], self.ke, num_valid_rows=self.nv,
                           out=self.outs[i % len(self.outs)], stream=stream)

    def graph(self, n_calls, stream, start=0):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            self.call(start, stream)  # first call on a device happens before capture
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for k in range(n_calls):
                    self.call(start + k, stream)
        return g

    def l2_note(self):
        if self.copies > 1:
            return (f"inputs rotated over {self.copies} copies "
                    f"({self.copies * self.X[0].numel() * 4 / self.l2_bytes:.1f}x L2)")
        return "input larger than L2 (no rotation needed)"

    def route_rates(self):
        import torch

        import exact_top_selection_gb300 as etk
        tr = torch.full((self.M, 8), -9, dtype=torch.int32, device=self.device)
        self.runner(self.X[0], self.ke, num_valid_rows=self.nv, out=self.outs[0], trace=tr)
        torch.cuda.synchronize(self.device)
        routes = tr[:, 0].cpu().tolist()
        counts = {}
        for r in routes:
            counts[etk.ROUTES[r] if 0 <= r < len(etk.ROUTES) else str(r)] = \
                counts.get(etk.ROUTES[r] if 0 <= r < len(etk.ROUTES) else str(r), 0) + 1
        long_rows = sum(v for k, v in counts.items() if k != "pad")
        band = counts.get("band", 0) + counts.get("exact_after_band", 0)
        exact = sum(counts.get(k, 0) for k in ("exact_after_band", "exact_no_band",
                                               "direct_exact", "guess_exact"))
        return {"counts": counts,
                "p_band": band / long_rows if long_rows else 0.0,
                "p_exact": exact / long_rows if long_rows else 0.0}


def time_schedule(case, steps, warmup, stream, max_nodes=512):
    """Runs `warmup` untimed calls, then times exactly `steps` calls (CUDA graph
    replays on `stream`, CUDA events on the same stream).  Returns seconds."""
    import torch
    G = max(1, min(max_nodes, steps, max(case.copies, 64)))
    full = case.graph(G, stream)
    rem = steps % G
    tail = case.graph(rem, stream) if rem else None
    with torch.cuda.stream(stream):
        for i in range(warmup):
            case.call(i, stream)
    torch.cuda.synchronize(case.device)
    barrier()
    torch.cuda.synchronize(case.device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // G):
            full.replay()
        if tail is not None:
            tail.replay()
        e1.record(stream)
    torch.cuda.synchronize(case.device)
    barrier()
    torch.cuda.synchronize(case.device)
    return e0.elapsed_time(e1) / 1e3


def median_per_call(case, stream, rounds=7, calls_per_round=None):
    """Paper-style protocol: conditioning sweeps, then rounds of graph replays;
    median over rounds of the mean per-call time (seconds)."""
    import torch
    n = calls_per_round or max(100, case.copies)
    n = min(n, 1024)
    g = case.graph(n, stream)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(case.device)
    times = []
    for _ in range(rounds):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize(case.device)
        times.append(e0.elapsed_time(e1) / 1e3 / n)
    times.sort()
    return times[len(times) // 2]


def keep_busy(case, stream, seconds):
    """Untimed replays so that clock samples exist for short timed regions."""
    import torch
    g = case.graph(min(256, max(case.copies, 16)), stream)
    t_end = time.time() + seconds
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize(case.device)


def guess_series_measure(device, stream, steps=16, M=64, N=65536, K=2048, seed=20260006,
                         rounds=5):
    """A decode batch followed over `steps` correlated steps (the optional guess
    source): step t passes step t-1's output as prev_topk.  The same series is
    timed with the guess and without it (sampled view), as CUDA-graph replays
    of the whole chain over inputs larger than L2."""
    import torch

    import exact_top_selection_gb300 as etk
    import workloads
    Xs, kes = workloads.decode_batch_series(M, N, K, steps, seed, device=str(device))
    runner = etk.ExactTopK(M, N, K, device=device)
    torch.cuda.synchronize(device)  # inputs come from the default stream
    outs = [torch.empty(M, K, dtype=torch.int32, device=device) for _ in range(steps)]
    traces = [torch.full((M, 8), -9, dtype=torch.int32, device=device) for _ in range(steps)]

    def chain(use_guess, with_trace=False):
        for t in range(steps):
            prev = outs[t - 1] if (use_guess and t) else None
            runner(Xs[t], kes[t], out=outs[t], prev_topk=prev,
                   trace=traces[t] if with_trace else None, stream=stream)

    result = {"steps": steps, "M": M, "N": N, "K": K, "drift": 0.05,
              "footprint_bytes": steps * M * N * 4}
    for use_guess in (True, False):
        with torch.cuda.stream(stream):
            chain(use_guess, with_trace=True)
        torch.cuda.synchronize(device)
        routes = torch.cat([tr[1:, 0] if use_guess else tr[:, 0] for tr in traces]).cpu().tolist()
        counts = {}
        for rt in routes:
            nm = etk.ROUTES[rt] if 0 <= rt < len(etk.ROUTES) else str(rt)
            counts[nm] = counts.get(nm, 0) + 1
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            chain(use_guess)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                chain(use_guess)
        g.replay()
        torch.cuda.synchronize(device)
        times = []
        for _ in range(rounds):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize(device)
            times.append(e0.elapsed_time(e1) / 1e3 / steps)
        times.sort()
        key = "guess" if use_guess else "sampled"
        result[f"us_per_call_{key}"] = times[len(times) // 2] * 1e6
        result[f"routes_{key}"] = counts
    del Xs, kes
    return result


def _time_calls(runner, Xs, ke, stream, calls=64, rounds=5, trace=None):
    """Median per-call seconds of graph replays cycling over the inputs Xs."""
    import torch
    out = torch.empty(runner.plan.num_rows, runner.plan.top_k, dtype=torch.int32,
                      device=Xs[0].device)
    if trace is not None:
        with torch.cuda.stream(stream):
            runner(Xs[0], ke, out=out, trace=trace, stream=stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        runner(Xs[0], ke, out=out, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for c in range(calls):
                runner(Xs[c % len(Xs)], ke, out=out, stream=stream)
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(rounds):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3 / calls)
    times.sort()
    return times[len(times) // 2]


def _route_stats(trace, K):
    import exact_top_selection_gb300 as etk
    tr = trace.cpu().numpy()
    routes = tr[:, 0]
    live = routes != 0
    n = max(1, int(live.sum()))
    counts = {}
    for rt in routes.tolist():
        nm = etk.ROUTES[rt] if 0 <= rt < len(etk.ROUTES) else str(rt)
        counts[nm] = counts.get(nm, 0) + 1
    band = sum(counts.get(k, 0) for k in ("band", "exact_after_band"))
    exact = sum(counts.get(k, 0) for k in ("exact_after_band", "exact_no_band", "direct_exact"))
    c0 = tr[live & (tr[:, 3] >= 0), 3]
    return {"routes": counts, "p_band": band / n, "p_exact": exact / n,
            "mean_c0_over_K": float(c0.mean()) / K if c0.size else None}


def run_sweep(args):
    """Planner studies on one GPU: one JSON line per point.  crossover: row
    width N against the row-local exact kernel and the two sampled policies;
    margins: retention margin rho and view stride s on prefill-shaped rows,
    with route rates; splits: KV-split segment count P on the few-long-rows
    workload; trace: a serving-style sequence of calls with N growing and
    M = 2^24 / N, each planned by the default planner, timed call by call and
    as one captured sequence; floor: per workload, a read-only kernel over the
    valid prefixes beside the selection, in the same replay harness."""
    import math

    import torch

    import exact_top_selection_gb300 as etk
    import workloads
    device = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size

    def copies_for(X):
        per = X.numel() * 4
        c = max(1, math.ceil(4 * l2 / per)) if per < 2 * l2 else 1
        out = [X] + [X.clone() for _ in range(c - 1)]
        torch.cuda.synchronize(device)  # made on the default stream, read on `stream`
        return out

    def emit(d):
        print(json.dumps(d), flush=True)

    K = 2048
    if args.sweep == "crossover":
        M = 1024
        for N in (8192, 12288, 16384, 24576, 32768, 49152, 65536, 98304, 131072):
            # full-length indexer-like rows (no padding inside the prefix)
            X = workloads.indexer_scores(M, N, workloads._gen(str(device), 20260010 + N),
                                         str(device))
            ke = torch.full((M,), N, dtype=torch.int32, device=device)
            Xs = copies_for(X)
            for name, kw in (("row_local_exact", dict(family=etk.FAMILY_ROW_LOCAL_EXACT)),
                             ("persistent_s64_primary", dict(family=etk.FAMILY_PERSISTENT_SAMPLED,
                                                             stride=64, dual=0)),
                             ("persistent_s128_dual", dict(family=etk.FAMILY_PERSISTENT_SAMPLED,
                                                           stride=128, dual=1))):
                runner = etk.ExactTopK(M, N, K, device=device, **kw)
                tr = torch.full((M, 8), -9, dtype=torch.int32, device=device)
                sec = _time_calls(runner, Xs, ke, stream, trace=tr)
                emit({"sweep": "crossover", "M": M, "N": N, "K": K, "policy": name,
                      "us_per_call": sec * 1e6, "gbs": (M * N * 4 + M * K * 4) / sec / 1e9,
                      **_route_stats(tr, K)})
            del X, Xs
            torch.cuda.empty_cache()
    elif args.sweep == "margins":
        M, N = 1024, 131072
        X, ke, _ = workloads.generate("prefill_causal", M=M, N=N, K=K, device=str(device))
        Xs = [X]
        torch.cuda.synchronize(device)
        alg = int(ke.to(torch.int64).clamp(0, N).sum().item()) * 4 + M * K * 4
        for s in (64, 128, 256):
            for rho in ((5, 4), (3, 2), (2, 1)):
                rho1 = (rho[0] * 4 + rho[1], rho[1] * 4)  # rho + 1/4
                runner = etk.ExactTopK(M, N, K, device=device,
                                       family=etk.FAMILY_PERSISTENT_SAMPLED, stride=s, dual=1,
                                       rho0=rho, rho1=rho1)
                tr = torch.full((M, 8), -9, dtype=torch.int32, device=device)
                sec = _time_calls(runner, Xs, ke, stream, trace=tr)
                emit({"sweep": "margins", "M": M, "N": N, "K": K, "stride": s,
                      "rho0": rho[0] / rho[1], "rho1": rho1[0] / rho1[1],
                      "us_per_call": sec * 1e6, "gbs": alg / sec / 1e9, **_route_stats(tr, K)})
    elif args.sweep == "trace":
        calls = workloads.trace_sequence(1 << 24, K, 20260020, device=str(device))
        torch.cuda.synchronize(device)
        runners, outs, total_rows, total_alg = [], [], 0, 0
        for i, (X, ke) in enumerate(calls):
            M, N = X.shape
            runner = etk.ExactTopK(M, N, K, device=device)
            tr = torch.full((M, 8), -9, dtype=torch.int32, device=device)
            sec = _time_calls(runner, copies_for(X), ke, stream, trace=tr)
            alg = int(ke.to(torch.int64).clamp(0, N).sum().item()) * 4 + M * K * 4
            total_rows += M
            total_alg += alg
            runners.append(runner)
            outs.append(torch.empty(M, K, dtype=torch.int32, device=device))
            emit({"sweep": "trace", "call": i, "M": M, "N": N, "K": K,
                  "family": etk.FAMILY_NAMES[runner.plan.family], "splits": runner.plan.splits,
                  "us_per_call": sec * 1e6, "gbs": alg / sec / 1e9, **_route_stats(tr, K)})
        # the whole sequence as one graph, replayed
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for (X, ke), runner, out in zip(calls, runners, outs):
                runner(X, ke, out=out, stream=stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for (X, ke), runner, out in zip(calls, runners, outs):
                    runner(X, ke, out=out, stream=stream)
        g.replay()
        torch.cuda.synchronize(device)
        times = []
        for _ in range(7):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize(device)
            times.append(e0.elapsed_time(e1) / 1e3)
        sec = sorted(times)[len(times) // 2]
        emit({"sweep": "trace_sequence", "calls": len(calls), "rows": total_rows,
              "us_per_sequence": sec * 1e6, "rows_per_s": total_rows / sec,
              "gbs": total_alg / sec / 1e9})
    elif args.sweep == "floor":
        # The attainable streaming time of each workload: a read-only kernel
        # over exactly the valid prefixes, in the selection plan's split
        # count (one segment per row for the single-CTA families), timed
        # like the selection itself over the same rotated input copies.
        import workloads as wl
        peak, _ = hbm_peak()
        for name in wl.ORDER:
            c = Case(name, device)
            sec_sel = median_per_call(c, stream)
            splits = c.plan.splits if c.plan.family in (2, 4) else 1
            outs = torch.empty(c.M, splits, dtype=torch.int32, device=device)
            n = min(1024, max(100, c.copies))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                etk.stream_floor(c.X[0], c.ke, splits, out=outs, stream=stream)
                stream.synchronize()
                with torch.cuda.graph(g, stream=stream):
                    for k in range(n):
                        etk.stream_floor(c.X[k % c.copies], c.ke, splits, out=outs, stream=stream)
            for _ in range(2):
                g.replay()
            torch.cuda.synchronize(device)
            times = []
            for _ in range(7):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                torch.cuda.synchronize(device)
                times.append(e0.elapsed_time(e1) / 1e3 / n)
            sec_floor = sorted(times)[len(times) // 2]
            score_bytes = c.alg_bytes - c.M * c.K * 4
            emit({"sweep": "floor", "workload": name, "M": c.M, "N": c.N, "splits": splits,
                  "family": KERNEL_NAMES[c.plan.family], "floor_us": sec_floor * 1e6,
                  "floor_frac": score_bytes / sec_floor / 1e9 / peak,
                  "selection_us": sec_sel * 1e6,
                  "selection_frac": c.alg_bytes / sec_sel / 1e9 / peak,
                  "selection_over_floor": sec_sel / sec_floor})
            del c, outs, g
            torch.cuda.empty_cache()
    elif args.sweep == "splits":
        X, ke, _ = workloads.generate("long_decode", device=str(device))
        M, N = X.shape
        Xs = copies_for(X)
        alg = int(ke.to(torch.int64).clamp(0, N).sum().item()) * 4 + M * K * 4
        for P in (8, 16, 32, 64):
            runner = etk.ExactTopK(M, N, K, device=device, family=etk.FAMILY_KV_SPLIT, splits=P)
            tr = torch.full((M, 8), -9, dtype=torch.int32, device=device)
            sec = _time_calls(runner, Xs, ke, stream, trace=tr)
            emit({"sweep": "splits", "M": M, "N": N, "K": K, "splits": P,
                  "us_per_call": sec * 1e6, "gbs": alg / sec / 1e9, **_route_stats(tr, K)})


def e2e_chunks(M, score_bytes):
    """Row chunks of the end-to-end pipeline: one below 256 MB of scores,
    where a chunk's host calls (copies, event, launch) would cost more than
    the selection they hide; else the largest of 8, 4, 2 that divides M (rows
    are independent, so chunks select separately)."""
    if score_bytes < (256 << 20):
        return 1
    for c in (8, 4, 2):
        if M % c == 0 and M >= c:
            return c
    return 1


def e2e_measure(case, steps, warmup, stream):
    """Same metric through the public API with host buffers: per step, H2D of
    the score matrix, lengths and live counts from pinned memory, the call,
    and D2H of the indices, all inside the timed region.  Large batches go in
    row chunks: a copy stream moves chunk i + 1 while the launching stream
    selects chunk i (one exact_topk_run per chunk, each with its own plan,
    counters and workspace) and returns its indices, so the selection hides
    behind the host link.  One chunk runs everything on the launching stream."""
    import torch

    import exact_top_selection_gb300 as etk
    C = e2e_chunks(case.M, case.X[0].numel() * 4)
    mc = case.M // C
    Xh = case.X[0].cpu().pin_memory()
    keh = case.ke.cpu().pin_memory()
    nvh = torch.full((C,), mc, dtype=torch.int32).pin_memory()
    outh = torch.empty(case.M, case.K, dtype=torch.int32).pin_memory()
    Xd = torch.empty_like(case.X[0])
    ked = torch.empty_like(case.ke)
    nvd = torch.empty(C, dtype=torch.int32, device=case.device)
    outd = torch.empty(case.M, case.K, dtype=torch.int32, device=case.device)
    runners = [case.runner] if C == 1 else \
        [etk.ExactTopK(mc, case.N, case.K, device=case.device) for _ in range(C)]
    copy = torch.cuda.Stream(case.device)
    landed = [torch.cuda.Event() for _ in range(C)]

    def step():
        if C == 1:
            Xd.copy_(Xh, non_blocking=True)
            ked.copy_(keh, non_blocking=True)
            nvd.copy_(nvh, non_blocking=True)
            case.runner(Xd, ked, num_valid_rows=nvd, out=outd, stream=stream)
            outh.copy_(outd, non_blocking=True)
            return
        copy.wait_stream(stream)  # the previous step's reads of the device buffers are done
        for c in range(C):
            rows = slice(c * mc, (c + 1) * mc)
            with torch.cuda.stream(copy):
                Xd[rows].copy_(Xh[rows], non_blocking=True)
                ked[rows].copy_(keh[rows], non_blocking=True)
                nvd[c:c + 1].copy_(nvh[c:c + 1], non_blocking=True)
                landed[c].record(copy)
            stream.wait_event(landed[c])
            runners[c](Xd[rows], ked[rows], num_valid_rows=nvd[c:c + 1], out=outd[rows],
                       stream=stream)
            with torch.cuda.stream(stream):
                outh[rows].copy_(outd[rows], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            step()
        torch.cuda.synchronize(case.device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize(case.device)
    dt = e0.elapsed_time(e1) / 1e3
    h2d = Xh.numel() * 4 + keh.numel() * 4 + nvh.numel() * 4
    d2h = outh.numel() * 4
    return dt, h2d, d2h, C


def cpu_baseline(case, seconds=10.0, rows_cap=None):
    """The oracle as it stands, on all host cores, over a bounded sample: the
    first `rows_cap` rows of the case's own (device-resident) matrix, copied
    to the host, selected again and again until `seconds` have passed."""
    import numpy as np

    import oracle
    M = case.M if rows_cap is None else max(1, min(rows_cap, case.M))
    X = case.X[0][:M].cpu().numpy()
    ke = case.ke[:M].cpu().numpy()
    K = case.K
    threads = oracle.hardware_threads()
    rows = 0
    t0 = time.perf_counter()
    while True:
        oracle.topk_rows(X, ke, K, nthreads=threads)
        rows += M
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    bytes_ = int(np.clip(ke.astype(np.int64), 0, X.shape[1]).sum()) * 4 + M * K * 4
    return {"value": rows / dt, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "gbs": bytes_ * (rows / M) / dt / 1e9,
            "sample": f"{case.name}: rows 0..{M - 1} of {case.M}, {rows // M} passes "
                      f"in {dt:.1f} s (std::nth_element per row, {threads} threads)"}


# rows of each workload the per-config CPU baseline selects per pass
CPU_SAMPLE_ROWS = {"short_iid": 4, "decode_batch": 64, "prefill_causal": 256, "long_decode": 8,
                   "adversarial": 256}


# ---------------------------------------------------------------- arms


def _e2e_entry(case, steps, warmup, stream):
    dt, h2d, d2h, chunks = e2e_measure(case, steps, warmup, stream)
    e_dt, e_rows = aggregate_over_ranks(dt, case.M * steps)
    return {"value": e_rows / e_dt, "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt / steps * 1e3,
            "path": "pinned host -> H2D -> exact_topk_run (C ABI) -> D2H, per step" + (
                f", in {chunks} row chunks pipelined over a copy stream and the launching stream"
                if chunks > 1 else "")}


def init_ranks(args):
    """Process group of a replica run (one process per GPU, rows split by
    rank, no collective on the data path; the group only carries the
    whole-job time and row totals).  Returns (rank, local_rank, world)."""
    rank, local_rank, world = dist_env()
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} disagrees with WORLD_SIZE={world}")
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (torch.cuda.is_available() and not args.stub) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    return rank, local_rank, world


def finish_ranks(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_stub(args):
    """The launcher and the whole-job aggregation without a GPU: every rank
    'times' a fixed sleep over a fixed row count.  Used by the CPU tests of
    the replica launcher; its line says "stub" and is not a measurement."""
    rank, _, world = init_ranks(args)
    rows = 64
    barrier()
    t0 = time.perf_counter()
    time.sleep(0.02 * (rank + 1))
    elapsed = time.perf_counter() - t0
    barrier()
    e_max, rows_total = aggregate_over_ranks(elapsed, rows * args.steps)
    if rank == 0:
        print(json.dumps({"stub": True, "metric": "rows/s (launcher test, no GPU)",
                          "value": rows_total / e_max, "unit": "rows/s", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": e_max / args.steps * 1e3, "higher_is_better": True,
                          "scaling": "weak", "rows_total": rows_total,
                          "max_rank_seconds": e_max}), flush=True)
    finish_ranks(world)


def run_ours(args):
    import torch

    rank, local_rank, world = init_ranks(args)
    device = torch.device("cuda", local_rank if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    peak, peak_src = hbm_peak()

    case = Case(args.workload, device, seed_offset=rank, rows=args.rows)
    sampler = ClockSampler(device.index).start()
    time.sleep(0.3)
    t_load0 = time.time()
    elapsed = time_schedule(case, args.steps, args.warmup, stream)
    if elapsed < 1.0:
        keep_busy(case, stream, 1.0 - elapsed)
    t_load1 = time.time()
    clocks = sampler.summary(t_load0, t_load1)
    e_max, rows_total = aggregate_over_ranks(elapsed, case.M * args.steps)
    value = rows_total / e_max
    per_call = elapsed / args.steps
    achieved = case.alg_bytes / per_call / 1e9
    kernel = KERNEL_NAMES[case.plan.family]
    traffic = profiled_traffic(kernel, case.name)
    e2e_steps = max(3, min(args.steps, 200))
    e2e = None if args.no_e2e else _e2e_entry(case, e2e_steps, args.warmup, stream)

    # Per-workload table (one process only: a replica run times the headline).
    per_config = {}
    if args.all_configs and world == 1:
        import workloads
        for name in workloads.ORDER:
            c = case if (name == case.name and args.rows is None) else \
                Case(name, device, seed_offset=rank)
            sec = median_per_call(c, stream)
            gbs = c.alg_bytes / sec / 1e9
            entry = {
                "workload": c.w.description, "M": c.M, "N": c.N, "K": c.K,
                "family": KERNEL_NAMES[c.plan.family], "stride": c.plan.stride,
                "dual": c.plan.dual, "splits": c.plan.splits, "workers": c.plan.workers,
                "us_per_call": sec * 1e6, "rows_per_s": c.M / sec, "gbs": gbs,
                "frac_of_hbm_peak": gbs / peak, "alg_bytes_per_call": c.alg_bytes,
                "l2": c.l2_note(), "routes": c.route_rates(),
                "traffic_bytes_per_launch": profiled_traffic(KERNEL_NAMES[c.plan.family], name),
            }
            if c is case:
                entry["e2e"] = e2e if e2e is not None else _e2e_entry(c, e2e_steps, args.warmup,
                                                                      stream)
            else:
                entry["e2e"] = _e2e_entry(c, e2e_steps, args.warmup, stream)
            if not args.no_cpu:
                entry["cpu_baseline"] = (
                    cpu_baseline(c, seconds=args.cpu_config_seconds,
                                 rows_cap=CPU_SAMPLE_ROWS.get(name)))
            per_config[name] = entry
            if c is not case:
                del c
                torch.cuda.empty_cache()
    guess_series = None
    if args.all_configs and world == 1:
        guess_series = guess_series_measure(device, stream)
        torch.cuda.empty_cache()
    sampler.stop()
    clocks_all = sampler.summary()

    cpu = None
    if world == 1 and not args.no_cpu:
        cpu = cpu_baseline(case, seconds=args.cpu_seconds,
                           rows_cap=CPU_SAMPLE_ROWS.get(case.name))

    if rank == 0:
        line = {
            "metric": "rows/s and score-row HBM GB/s (fraction of GB300 peak) per config, 1 GPU",
            "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": e_max / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; indexer-like scores stand in for the paper's captures)",
            "config": {"workload": case.w.description, "name": case.name, "M": case.M,
                       "N": case.N, "K": case.K, "l2": case.l2_note(),
                       "family": KERNEL_NAMES[case.plan.family], "stride": case.plan.stride,
                       "dual": case.plan.dual, "splits": case.plan.splits,
                       "parallelism": f"replicas x{world} (rows are independent)"},
            "score_row_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "kernel": kernel,
                         "peak_source": peak_src,
                         "alg_bytes_per_launch": case.alg_bytes},
            "gpu_launches": args.steps,
            "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "clock_samples": clocks.get("samples"),
            "e2e": e2e,
            "cpu_baseline": cpu,
            "per_config": per_config,
            "decode_guess_series": guess_series,
            "clocks_whole_run": clocks_all,
        }
        print(json.dumps(line), flush=True)
    finish_ranks(world)


def launch_replicas(args, argv):
    """`bench.py --gpus N` started without a launcher: start N copies of this
    script, one per GPU (RANK = LOCAL_RANK = i, WORLD_SIZE = N, rendezvous on
    127.0.0.1), pass rank 0's JSON line through and fail if any rank fails."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    procs = []
    for r in range(args.gpus):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(args.gpus),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv],
                                      env=env, stdout=subprocess.PIPE if r == 0 else
                                      subprocess.DEVNULL, text=True))
    out, _ = procs[0].communicate()
    rc = procs[0].returncode
    for p in procs[1:]:
        rc = max(rc, p.wait())
    sys.stdout.write(out)
    sys.stdout.flush()
    return rc


def run_reference(args):
    """The reference arm: the CPU oracle, timed on the host's cores, on the
    same workload, each step a bounded sample of its rows."""
    import numpy as np

    import oracle
    import workloads
    rank, _, world = dist_env()
    if rank != 0:
        return
    # The same matrix as our arm's rank 0 (made by the seeded generator on the
    # GPU when there is one, which is only faster), selected on the host.
    import torch
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    X, ke, K = workloads.generate(args.workload, device=gen_dev)
    X, ke = X.cpu().numpy(), ke.cpu().numpy()
    M, N = X.shape
    threads = oracle.hardware_threads()
    t0 = time.perf_counter()
    oracle.topk_rows(X[:min(M, 8)], ke[:min(M, 8)], K, nthreads=threads)
    per_row = (time.perf_counter() - t0) / min(M, 8)
    budget = args.reference_seconds / max(1, args.steps + args.warmup)
    rows_per_step = int(max(1, min(M, budget / max(per_row, 1e-9))))
    for i in range(args.warmup):
        oracle.topk_rows(X[:rows_per_step], ke[:rows_per_step], K, nthreads=threads)
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        lo = (i * rows_per_step) % M
        hi = min(M, lo + rows_per_step)
        oracle.topk_rows(X[lo:hi], ke[lo:hi], K, nthreads=threads)
        done += hi - lo
    dt = time.perf_counter() - t0
    value = done / dt
    w = workloads.WORKLOADS[args.workload]
    cpu = {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
           "sample": f"{rows_per_step} of {M} rows per step"}
    line = {"impl": "reference",
            "metric": "rows/s and score-row HBM GB/s (fraction of GB300 peak) per config, 1 GPU",
            "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / max(1, args.steps) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": w.description, "name": w.name, "M": M,
                                            "N": N, "K": K},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--rows", type=int, default=None,
                    help="row count override (smaller cases for profiling)")
    ap.add_argument("--all-configs", dest="all_configs", action="store_true", default=True)
    ap.add_argument("--headline-only", dest="all_configs", action="store_false")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-config-seconds", type=float, default=3.0,
                    help="CPU-oracle sample length of each per-config entry")
    ap.add_argument("--stub", action="store_true",
                    help="launcher/aggregation test without a GPU (the line is not a measurement)")
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--sweep", choices=["crossover", "margins", "splits", "trace", "floor"],
                    default=None,
                    help="planner study instead of the bench line (one JSON line per point)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    return args


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if args.gpus < 1:
        raise SystemExit("bench.py: --gpus must be >= 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch_replicas(args, argv)
    if args.stub:
        return run_stub(args)
    if args.impl == "reference":
        run_reference(args)
    else:
        import __graft_entry__
        __graft_entry__.build()
        if args.sweep:
            run_sweep(args)
        else:
            run_ours(args)


if __name__ == "__main__":
    sys.exit(main() or 0)
