#!/usr/bin/env python3
"""Benchmark of the LLM.int8() decomposition linear on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload large|prefill|decode|decode_k8192|sweep|tiny|blockwise]

Prints ONE JSON line (rank 0).  Metric: effective TOPS = 2*T*N*K / time of
the int8 decomposition linear, whole job.

Default workload: the large MLP configuration (X fp16 [4096, 8192] with 8
seeded outlier columns x U(8,60), W fp16 [28672, 8192] ~ N(0, 0.015), tau 6),
the largest configuration that fits one GPU.  A step is R replays of a CUDA
graph of L library calls, one per distinct layer (own int8 weight, fp16
weight, input and output; L such that the streamed bytes exceed twice the L2,
queried from the device), with R chosen so that the timed region lasts at
least --min-timed-s (1.2 s) at the given --steps.  Inputs are resident in HBM.

`roofline` is for the dominant kernel: its algorithmic flops (tensor-bound
GEMM) or bytes (HBM-bound decode kernel) per launch over its average
duration, timed with CUDA events over a loop of about a second of graphs of
main-kernel-only calls (bnb_int8_linear_opts with BNB_OPT_MAIN_ONLY: the GEMM
on the activation-pass results the timed calls left in the workspace, or the
whole fused decode kernel).  The GEMM's denominator is the sustained bf16
figure of MEASURED_PEAKS.json (the burst one beside it); the decode kernel's
is the measured HBM copy bandwidth.

`other_regimes` measures, in the same run and the same way, the decode GEMV
configuration (X [16, 4096], W [4096, 4096]), a decode step through the large
MLP weight (X [16, 8192], W [28672, 8192]) and the prefill configuration.

`e2e` is the same metric through the public API with host buffers: every
call is bnb_int8_linear_from_host (a pinned host->device copy of X, the
layer, a device->host copy of Y), all inside the timed region; consecutive
calls alternate over two streams with their own device buffers and
workspaces, so that copies overlap the neighbouring call's kernel.  It has
its own warm-up (--e2e-warmup calls), then --e2e-calls timed calls (2000), fewer only
where they would take longer than --e2e-timed-s (10 s).

`--impl reference` times the CPU oracle (the reference arm of this build):
each step is a bounded sample of the same workload (all rows of X, a
rotating slice of output channels), so that the whole run ends in minutes.

Multi-GPU (torchrun): replicas.  Each rank runs the same workload on its own
batch with no collective on the data path (weak scaling); the time is the
maximum over ranks between barriers.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import inputs  # noqa: E402

METRIC = "int8-decomposed linear effective TOPS (2*T*N*K/s)"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def make_workload(name: str, T: int):
    if name == "decode":
        return inputs.decode(T=T)
    if name == "decode_t1":  # the decode workload at one token (batch-1 generation)
        return inputs.decode(T=1)
    if name == "decode_k8192":  # a decode step through the large MLP weight
        return inputs.decode(T=T, K=8192, N=28672)
    if name == "decode_n11008":  # a decode step through the prefill weight
        return inputs.decode(T=T, K=4096, N=11008)
    if name == "prefill":
        return inputs.prefill()
    if name == "large":
        return inputs.large()
    if name == "sweep":
        return inputs.sweep(0.001, 6.0)
    if name == "tiny":
        return inputs.tiny()
    raise ValueError(name)


def algorithmic_bytes(T, N, K, nO, bias=False, wq_only=False):
    """Bytes the method must move for one call: X read once, Wq + scales read
    once, the outlier columns of W16 (none with only the int8 weight), the fp16
    bias if any, Y written once."""
    w16 = 0 if wq_only else 2 * N * nO
    return 2 * T * K + N * K + 4 * N + w16 + 2 * T * N + (2 * N if bias else 0)


# DRAM bytes per launch of a dominant kernel from an ncu capture of this
# benchmark's own workload (profiles/), valid only while the kernel's source
# is the one that was captured (first 16 hex digits of its SHA-256).
MEASURED_TRAFFIC = {
    # (kernel, T, K, N): (source file, source digest, dram read + write bytes)
    # one ncu capture of the large workload's GEMM launch: 930.92 MB read + 247.37 MB written
    ("gemm_tc", 4096, 8192, 28672): ("gemm_tc.cu", "25383f2e26f639e0", 1_178_290_000),
    # one ncu capture of the decode workload's kernel (bytes): T 16 (the
    # clustered kernel) and T 1 (the kernel without clusters), nothing written
    # (captured on decode.cu 902e6ba0c69afeb9, whose kernels the recorded
    # source keeps unchanged: it differs in one comment)
    ("dec_fused", 16, 4096, 4096): ("decode.cu", "892163d0c55e4732", 19_117_824),
    ("dec_local", 1, 4096, 4096): ("decode.cu", "892163d0c55e4732", 18_957_568),
}


def measured_traffic(kernel, T, K, N):
    import hashlib
    rec = MEASURED_TRAFFIC.get((kernel, T, K, N))
    if rec is None:
        return None
    path = os.path.join(ROOT, "int8_mixed_precision_04_b300", "csrc", rec[0])
    if not os.path.exists(path):
        return None
    digest = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    return rec[2] if digest == rec[1] else None


def kernel_algorithmic(kernel, T, N, K, nO, bias=False, wq_only=False):
    """(bytes, flops) per launch of one kernel, for the roofline."""
    b = 2 * N if bias else 0
    w16 = 0 if wq_only else 2 * N * nO  # the int8-weight-only GEMM reads compacted codes instead
    if kernel in ("dec_fused", "dec_local"):
        # the whole decode call: X read once, weight codes + scales + outlier
        # weight columns (+ bias), Y written once
        return 2 * T * K + N * K + 4 * N + w16 + 2 * T * N + b, 2 * T * N * K
    if kernel in ("gemm_mma", "gemm_tc"):
        return (N * K + 2 * T * K + 2 * T * N + (2 * N * nO) + b,
                2 * T * N * K + 2 * T * N * nO)
    if kernel == "outlier_scan":
        return 2 * T * K, 0
    if kernel == "quantize_rows":
        return 2 * T * K + T * K + 2 * T * nO, 0
    return 0, 0


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML reads only; nothing is set)
# ---------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clock and clock-event reasons with an nvidia-smi subprocess
    (read-only queries) while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int, period_ms: int = 50):
        self.cmd = ["nvidia-smi", "-i", str(index), "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", str(period_ms)]
        self.lines = []  # (arrival time, fields)
        self.t0 = self.t1 = None
        self.p = None

    def _reader(self):
        for line in self.p.stdout:
            self.lines.append((time.perf_counter(), [f.strip() for f in line.split(",")]))

    def __enter__(self):
        import subprocess
        try:
            self.p = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                      text=True)
        except OSError:
            self.p = None
            return self
        self.th = threading.Thread(target=self._reader, daemon=True)
        self.th.start()
        deadline = time.perf_counter() + 5.0
        while not self.lines and time.perf_counter() < deadline:  # first sample in
            time.sleep(0.01)
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_stop(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *a):
        if self.p is not None:
            time.sleep(0.06)
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
            self.th.join(timeout=5)

    def summary(self):
        if self.p is None or not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [f for (t, f) in self.lines
                  if self.t0 is not None and self.t0 <= t <= self.t1 + 0.06]
        window = "timed region"
        if not inside:  # region shorter than the sampling period: nearest samples
            inside = [f for (t, f) in self.lines][-3:]
            window = "samples adjacent to a timed region shorter than the sampling period"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(f[0]) for f in inside if num(f[0]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for f in inside:
            for name, val in zip(names, f[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][1]), "samples": len(inside), "window": window,
                "power_w_max": max((num(f[2]) or 0) for f in inside),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------

def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def _l2_bytes(dev) -> int:
    import torch
    v = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
    return int(v) if v else 126 * 1024 * 1024


def _graph(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def _time_replays(g, reps, stream, sampler=None, world=1, dev=None):
    """ms of `reps` replays of graph g on `stream` (CUDA events, synchronised
    on both sides; max over ranks)."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        barrier(world)
        torch.cuda.synchronize()
        if sampler:
            sampler.mark_start()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if sampler:
            sampler.mark_stop()
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1), world, dev)


def measure_layer(args, w, dev, world, local, steps, min_timed_s, min_layers=2,
                  with_e2e=True, with_kernel=True):
    """One workload measured the bench's way.  A step is R replays of a CUDA
    graph of L library calls, one per distinct layer (own int8 weight, fp16
    weight, input and output), with L large enough that the bytes the calls
    stream exceed twice the L2 and R large enough that `steps` steps take at
    least `min_timed_s`."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    lib = binding.load()
    T, K, N, tau = w.T, w.K, w.N, w.tau
    l2 = _l2_bytes(dev)
    layers = max(min_layers, math.ceil(2 * l2 / (N * K + 2 * T * K)))
    layers = min(layers, args.max_layers)
    edt = torch.bfloat16 if args.bf16 else torch.float16
    Xh = torch.from_numpy(w.X).to(edt)
    W16_0 = torch.from_numpy(w.W).to(dev).to(edt)
    W16s, Wqs, sws = [], [], []
    for i in range(layers):
        # distinct copies of the same weight (same numbers, distinct memory);
        # with --wq-only no fp16 weight stays resident
        Wc = W16_0.clone() if i else W16_0
        Wq, sw = binding.quantize_weight(Wc)
        W16s.append(None if args.wq_only else Wc)
        Wqs.append(Wq)
        sws.append(sw)
    Xs = [Xh.to(dev) for _ in range(layers)]
    Bs = ([torch.from_numpy(inputs.bias(N, K, seed=i)).to(dev).to(edt) for i in range(layers)]
          if args.bias else [None] * layers)
    Ys = [torch.empty((T, N), dtype=edt, device=dev) for _ in range(layers)]
    ws = torch.empty(binding.workspace_bytes(T, N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def calls(opts=0):
        for i in range(layers):
            if opts:
                binding.linear_opts(Xs[i], Wqs[i], sws[i], W16s[i], tau, opts, bias=Bs[i],
                                    Y=Ys[i], workspace=ws, stream=stream)
            elif args.wq_only:
                binding.linear_wq_only(Xs[i], Wqs[i], sws[i], Bs[i], tau, Y=Ys[i], workspace=ws,
                                       stream=stream)
            elif args.bias or args.bf16:
                binding.linear_ex(Xs[i], Wqs[i], sws[i], W16s[i], Bs[i], tau, Y=Ys[i],
                                  workspace=ws, stream=stream)
            else:
                binding.linear(Xs[i], Wqs[i], sws[i], W16s[i], tau, Y=Ys[i], workspace=ws,
                               stream=stream)

    dbg = binding.linear_debug(Xs[0], Wqs[0], sws[0], W16s[0], tau, want_acc=False)
    nO = int(dbg["nO"].item())
    del dbg
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            calls()
    stream.synchronize()
    before = lib.bnb_launch_count()
    g = _graph(calls, stream)
    launches_per_graph = lib.bnb_launch_count() - before
    for _ in range(3):
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()
    probe_ms = _time_replays(g, 5, stream, world=world, dev=dev) / 5
    R = max(1, math.ceil(min_timed_s * 1e3 / (steps * probe_ms)))
    sampler = ClockSampler(local)
    with sampler:
        ms = _time_replays(g, steps * R, stream, sampler, world, dev)
    ncalls = steps * R * layers
    ops = 2 * T * N * K
    value = world * ncalls * ops / (ms * 1e-3) / 1e12
    alg_bytes = algorithmic_bytes(T, N, K, nO, args.bias, args.wq_only)
    out = {
        "value": value, "ms_per_step": ms / steps, "us_per_call": ms * 1e3 / ncalls,
        "calls_per_step": R * layers, "layers": layers, "graph_replays_per_step": R,
        "timed_s": ms * 1e-3, "n_outliers": nO, "gb_per_s": world * ncalls * alg_bytes / (ms * 1e-3) / 1e9,
        "alg_bytes_per_call": alg_bytes, "path": lib.bnb_int8_linear_path(T, N, K),
        "gpu_launches": int(steps * R * launches_per_graph),
        "launches_per_call": launches_per_graph / layers,
        "clocks": sampler.summary(),
        "l2_bytes": l2,
    }
    # time x clock: SM cycles per call at the median clock of the timed region,
    # comparable between runs that the power cap holds at different clocks
    if out["clocks"].get("sm_mhz"):
        out["clocks"]["sm_cycles_per_call"] = out["us_per_call"] * out["clocks"]["sm_mhz"]
    peaks, peak_src = load_peaks()
    if with_kernel:
        # the dominant kernel alone: graphs of main-kernel-only calls (the GEMM
        # on the activation-pass results the calls above left in the workspace,
        # or the whole fused decode kernel), in the chain (programmatic
        # dependent launch on, as the library runs) and, for decode, also with
        # no overlap between consecutive launches
        path = out["path"]
        kname = {1: "dec_fused", 2: "gemm_tc", 3: "gemm_mma"}[path]
        if path == 1 and binding.decode_cluster(T, N, K) == 1:
            kname = "dec_local"  # the decode kernel without clusters
        kb, kf = kernel_algorithmic(kname, T, N, K, nO, args.bias, args.wq_only)
        res = {}
        for tag, opts in (("chain", binding.OPT_MAIN_ONLY),
                          ("alone", binding.OPT_MAIN_ONLY | binding.OPT_NO_PDL)):
            if tag == "alone" and path != 1:
                continue
            gk = _graph(lambda: calls(opts), stream)
            with torch.cuda.stream(stream):
                gk.replay()
            torch.cuda.synchronize()
            pk = _time_replays(gk, 3, stream, world=world, dev=dev) / 3
            Rk = max(3, math.ceil(min(args.kernel_timed_s, 2.0) * 1e3 / pk))
            kms = _time_replays(gk, Rk, stream, world=world, dev=dev)
            res[tag] = (kms * 1e-3 / (Rk * layers), Rk)
        kavg_s, Rk = res["chain"]
        if path == 1:
            roof = {"bound": "hbm", "achieved": kb / kavg_s / 1e9, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s"}
        else:
            # timed over a loop of about a second: the sustained figure is the
            # denominator; the burst one is reported beside it
            roof = {"bound": "tensor", "achieved": kf / kavg_s / 1e12,
                    "peak": peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
                    "unit": "TFLOP/s",
                    "peak_burst": peaks["bf16_tflops"],
                    "frac_of_burst": kf / kavg_s / 1e12 / peaks["bf16_tflops"]}
        roof["frac"] = roof["achieved"] / roof["peak"]
        # every kernel's algorithmic bytes against HBM too (the bound of
        # decode-sized calls, whichever kernel runs them)
        roof["alg_gbs"] = kb / kavg_s / 1e9
        roof["hbm_frac"] = roof["alg_gbs"] / peaks["hbm_gbs"]
        roof["traffic"] = (args.traffic if args.traffic is not None
                           else None if args.bias or args.wq_only or args.bf16
                           else measured_traffic(kname, T, K, N))
        roof["kernel"] = kname
        roof["peak_source"] = ("measured (MEASURED_PEAKS.json)" if peak_src == "measured"
                               else "fallback")
        # a decode call whose channels take several launches: per-launch figures
        # are the call's over its launches (achieved is the same either way)
        lpc = out["launches_per_call"] if path == 1 else 1
        roof["launches_per_call"] = lpc
        roof["kernel_avg_us"] = kavg_s * 1e6 / lpc
        roof["alg_bytes_per_launch"] = kb / lpc
        roof["alg_flops_per_launch"] = kf / lpc
        roof["timing"] = (f"graph of {layers} main-kernel-only calls x {Rk} replays "
                          f"(programmatic dependent launch on), CUDA events")
        if "alone" in res:
            a_s = res["alone"][0]
            roof["alone_us"] = a_s * 1e6
            roof["alone_frac"] = kb / a_s / 1e9 / peaks["hbm_gbs"]
        if path != 1:
            # the activation pass (workspace clear, column scan, row pass) alone
            ga = _graph(lambda: calls(binding.OPT_ACT_ONLY), stream)
            with torch.cuda.stream(stream):
                ga.replay()
            torch.cuda.synchronize()
            pa = _time_replays(ga, 3, stream, world=world, dev=dev) / 3
            Ra = max(3, math.ceil(0.3e3 / pa))
            ams = _time_replays(ga, Ra, stream, world=world, dev=dev)
            a_us = ams * 1e3 / (Ra * layers)
            roof["act_pass_us"] = a_us
            roof["act_pass_gbs"] = (4 * T * K + 2 * T * K) / (a_us * 1e-6) / 1e9
        out["roofline"] = roof

    if with_e2e:
        # e2e through the public API with host buffers: bnb_int8_linear_from_host
        # (pinned H2D of X, the layer, D2H of Y in one call), calls alternating
        # over two streams, each with its own device buffers and workspace
        streams2 = [stream, torch.cuda.Stream(device=dev)]
        Xpin = [Xh.pin_memory(), Xh.pin_memory()]
        Ypin = [torch.empty((T, N), dtype=edt).pin_memory() for _ in range(2)]
        Xdev = [Xs[0], torch.empty_like(Xs[0])]
        Ydev = [Ys[0], torch.empty_like(Ys[0])]
        wss = [ws, torch.empty_like(ws)]

        def e2e_call(i):
            j = i % 2
            binding.linear_from_host(Xpin[j], Wqs[i % layers], sws[i % layers], W16s[i % layers],
                                     tau, Ypin[j], Xdev[j], Ydev[j], wss[j], stream=streams2[j],
                                     bias=Bs[i % layers])

        def e2e_run(n):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            eb = torch.cuda.Event()
            torch.cuda.synchronize()
            barrier(world)
            e0.record(streams2[0])
            streams2[1].wait_event(e0)
            for i in range(n):
                e2e_call(i)
            eb.record(streams2[1])
            streams2[0].wait_event(eb)
            e1.record(streams2[0])
            torch.cuda.synchronize()
            return max_over_ranks(e0.elapsed_time(e1), world, dev)

        warm = e2e_run(max(2, args.e2e_warmup))  # also the estimate of a call's time
        per_call_ms = warm / max(2, args.e2e_warmup)
        n = int(min(args.e2e_calls, max(50, math.ceil(args.e2e_timed_s * 1e3 / per_call_ms))))
        e2e_ms = e2e_run(n)
        xb, yb = 2 * T * K, 2 * T * N
        out["e2e"] = {"value": world * n * ops / (e2e_ms * 1e-3) / 1e12, "unit": "TOPS",
                      "h2d_bytes_per_step": xb * R * layers, "d2h_bytes_per_step": yb * R * layers,
                      "calls": n, "warmup_calls": max(2, args.e2e_warmup),
                      "us_per_call": e2e_ms * 1e3 / n,
                      "note": "a step is the same calls_per_step calls; each call is "
                              "bnb_int8_linear_from_host (pinned H2D of X, the layer, D2H of Y); "
                              "calls alternate over two streams with their own device buffers "
                              "and workspaces"}
    del Xs, Ys, Wqs, W16s, ws
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import torch

    from int8_mixed_precision_04_b300 import binding, build
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()

    w = make_workload(args.workload, args.T)
    main = measure_layer(args, w, dev, world, local, args.steps, args.min_timed_s,
                         min_layers=16 if args.workload == "decode" else 2)
    T, K, N, tau = w.T, w.K, w.N, w.tau
    form = "bf16" if args.bf16 else "fp16"
    line = {
        "metric": METRIC,
        "value": main["value"],
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": main["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("int8xint8->int32 + bf16 outliers, bf16 out" if args.bf16
                  else "int8xint8->int32 + fp16 outliers, fp16 out"),
        "data": "synthetic (seeded, inputs module)",
        "config": {
            "workload": f"{args.workload}: X {form} [{T},{K}], W {form} [{N},{K}], tau {tau}",
            "T": T, "K": K, "N": N, "tau": tau, "n_outliers": main["n_outliers"],
            "bias": bool(args.bias), "fp16_weight_resident": not args.wq_only,
            "layers": main["layers"], "calls_per_step": main["calls_per_step"],
            "l2": (f"inputs larger than L2: {main['layers']} distinct layers cycled "
                   f"({main['layers'] * (N * K + 2 * T * K) / 1e6:.0f} MB of int8 weights and "
                   f"16-bit activations) vs {main['l2_bytes'] / 2**20:.0f} MiB L2"),
            "timing": (f"CUDA graph of {main['layers']} library calls replayed "
                       f"{main['graph_replays_per_step']} times per step; CUDA events; "
                       f"timed region {main['timed_s']:.2f} s"),
            "parallelism": f"replicas x{world}",
            "path": main["path"],
        },
        "us_per_call": main["us_per_call"],
        "gb_per_s": main["gb_per_s"],
        "alg_bytes_per_call": main["alg_bytes_per_call"],
        "e2e": main["e2e"],
        "gpu_launches": main["gpu_launches"],
        "launches_per_call": main["launches_per_call"],
        "roofline": main["roofline"],
        "clocks": main["clocks"],
    }
    # the other regimes of the layer, measured the same way in the same run
    subs = {}
    for name in [s for s in args.sub.split(",") if s and s != args.workload]:
        ws_ = make_workload(name, args.T)
        r = measure_layer(args, ws_, dev, world, local, args.steps, args.sub_timed_s,
                          min_layers=16 if name.startswith("decode") else 2, with_e2e=False)
        subs[name] = {"workload": f"X [{ws_.T},{ws_.K}], W [{ws_.N},{ws_.K}], tau {ws_.tau}",
                      "value_tops": r["value"], "us_per_call": r["us_per_call"],
                      "gb_per_s": r["gb_per_s"], "path": r["path"], "layers": r["layers"],
                      "calls_timed": args.steps * r["calls_per_step"],
                      "roofline": r["roofline"], "clocks": r["clocks"]}
    if subs:
        line["other_regimes"] = subs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget, **_forms(args))
    return line


# ---------------------------------------------------------------------------
# the oracle on the host cores: cpu_baseline and --impl reference
# ---------------------------------------------------------------------------

class OracleArm:
    """One bounded sample of the workload per step: activation pass over all
    T rows, then S4..S6 for all T rows against a rotating slice of `n_slice`
    output channels."""

    def __init__(self, w, n_slice: int, bias: bool = False, wq_only: bool = False,
                 bf16: bool = False):
        import oracle
        self.orc = oracle.get()
        self.w = w
        self.fmt = "bf16" if bf16 else "fp16"
        self.X, self.W = w.X, w.W
        self.b = inputs.bias(w.N, w.K, seed=0) if bias else None
        if bf16:  # the same values rounded to bf16, as the GPU arm's casts do
            self.X, self.W = _bf16_bits(w.X), _bf16_bits(w.W)
            self.b = None if self.b is None else _bf16_bits(self.b)
        self.wq_only = wq_only
        self.Wq, self.sw = self.orc.quantize_weight(self.W, fmt=self.fmt)
        self.n_slice = max(1, min(n_slice, w.N))
        self.pos = 0

    def step(self):
        n0 = self.pos
        n1 = min(self.w.N, n0 + self.n_slice)
        self.pos = 0 if n1 >= self.w.N else n1
        self.orc.linear(self.X, self.Wq[n0:n1], self.sw[n0:n1],
                        None if self.wq_only else self.W[n0:n1], self.w.tau,
                        bias=None if self.b is None else self.b[n0:n1], fmt=self.fmt)
        return 2 * self.w.T * (n1 - n0) * self.w.K


def _bf16_bits(a):
    """fp16 (or fp32) values -> bfloat16 bit patterns, nearest-even."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _forms(args):
    return dict(bias=bool(getattr(args, "bias", False)),
                wq_only=bool(getattr(args, "wq_only", False)),
                bf16=bool(getattr(args, "bf16", False)))


def _calibrate(w, target_s, **forms):
    arm = OracleArm(w, 64, **forms)
    t0 = time.perf_counter()
    arm.step()
    dt = time.perf_counter() - t0
    per_chan = dt / 64
    return max(1, int(target_s / max(per_chan, 1e-9)))


def cpu_baseline(w, budget_s: float = 15.0, **forms):
    import oracle
    n_slice = _calibrate(w, budget_s / 4, **forms)
    arm = OracleArm(w, n_slice, **forms)
    ops = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        ops += arm.step()
    dt = time.perf_counter() - t0
    return {"value": ops / dt / 1e12, "unit": "TOPS", "cores": oracle.get().num_threads(),
            "kind": "oracle",
            "sample": f"{w.name}: all {w.T} rows x {ops // (2 * w.T * w.K)} output channels "
                      f"({dt:.1f} s, slices of {n_slice} channels)"}


def run_reference(args, world, rank, local):
    if rank != 0:
        return None
    import oracle
    w = make_workload(args.workload, args.T)
    total_steps = args.steps + args.warmup
    per_step = min(2.0, args.ref_budget / max(total_steps, 1))
    forms = _forms(args)
    n_slice = _calibrate(w, per_step, **forms)
    arm = OracleArm(w, n_slice, **forms)
    for _ in range(args.warmup):
        arm.step()
    ops = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ops += arm.step()
    dt = time.perf_counter() - t0
    val = ops / dt / 1e12
    cores = oracle.get().num_threads()
    sample = (f"{w.name}: per step all {w.T} rows x {n_slice} output channels "
              f"(of {w.N}), K={w.K}")
    return {
        "impl": "reference",
        "metric": METRIC, "value": val, "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (f"int8xint8->int32 + {'bf16' if forms['bf16'] else 'fp16'} outliers "
                  f"(CPU oracle, fp64 epilogue)"),
        "data": "synthetic (seeded, inputs module)",
        "config": {"workload": (f"{args.workload}: X {'bf16' if forms['bf16'] else 'fp16'} "
                                f"[{w.T},{w.K}], W {'bf16' if forms['bf16'] else 'fp16'} "
                                f"[{w.N},{w.K}], tau {w.tau}"),
                   "T": w.T, "K": w.K, "N": w.N, "tau": w.tau, "bias": forms["bias"],
                   "fp16_weight_resident": not forms["wq_only"]},
        "cpu_baseline": {"value": val, "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_blockwise(args, world, rank, local):
    """The blockwise 8-bit codec of optimizer states: one step quantizes the
    fp32 state of the large MLP weight (28672 x 8192 values, 940 MB) in blocks
    of 256 and decodes it back.  Metric: algorithmic GB/s of the step
    (quantize reads 4n and writes n + 4n/B; dequantize reads n + 4n/B and
    writes 4n)."""
    import torch

    from int8_mixed_precision_04_b300 import binding, build
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()
    peaks, peak_src = load_peaks()
    n, B = 28672 * 8192, 256
    nb = (n + B - 1) // B
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    x = torch.randn(n, generator=g, device=dev, dtype=torch.float32) * 1e-3
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    absmax = torch.empty(nb, dtype=torch.float32, device=dev)
    y = torch.empty(n, dtype=torch.float32, device=dev)
    qbytes, dbytes = 4 * n + n + 4 * nb, n + 4 * nb + 4 * n
    stream = torch.cuda.Stream(device=dev)

    def graph_of(fn, reps):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for _ in range(reps):
                fn()
        return gr

    def timed(gr, reps, replays, sampler=None):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            gr.replay()
            barrier(world)
            torch.cuda.synchronize()
            if sampler:
                sampler.mark_start()
            e0.record(stream)
            for _ in range(replays):
                gr.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            if sampler:
                sampler.mark_stop()
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / (reps * replays)

    def quant():
        binding.quantize_blockwise(x, B, codes=codes, absmax=absmax, stream=stream)

    def dequant():
        binding.dequantize_blockwise(codes, absmax, B, y=y, stream=stream)

    def step():
        quant()
        dequant()

    reps = 4
    replays = max(1, args.steps // reps) if args.steps < 10000 else 10
    gs = graph_of(step, reps)
    sampler = ClockSampler(local)
    with sampler:
        step_ms = timed(gs, reps, replays, sampler)
    q_ms = timed(graph_of(quant, reps), reps, replays)
    d_ms = timed(graph_of(dequant, reps), reps, replays)
    value = world * (qbytes + dbytes) / (step_ms * 1e-3) / 1e9
    q_gbs = qbytes / (q_ms * 1e-3) / 1e9
    # e2e: the fp32 state from pinned host memory, the codec, the decoded
    # state back to pinned host memory
    xh = x.cpu().pin_memory()
    yh = torch.empty(n, dtype=torch.float32).pin_memory()
    with torch.cuda.stream(stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(2):
            x.copy_(xh, non_blocking=True)
            step()
            yh.copy_(y, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / 2
    line = {
        "metric": "blockwise int8 codec GB/s (algorithmic bytes of quantize + dequantize)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": reps * replays,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp32 -> int8 + fp32 absmax -> fp32",
        "data": "synthetic (seeded torch normal x 1e-3)",
        "config": {"workload": f"blockwise: fp32 state [{n}] (28672 x 8192), blocks of {B}",
                   "n": n, "block": B,
                   "l2": "inputs larger than L2: 940 MB state vs 126 MB L2",
                   "timing": "CUDA graph replay, CUDA events", "parallelism": f"replicas x{world}"},
        "e2e": {"value": (qbytes + dbytes) / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 4 * n, "calls": 2,
                "note": "pinned H2D of the state, quantize + dequantize, D2H of the decoded state"},
        "gpu_launches": 2 * reps * replays,
        "roofline": {"bound": "hbm", "achieved": q_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": q_gbs / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "quantize_blockwise", "peak_source": peak_src,
                     "kernel_avg_us": q_ms * 1e3, "alg_bytes_per_launch": qbytes,
                     "dequantize_avg_us": d_ms * 1e3,
                     "dequantize_gbs": dbytes / (d_ms * 1e-3) / 1e9},
        "clocks": sampler.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        orc = oracle.get()
        m = 1 << 24
        xs = x[:m].cpu().numpy()
        t0 = time.perf_counter()
        reps_cpu = 0
        while time.perf_counter() - t0 < args.cpu_budget:
            q_o, a_o = orc.quantize_blockwise(xs, B)
            orc.dequantize_blockwise(q_o, a_o, B)
            reps_cpu += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": reps_cpu * (10 * m + 8 * (m // B)) / dt / 1e9,
                                "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                                "sample": f"the first {m} values, {reps_cpu} passes in {dt:.1f} s"}
    return line


def run_reference_blockwise(args, world, rank, local):
    """The reference arm of the codec workload: the oracle's codec, as it
    stands, on a bounded sample of the same state (the first 2^22 values of a
    seeded normal x 1e-3 state), each step one quantize + decode pass."""
    if rank != 0:
        return None
    import oracle
    orc = oracle.get()
    n, B, m = 28672 * 8192, 256, 1 << 22
    rng = np.random.default_rng(1234)
    xs = (rng.standard_normal(m) * 1e-3).astype(np.float32)
    step_bytes = 10 * m + 8 * ((m + B - 1) // B)
    for _ in range(args.warmup):
        orc.dequantize_blockwise(*orc.quantize_blockwise(xs, B), B)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.dequantize_blockwise(*orc.quantize_blockwise(xs, B), B)
    dt = time.perf_counter() - t0
    val = args.steps * step_bytes / dt / 1e9
    sample = f"the first {m} values of the state per step, blocks of {B}"
    return {
        "impl": "reference",
        "metric": "blockwise int8 codec GB/s (algorithmic bytes of quantize + dequantize)",
        "value": val, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 -> int8 + fp32 absmax -> fp32 (CPU oracle)",
        "data": "synthetic (seeded normal x 1e-3)",
        "config": {"workload": f"blockwise: fp32 state [{n}] (28672 x 8192), blocks of {B}",
                   "n": n, "block": B},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large",
                    choices=["decode", "decode_t1", "decode_k8192", "decode_n11008", "prefill",
                             "large", "sweep", "tiny", "blockwise"])
    ap.add_argument("--T", type=int, default=16, help="tokens of the decode workloads")
    ap.add_argument("--max-layers", type=int, default=64)
    ap.add_argument("--min-timed-s", type=float, default=1.2,
                    help="the timed region lasts at least this long (graph replays per step)")
    ap.add_argument("--kernel-timed-s", type=float, default=1.0,
                    help="length of the dominant-kernel timing loop")
    ap.add_argument("--sub", default="decode,decode_t1,decode_k8192,decode_n11008,prefill",
                    help="other regimes measured in the same run (comma list, '' for none)")
    ap.add_argument("--sub-timed-s", type=float, default=0.5)
    ap.add_argument("--e2e-calls", type=int, default=2000)
    ap.add_argument("--e2e-warmup", type=int, default=100)
    ap.add_argument("--e2e-timed-s", type=float, default=10.0,
                    help="upper bound on the e2e timed region: --e2e-calls calls unless fewer fit")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bias", action="store_true",
                    help="layers with an fp16 bias (bnb_int8_linear_bias)")
    ap.add_argument("--bf16", action="store_true",
                    help="X, W16, bias and Y in bf16 (bnb_int8_linear_ex)")
    ap.add_argument("--wq-only", action="store_true",
                    help="only the int8 weight resident (bnb_int8_linear_wq_only)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference" and args.workload == "blockwise":
        line = run_reference_blockwise(args, world, rank, local)
    elif args.impl == "reference":
        line = run_reference(args, world, rank, local)
    elif args.workload == "blockwise":
        line = run_blockwise(args, world, rank, local)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
