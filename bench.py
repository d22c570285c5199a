#!/usr/bin/env python3
"""Benchmark of the Q8_0 quantized projection on GB300.

Default workload: the decode-step projections of a d = 4096 Llama-shaped
layer at rows = 1 -- Wqkv 6144x4096, Wo 4096x4096, fused gate+up 28672x4096,
down 4096x14336, all Q8_0 -- each fed by its producer (RMSNorm of an N(0,1)
hidden vector, quantized in the producer's epilogue), in all three activation
modes (two-word ~14-bit, one int8 word, f32 with f64 sums).  One step runs the
12 fused producer+projection calls.  Two rotating copies of the weights
(463 MB) keep every step's reads larger than the 129 MB L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line on rank 0.  Under torchrun (N > 1) every rank runs its own
replica (the projection has no exchange step on one node here), the time is
the maximum over ranks and `value` sums the ranks' bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from q8_quantized_projection_gb300 import synth  # noqa: E402

METRIC = "Q8_0 proj weight GB/s (% of GB300 HBM peak) at rows 1–256; rows/s"
MODES = ("i8x2", "i8", "f32")
WORKLOAD = "decode_layer_d4096_rows1"
COPIES = 2
QK = 32


def weight_bytes(n, k):
    return n * k + n * (k // QK) * 2     # 34 bytes per 32 weights


LAYER_BYTES = sum(weight_bytes(n, k) for _, n, k in synth.LAYER_D4096)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- distributed

def dist_init():
    """One process per GPU (replicas: no data-path collective).  Q8_BENCH_BACKEND
    overrides the process-group backend (the CPU tests use gloo)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("Q8_BENCH_BACKEND") or (
            "nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_gbps(world, bytes_per_rank_step, ms_per_step_max):
    """Whole-job rate: the bytes every rank streamed per step over the slowest
    rank's step time (replicas, weak scaling)."""
    return world * bytes_per_rank_step / (ms_per_step_max * 1e-3) / 1e9


def max_over_ranks(world, v):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- inputs

def make_host_inputs(seed=0):
    rng = synth.rng_for(seed)
    mats, hs = [], []
    for name, n, k in synth.LAYER_D4096:
        q, s = synth.q8_weights(rng, n, k)
        mats.append((name, q, s))
        hs.append(synth.activations(rng, 1, k))
    return mats, hs


# ------------------------------------------------------------- oracle arm

def oracle_step(mats, hs, modes=MODES):
    """One step of the workload on the CPU oracle: producer then projection."""
    from oracle import oracle as orc
    for mode in modes:
        for (_, q, s), h in zip(mats, hs):
            x, _ = orc.rmsnorm(h)
            orc.project(mode, q, s, orc.quantize(mode, x))


def _timed_oracle_steps(mats, hs, budget_s):
    t0 = time.perf_counter()
    steps = 0
    while True:
        oracle_step(mats, hs)
        steps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return steps, time.perf_counter() - t0


def cpu_baseline(mats, hs, budget_s=10.0):
    """The oracle on the host cores (OpenMP over output rows), then the same
    code on one thread for a shorter sample (results are identical: each
    output's order of operations does not depend on the thread count)."""
    from oracle import oracle as orc
    orc.build()
    steps, dt = _timed_oracle_steps(mats, hs, budget_s)
    cores = orc.threads()
    orc.set_threads(1)
    try:
        steps1, dt1 = _timed_oracle_steps(mats, hs, budget_s * 0.3)
    finally:
        orc.set_threads(cores)
    return {"value": round(steps * len(MODES) * LAYER_BYTES / dt / 1e9, 4), "unit": "GB/s",
            "cores": cores, "kind": "oracle", "arch": platform.machine(),
            "sample": f"{steps} full step(s) of {WORKLOAD} (3 modes x 4 projections, RMSNorm + "
                      f"quantize + projection) in {dt:.1f} s; plain C oracle, OpenMP over "
                      f"output rows",
            "single_thread": {"value": round(steps1 * len(MODES) * LAYER_BYTES / dt1 / 1e9, 4),
                              "unit": "GB/s", "cores": 1,
                              "sample": f"{steps1} full step(s) in {dt1:.1f} s, one thread"}}


def run_reference(args, world, rank):
    if rank != 0:
        return
    from oracle import oracle as orc
    orc.build()
    mats, hs = make_host_inputs()
    for _ in range(args.warmup):
        oracle_step(mats, hs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(mats, hs)
    dt = time.perf_counter() - t0
    ms = dt / args.steps * 1e3
    value = len(MODES) * LAYER_BYTES / (ms * 1e-3) / 1e9
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "int8/f32(f64-sum)", "data": "synthetic",
           "config": {"workload": WORKLOAD, "rows": 1, "modes": list(MODES),
                      "matrices": [f"{n}x{k}" for _, n, k in synth.LAYER_D4096]},
           "rows_per_s": round(len(MODES) * 4 / (ms * 1e-3), 2),
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": orc.threads(),
                            "kind": "oracle", "arch": platform.machine(),
                            "sample": f"the whole step, {args.steps} timed steps"},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# --------------------------------------------------------------- our arm

# The sources the fused decode kernels are compiled from (the decode kernel
# of the f32 mode and the row-per-lane kernel of the int8 modes, their headers
# and three instantiation units); the C-ABI layer and the other kernels are not.
DECODE_KERNEL_SOURCES = ("common.cuh", "launch.h", "gemv.cuh", "gemv_row.cuh", "gemv_rpl.cuh", "rmsnorm.cuh",
                         "gemv_f32.cu", "gemv_i8.cu", "gemv_i8x2.cu")

# The kernel each mode's fused decode launch runs (the layer's K are all
# multiples of 1024 and at most 16384, which the row-per-lane kernel takes)
FUSED_KERNEL = {"f32": "gemv_rpl_kernel<0,1,1,0,0,0>", "i8": "gemv_rpl_kernel<1,1,1,0,0,0>",
                "i8x2": "gemv_rpl_kernel<2,1,1,0,0,0>"}


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "q8_quantized_projection_gb300", "csrc")
    for name in DECODE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it is current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("source_hash") == kernel_source_hash():
            return e.get("bytes_per_launch")
    except Exception:
        pass
    return None


def run_ours(args, world, rank, local):
    import torch
    from q8_quantized_projection_gb300 import build, native
    if rank == 0:
        build.build()
    barrier(world)
    native.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    mats, hs = make_host_inputs()
    Q = [[], []]
    S = [[], []]
    for _, q, s in mats:
        qd = torch.from_numpy(q).to(dev)
        sd = torch.from_numpy(s.view(np.int16)).to(dev)
        Q[0].append(qd)
        S[0].append(sd)
        for c in range(1, COPIES):
            Q[c].append(qd.clone())
            S[c].append(sd.clone())
    # the step's inputs in one buffer and each mode's outputs in one buffer (views
    # per projection, every offset a multiple of 128 bytes), so the end-to-end
    # step moves them with one copy each
    ks = [k for _, _, k in synth.LAYER_D4096]
    ns = [n for _, n, _ in synth.LAYER_D4096]
    H_all = torch.from_numpy(np.concatenate([h.reshape(-1) for h in hs])).to(dev)
    H = [H_all.narrow(0, sum(ks[:p]), ks[p]).view(1, ks[p]) for p in range(4)]
    Y_all = {m: torch.empty(sum(ns), dtype=torch.float32, device=dev) for m in MODES}
    Y = {m: [Y_all[m].narrow(0, sum(ns[:p]), ns[p]).view(1, ns[p]) for p in range(4)]
         for m in MODES}
    WS = {m: [torch.empty(native.q8_proj_fused_workspace(m, 1, k), dtype=torch.uint8, device=dev)
              for _, _, k in synth.LAYER_D4096] for m in MODES}
    launches_per_fused = 1   # every mode runs its producer inside the decode kernel

    def step(i, modes=MODES):
        c = i % COPIES
        for m in modes:
            for p in range(4):
                native.q8_proj_fused(m, Q[c][p], S[c][p], H[p], Y[m][p], WS[m][p])

    # The lane replays each step as one captured CUDA graph; so does the bench:
    # one graph per rotating weight copy, so host launch cost is not measured.
    def capture(fn):
        graphs = []
        for c in range(COPIES):
            fn(c)                      # eager run first: attributes, first-call set-up
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                fn(c)
            graphs.append(g)
        torch.cuda.synchronize(dev)
        return graphs

    cap_stream = torch.cuda.Stream(dev)

    def timed(graphs, nsteps):
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(nsteps):
            graphs[i % COPIES].replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return e0.elapsed_time(e1) / nsteps

    if args.case:
        # one projection's kernel, warmup+steps eager launches (a profiler case)
        parts = args.case.split(":")
        if parts[0] == "head":
            # the LM head with its arg-max: head:MODE:ROWS
            mode, rows = parts[1], int(parts[2])
            nh, kh = synth.HEAD_SHAPE
            qh, sh, hh, _ = synth.planted_head(4, nh, kh, rows)
            qd = torch.from_numpy(qh).to(dev)
            sd = torch.from_numpy(sh.view(np.int16)).to(dev)
            xq, xd = native.activation_buffers(mode, rows, kh, device=dev)
            native.act_quant(mode, torch.from_numpy(hh).to(dev), xq, xd, norm=True)
            tok = torch.empty(rows, dtype=torch.int32, device=dev)
            ws = native.argmax_workspace(rows, device=dev)
            for i in range(args.warmup + args.steps):
                native.head_argmax(mode, qd, sd, xq, xd, rows, tok, ws)
            torch.cuda.synchronize(dev)
            if rank == 0:
                print(json.dumps({"case": args.case, "launches": args.warmup + args.steps}))
            return
        if parts[0] == "chunk":
            # a prefill chunk: chunk:MODE:PROJ:T
            mode, proj, T = parts[1], parts[2], int(parts[3])
            p = [nm for nm, _, _ in synth.LAYER_D4096].index(proj)
            n, k = synth.LAYER_D4096[p][1], synth.LAYER_D4096[p][2]
            h = torch.from_numpy(synth.activations(synth.rng_for(3), T, k)).to(dev)
            xq, xd = native.activation_buffers(mode, T, k, device=dev)
            native.act_quant(mode, h, xq, xd, norm=True)
            y = torch.empty((T, n), dtype=torch.float32, device=dev)
            for i in range(args.warmup + args.steps):
                native.q8_proj_chunk(mode, Q[i % COPIES][p], S[i % COPIES][p], xq, xd, T, y)
            torch.cuda.synchronize(dev)
            if rank == 0:
                print(json.dumps({"case": args.case, "launches": args.warmup + args.steps}))
            return
        # MODE:PROJ[:fused | :rowsR], PROJ one of the layer's matrices or "all"
        # (the four in layer order each iteration); rowsR: a batch of R rows
        # through q8_proj (R seeded RMSNorm(N(0,1)) rows)
        mode, proj = parts[0], parts[1]
        fused = len(parts) > 2 and parts[2] == "fused"
        nrows = int(parts[2][4:]) if len(parts) > 2 and parts[2].startswith("rows") else 1
        names = [nm for nm, _, _ in synth.LAYER_D4096]
        projs = list(range(len(names))) if proj == "all" else [names.index(proj)]
        acts, Yb = {}, {}
        for p in projs:
            k = synth.LAYER_D4096[p][2]
            acts[p] = native.activation_buffers(mode, nrows, k, device=dev)
            hb = H[p] if nrows == 1 else torch.from_numpy(
                synth.activations(np.random.default_rng(20 + p), nrows, k)).to(dev)
            native.act_quant(mode, hb, acts[p][0], acts[p][1], norm=True)
            Yb[p] = Y[mode][p] if nrows == 1 else torch.empty(
                (nrows, synth.LAYER_D4096[p][1]), dtype=torch.float32, device=dev)
        for i in range(args.warmup + args.steps):
            for p in projs:
                if fused:
                    native.q8_proj_fused(mode, Q[i % COPIES][p], S[i % COPIES][p], H[p],
                                         Y[mode][p], WS[mode][p])
                else:
                    native.q8_proj(mode, Q[i % COPIES][p], S[i % COPIES][p], acts[p][0],
                                   acts[p][1], nrows, Yb[p])
        torch.cuda.synchronize(dev)
        if rank == 0:
            print(json.dumps({"case": args.case,
                              "launches": (args.warmup + args.steps) * len(projs)}))
        return

    step_graphs = capture(lambda c: step(c))
    for i in range(args.warmup):
        step_graphs[i % COPIES].replay()
    torch.cuda.synchronize(dev)

    if args.quick:
        ms = max_over_ranks(world, timed(step_graphs, args.steps))
        if rank == 0:
            print(json.dumps({"quick": True, "ms_per_step": ms,
                              "GB/s": len(MODES) * LAYER_BYTES / (ms * 1e-3) / 1e9}))
        return

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ms = timed(step_graphs, args.steps)
    # keep the same load running so the clock samples cover it
    t_hold = time.perf_counter()
    while time.perf_counter() - t_hold < 1.0:
        for i in range(50):
            step_graphs[i % COPIES].replay()
        torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(world, ms)
    step_bytes = len(MODES) * LAYER_BYTES
    value = aggregate_gbps(world, step_bytes, ms)

    # per-mode breakdown (same protocol): each mode's four fused launches in
    # layer order -- the kernels the step runs
    per_mode = {}
    # algorithmic bytes of one fused launch: 34/32 B per weight, the producer's
    # f32 input h and the f32 output
    mode_alg = float(sum(weight_bytes(n, k) + 4 * k + 4 * n for _, n, k in synth.LAYER_D4096))
    for m in MODES:
        gm = capture(lambda c, m=m: step(c, (m,)))
        for i in range(args.warmup):
            gm[i % COPIES].replay()
        mms = max_over_ranks(world, timed(gm, args.steps))
        per_mode[m] = {"ms_per_step": round(mms, 5),
                       "GB/s": round(LAYER_BYTES / (mms * 1e-3) / 1e9, 2),
                       "alg_GB/s": round(mode_alg / (mms * 1e-3) / 1e9, 2)}
        del gm

    # dominant kernel: the fused decode kernel of the mode that takes the
    # largest share of the step, timed as the step runs it (four launches in
    # layer order, chained by programmatic dependent launch, CUDA events on
    # the launching stream)
    peak, peak_kind = load_peaks()
    dom = max(MODES, key=lambda m: per_mode[m]["ms_per_step"])
    achieved = mode_alg / (per_mode[dom]["ms_per_step"] * 1e-3) / 1e9

    # sub-record: each fused projection replayed alone from graphs of REPS
    # launches, rotating over enough weight copies that each projection's
    # copies exceed twice the L2 (so no launch finds its weights in L2)
    reps = 20
    l2 = 129e6
    iso = {}
    for p, (nm, n, k) in enumerate(synth.LAYER_D4096):
        ncp = max(COPIES, int(np.ceil(2.2 * l2 / weight_bytes(n, k))))
        Qp = [Q[c % COPIES][p] if c < COPIES else Q[0][p].clone() for c in range(ncp)]
        Sp = [S[c % COPIES][p] if c < COPIES else S[0][p].clone() for c in range(ncp)]
        for m in MODES:
            def launches(c, p=p, m=m, Qp=Qp, Sp=Sp, ncp=ncp):
                for i in range(reps):
                    j = (c * reps + i) % ncp
                    native.q8_proj_fused(m, Qp[j], Sp[j], H[p], Y[m][p], WS[m][p])
            gp = capture(launches)
            for i in range(3):
                gp[i % COPIES].replay()
            us = timed(gp, max(args.steps // 5, 4)) / reps * 1e3
            alg = weight_bytes(n, k) + 4 * k + 4 * n
            iso.setdefault(m, {})[nm] = {"us": round(us, 2), "GB/s": round(alg / (us * 1e-6) / 1e9, 1),
                                         "weight_copies": ncp}
            del gp
        del Qp, Sp
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": committed_traffic(f"fused_{dom}"),
                "kernel": f"{FUSED_KERNEL[dom]} ({dom} mode, producer fused)",
                "peak_source": peak_kind, "launches": 4,
                "per_launch_us": round(per_mode[dom]["ms_per_step"] * 1e3 / 4, 3),
                "alg_bytes_per_launch": round(mode_alg / 4),
                "per_mode_GBps": {m: per_mode[m]["alg_GB/s"] for m in MODES},
                "isolated_replay": {"note": f"each fused projection replayed alone, graphs of {reps} "
                                            "launches rotating over weight copies > 2x L2",
                                    "per_projection": iso},
                "note": "the dominant kernel as the step runs it: its four fused launches "
                        "(Wqkv, Wo, gate+up, down) in layer order; achieved = their algorithmic "
                        "bytes (34/32 B per weight + f32 h in + f32 y out) over their time"}

    # end to end through the C ABI: pinned host inputs in, outputs back, every step.
    # One H2D copy of the step's inputs; each mode's outputs go back in one D2H
    # copy on a side stream as soon as that mode's four calls are done, while the
    # next mode computes; the step ends when every copy has landed.
    h_host = torch.from_numpy(np.concatenate([h.reshape(-1) for h in hs])).pin_memory()
    y_host = {m: torch.empty(sum(ns), dtype=torch.float32).pin_memory() for m in MODES}
    h2d = h_host.numel() * 4
    d2h = sum(y_host[m].numel() * 4 for m in MODES)
    side = torch.cuda.Stream(dev)

    def e2e_body(c):
        cur = torch.cuda.current_stream(dev)
        H_all.copy_(h_host, non_blocking=True)
        for m in MODES:
            step(c, (m,))
            ev = torch.cuda.Event()
            ev.record(cur)
            side.wait_event(ev)
            with torch.cuda.stream(side):
                y_host[m].copy_(Y_all[m], non_blocking=True)
        done = torch.cuda.Event()
        done.record(side)
        cur.wait_event(done)

    e2e_graphs = capture(e2e_body)
    for i in range(args.warmup):
        e2e_graphs[i % COPIES].replay()
        torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_graphs[i % COPIES].replay()
        torch.cuda.synchronize(dev)      # the host reads every step's outputs
    e2e_ms = max_over_ranks(world, (time.perf_counter() - t0) / args.steps * 1e3)
    e2e = {"value": round(aggregate_gbps(world, step_bytes, e2e_ms), 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
           "note": "host wall clock per step: graph replay of one H2D copy of the inputs, "
                   "12 C-ABI calls, one D2H copy of each mode's outputs (overlapping the next "
                   "mode's calls), then stream sync"}

    sweeps = {} if args.no_sweeps else run_sweeps(native, torch, dev, capture, timed, Q, S, mats,
                                                  oracle_slices=(rank == 0 and world == 1 and
                                                                 not args.no_cpu_baseline))

    # a kernel whose bounded wait ran out reports it here; its timings are void
    dev_err = native.q8_device_error()
    if dev_err:
        print(f"bench: device error word {dev_err}: a kernel wait timed out", file=sys.stderr)

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(mats, hs, budget_s=args.cpu_budget)

    if rank == 0:
        out = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "int8/f32(f64-sum)", "data": "synthetic",
               "config": {"workload": WORKLOAD, "rows": 1, "modes": list(MODES),
                          "matrices": [f"{nm} {n}x{k}" for nm, n, k in synth.LAYER_D4096],
                          "producer": "RMSNorm(N(0,1)) quantized in the producer (fused call)",
                          "l2": f"inputs larger than L2: {COPIES} rotating weight copies, "
                                f"{COPIES * LAYER_BYTES / 1e6:.0f} MB",
                          "parallelism": "replicas" if world > 1 else "single GPU"},
               "pct_hbm_peak": round(100 * value / world / peak, 2),
               "rows_per_s": round(world * len(MODES) * 4 / (ms * 1e-3), 1),
               "modes": per_mode, "roofline": roofline, "cpu_baseline": base, "e2e": e2e,
               "gpu_launches": args.steps * len(MODES) * 4 * launches_per_fused,
               "clocks": clocks, "sweeps": sweeps, "device_error": dev_err}
        print(json.dumps(out), flush=True)
    if dev_err:
        sys.exit(3)


def oracle_slice_us(fn, reps=3):
    """Host time of fn (the oracle on a slice of a workload), best of reps."""
    best = None
    for _ in range(reps):
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    return best * 1e6


def e2e_us(torch, dev, capture, body, steps=20):
    """Host wall clock per step of a captured step that copies its inputs in
    from pinned host memory and its results out, the host waiting for each."""
    graphs = capture(body)
    for i in range(3):
        graphs[i % COPIES].replay()
        torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(steps):
        graphs[i % COPIES].replay()
        torch.cuda.synchronize(dev)
    dt = (time.perf_counter() - t0) / steps
    del graphs
    return dt * 1e6


def run_sweeps(native, torch, dev, capture, timed, Q, S, mats, oracle_slices=True):
    """The other workload configurations, each graph-replayed with rotating
    inputs larger than L2: the 1024x1024 GEMV, batched decode, prefill chunks
    and the LM head with its arg-max.  The prefill chunk at T = 256 and the
    16-row head also run end to end (host buffers in and out through the C
    ABI), and the CPU oracle is timed on a slice of each (scaled to the whole
    workload, and labelled so)."""
    out = {}
    rng = synth.rng_for(7)
    if oracle_slices:
        from oracle import oracle as orc
        orc.build()

    def per_call_us(body, calls, nrep=10):
        graphs = capture(body)
        for i in range(3):
            graphs[i % COPIES].replay()
        ms = timed(graphs, nrep)
        del graphs
        return ms * 1e3 / calls

    # 1024 x 1024, rows = 1: launch-latency bound; 128 rotating copies (142 MB)
    q0, s0 = synth.q8_weights(rng, 1024, 1024)
    nrot = 128
    Q0 = [torch.from_numpy(q0).to(dev) for _ in range(nrot)]
    S0 = [torch.from_numpy(s0.view(np.int16)).to(dev) for _ in range(nrot)]
    h0 = torch.from_numpy(synth.activations(rng, 1, 1024)).to(dev)
    y0 = torch.empty((1, 1024), dtype=torch.float32, device=dev)
    cfg0 = {}
    for m in MODES:
        ws = torch.empty(native.q8_proj_fused_workspace(m, 1, 1024), dtype=torch.uint8, device=dev)

        def body(c, m=m, ws=ws):
            for i in range(nrot // COPIES):
                j = c * (nrot // COPIES) + i
                native.q8_proj_fused(m, Q0[j], S0[j], h0, y0, ws)
        us = per_call_us(body, nrot // COPIES)
        cfg0[m] = {"us_per_call": round(us, 2),
                   "GB/s": round(weight_bytes(1024, 1024) / (us * 1e-6) / 1e9, 1)}
    out["gemv_1024x1024_rows1"] = cfg0
    del Q0, S0

    # the decode layer with the residual added before the norm in every
    # producer (s = h + r written back), against the plain fused layer
    resid = {}
    Hs = [torch.from_numpy(synth.activations(rng, 1, k)).to(dev) for _, _, k in synth.LAYER_D4096]
    R_in = [torch.from_numpy(synth.activations(rng, 1, k)).to(dev) for _, _, k in synth.LAYER_D4096]
    S_out = [torch.empty((1, k), dtype=torch.float32, device=dev) for _, _, k in synth.LAYER_D4096]
    for m in MODES:
        ws = [torch.empty(native.q8_proj_fused_workspace(m, 1, k), dtype=torch.uint8, device=dev)
              for _, _, k in synth.LAYER_D4096]
        ys = [torch.empty((1, n), dtype=torch.float32, device=dev) for _, n, _ in synth.LAYER_D4096]

        def body_r(c, m=m, ws=ws, ys=ys):
            for p in range(4):
                native.q8_proj_fused_residual(m, Q[c][p], S[c][p], Hs[p], R_in[p], ys[p], ws[p],
                                              s_out=S_out[p])

        def body_p(c, m=m, ws=ws, ys=ys):
            for p in range(4):
                native.q8_proj_fused(m, Q[c][p], S[c][p], Hs[p], ys[p], ws[p])
        us_r = per_call_us(body_r, 1)
        us_p = per_call_us(body_p, 1)
        resid[m] = {"us_per_layer": round(us_r, 2), "plain_fused_us_per_layer": round(us_p, 2),
                    "GB/s": round(LAYER_BYTES / (us_r * 1e-6) / 1e9, 1)}
    out["decode_layer_residual_d4096"] = resid

    # the down projection (4096 x 14336) fed by its SwiGLU producer from the
    # gate+up output (2 x 14336 values), against the RMSNorm producer
    swi = {}
    _, n_dn, k_dn = synth.LAYER_D4096[3]
    GU = torch.from_numpy((synth.activations(rng, 1, 2 * k_dn) * 3.0).astype(np.float32)).to(dev)
    for m in MODES:
        ws = torch.empty(native.q8_proj_fused_workspace(m, 1, k_dn), dtype=torch.uint8, device=dev)
        yd = torch.empty((1, n_dn), dtype=torch.float32, device=dev)

        def body_s(c, m=m, ws=ws, yd=yd):
            native.q8_proj_fused_swiglu(m, Q[c][3], S[c][3], GU, yd, ws)

        def body_n(c, m=m, ws=ws, yd=yd):
            native.q8_proj_fused(m, Q[c][3], S[c][3], Hs[3], yd, ws)
        us_s = per_call_us(body_s, 1, nrep=20)
        us_n = per_call_us(body_n, 1, nrep=20)
        swi[m] = {"us_per_call": round(us_s, 2), "rmsnorm_producer_us_per_call": round(us_n, 2),
                  "GB/s": round(weight_bytes(n_dn, k_dn) / (us_s * 1e-6) / 1e9, 1)}
    out["down_swiglu_4096x14336"] = swi

    # Wqkv (q 4096 | K 1024 | V 1024) with the K/V slices written into the
    # cache rows a device position names (4096-row caches), against plain
    kvl = {}
    _, n_qkv, k_qkv = synth.LAYER_D4096[0]
    KC = torch.zeros((1, 4096, 1024), dtype=torch.float32, device=dev)
    VC = torch.zeros((1, 4096, 1024), dtype=torch.float32, device=dev)
    POS = torch.tensor([1234], dtype=torch.int32, device=dev)
    for m in MODES:
        ws = torch.empty(native.q8_proj_fused_workspace(m, 1, k_qkv), dtype=torch.uint8, device=dev)
        yq = torch.empty((1, n_qkv), dtype=torch.float32, device=dev)

        def body_kv(c, m=m, ws=ws, yq=yq):
            native.q8_proj_fused_kv(m, Q[c][0], S[c][0], Hs[0], yq, ws, POS, 4096, KC, VC)

        def body_q(c, m=m, ws=ws, yq=yq):
            native.q8_proj_fused(m, Q[c][0], S[c][0], Hs[0], yq, ws)
        us_kv = per_call_us(body_kv, 1, nrep=20)
        us_q = per_call_us(body_q, 1, nrep=20)
        kvl[m] = {"us_per_call": round(us_kv, 2), "plain_fused_us_per_call": round(us_q, 2)}
    out["wqkv_kv_rows_6144x4096"] = kvl

    # batched decode: B stacked rows, each weight read once per batch
    batch = {}
    for m in ("i8", "i8x2", "f32"):
        batch[m] = {}
        for B in ((1, 2, 4, 8, 12, 16, 32, 64) if m != "f32" else (1, 2, 4, 8, 16)):
            acts = []
            for p, (_, n, k) in enumerate(synth.LAYER_D4096):
                h = torch.from_numpy(synth.activations(rng, B, k)).to(dev)
                xq, xd = native.activation_buffers(m, B, k, device=dev)
                native.act_quant(m, h, xq, xd, norm=True)
                acts.append((xq, xd, torch.empty((B, n), dtype=torch.float32, device=dev)))

            def body(c, m=m, B=B, acts=acts):
                for p in range(4):
                    xq, xd, y = acts[p]
                    native.q8_proj(m, Q[c][p], S[c][p], xq, xd, B, y)
            us = per_call_us(body, 1)
            batch[m][str(B)] = {"us_per_layer": round(us, 2),
                                "GB/s": round(LAYER_BYTES / (us * 1e-6) / 1e9, 1),
                                "rows_per_s": round(B * 4 / (us * 1e-6), 1)}
    out["batched_decode_d4096"] = batch

    # prefill chunks: T rows, producer (RMSNorm -> quant) then the chunk projection
    chunk = {}
    flops_row = 2.0 * sum(n * k for _, n, k in synth.LAYER_D4096)
    for m in ("i8", "i8x2"):
        chunk[m] = {}
        for T in (2, 4, 8, 16, 32, 64, 128, 256):
            bufs = []
            for p, (_, n, k) in enumerate(synth.LAYER_D4096):
                h = torch.from_numpy(synth.activations(rng, T, k)).to(dev)
                xq, xd = native.activation_buffers(m, T, k, device=dev)
                bufs.append((h, xq, xd, torch.empty((T, n), dtype=torch.float32, device=dev)))

            def body(c, m=m, T=T, bufs=bufs):
                for p in range(4):
                    h, xq, xd, y = bufs[p]
                    native.act_quant(m, h, xq, xd, norm=True)
                    native.q8_proj_chunk(m, Q[c][p], S[c][p], xq, xd, T, y)
            us = per_call_us(body, 1)
            chunk[m][str(T)] = {"us_per_layer": round(us, 2),
                                "GB/s": round(LAYER_BYTES / (us * 1e-6) / 1e9, 1),
                                "tokens_per_s": round(T / (us * 1e-6), 1),
                                "TFLOP/s": round(flops_row * T / (us * 1e-6) / 1e12, 1)}
            if T == 256:
                # end to end: each layer step copies its T x K inputs in from
                # pinned host memory and its T x N outputs back
                h_host = [bufs[p][0].cpu().pin_memory() for p in range(4)]
                y_host = [torch.empty(bufs[p][3].shape, dtype=torch.float32).pin_memory() for p in range(4)]

                def body_e2e(c, m=m, T=T, bufs=bufs, h_host=h_host, y_host=y_host):
                    for p in range(4):
                        h, xq, xd, y = bufs[p]
                        h.copy_(h_host[p], non_blocking=True)
                        native.act_quant(m, h, xq, xd, norm=True)
                        native.q8_proj_chunk(m, Q[c][p], S[c][p], xq, xd, T, y)
                        y_host[p].copy_(y, non_blocking=True)
                ue = e2e_us(torch, dev, capture, body_e2e)
                chunk[m][str(T)]["e2e"] = {
                    "us_per_layer": round(ue, 2), "tokens_per_s": round(T / (ue * 1e-6), 1),
                    "h2d_bytes_per_step": sum(int(x.numel()) * 4 for x in h_host),
                    "d2h_bytes_per_step": sum(int(x.numel()) * 4 for x in y_host),
                    "note": "host wall clock: one captured layer step with the inputs copied in "
                            "from pinned host memory and the outputs copied back, then stream sync"}
                if oracle_slices and m == "i8":
                    # the oracle (RMSNorm, quantisation, projection) on 32 output
                    # rows of each matrix, scaled to the matrix's N
                    tot = 0.0
                    for p, (nm, n, k) in enumerate(synth.LAYER_D4096):
                        hp = bufs[p][0].cpu().numpy()
                        qs_, ss_ = mats[p][1][:32], mats[p][2][:32]
                        t_us = oracle_slice_us(lambda: orc.project(m, qs_, ss_, orc.quantize(m, orc.rmsnorm(hp)[0])))
                        tot += t_us * n / 32
                    chunk[m][str(T)]["cpu_oracle"] = {
                        "us_per_layer": round(tot, 1), "tokens_per_s": round(T / (tot * 1e-6), 2),
                        "cores": orc.threads(), "arch": platform.machine(),
                        "sample": "32 output rows of each matrix at T = 256, timed on the host "
                                  "(best of 3) and scaled linearly to the matrix's rows"}
    out["prefill_chunk_d4096"] = chunk

    # LM head 128256 x 4096 with planted rows, fused arg-max
    nh, kh = synth.HEAD_SHAPE
    qh, sh, hh16, pos = synth.planted_head(4, nh, kh, 16)
    QH = [torch.from_numpy(qh).to(dev)]
    SH = [torch.from_numpy(sh.view(np.int16)).to(dev)]
    QH.append(QH[0].clone())
    SH.append(SH[0].clone())
    head = {}
    for m in ("i8", "f32"):
        head[m] = {}
        for rows in (1, 16):
            h = torch.from_numpy(np.ascontiguousarray(hh16[:rows])).to(dev)
            xq, xd = native.activation_buffers(m, rows, kh, device=dev)
            native.act_quant(m, h, xq, xd, norm=True)
            tok = torch.empty(rows, dtype=torch.int32, device=dev)
            ws = native.argmax_workspace(rows, device=dev)

            def body(c, m=m, rows=rows, xq=xq, xd=xd, tok=tok, ws=ws):
                native.head_argmax(m, QH[c], SH[c], xq, xd, rows, tok, ws)
            us = per_call_us(body, 1)
            ok = bool(np.array_equal(tok.cpu().numpy(), pos[np.arange(rows) % 8]))
            head[m][str(rows)] = {"us": round(us, 2),
                                  "GB/s": round(weight_bytes(nh, kh) / (us * 1e-6) / 1e9, 1),
                                  "tokens_per_s": round(rows / (us * 1e-6), 1),
                                  "argmax_matches_planted": ok}
            if rows == 16:
                # end to end: the hidden rows in from pinned host memory, the
                # producer, the head with its arg-max, the tokens back
                h_host = h.cpu().pin_memory()
                tok_host = torch.empty(rows, dtype=torch.int32).pin_memory()

                def body_e2e(c, m=m, rows=rows, h=h, xq=xq, xd=xd, tok=tok, ws=ws, h_host=h_host,
                             tok_host=tok_host):
                    h.copy_(h_host, non_blocking=True)
                    native.act_quant(m, h, xq, xd, norm=True)
                    native.head_argmax(m, QH[c], SH[c], xq, xd, rows, tok, ws)
                    tok_host.copy_(tok, non_blocking=True)
                ue = e2e_us(torch, dev, capture, body_e2e)
                head[m][str(rows)]["e2e"] = {
                    "us": round(ue, 2), "tokens_per_s": round(rows / (ue * 1e-6), 1),
                    "h2d_bytes_per_step": int(h_host.numel()) * 4, "d2h_bytes_per_step": rows * 4,
                    "note": "host wall clock: hidden rows in, RMSNorm -> quant, head + arg-max, "
                            "tokens out, then stream sync"}
                if oracle_slices:
                    act_h = orc.quantize(m, orc.rmsnorm(h.cpu().numpy())[0])
                    t_us = oracle_slice_us(lambda: orc.project(m, qh[:512], sh[:512], act_h)) * nh / 512
                    head[m][str(rows)]["cpu_oracle"] = {
                        "us": round(t_us, 1), "tokens_per_s": round(rows / (t_us * 1e-6), 2),
                        "cores": orc.threads(), "arch": platform.machine(),
                        "sample": "512 of the 128256 head rows, 16 activation rows, timed on the "
                                  "host (best of 3) and scaled linearly to the whole head"}
    out["lm_head_128256x4096"] = head
    del QH, SH
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweeps", action="store_true",
                    help="skip the other workload configurations")
    ap.add_argument("--quick", action="store_true",
                    help="warm-up and timed steps only (for launch lists under a profiler)")
    ap.add_argument("--case", default=None,
                    help="MODE:PROJ[:fused] (PROJ a matrix of the layer or 'all'), "
                         "chunk:MODE:PROJ:T or head:MODE:ROWS -- only those launches, "
                         "warmup+steps eager launches each (a case for a profiler capture)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
