"""Benchmark of the HiMuon hot path on B300: one fused optimizer step (momentum,
tiled Newton-Schulz with T = 128 and K = 5, weight update) over the 2-D weights
of a Llama-3-8B-shaped model (32 layers x {Q, O 4096^2; K, V 1024 x 4096; gate,
up 14336 x 4096; down 4096 x 14336}: 224 matrices, 6.98 G parameters), with
synthetic low-rank-plus-noise gradients resident in HBM.

Prints one JSON line. ``value`` is the algorithmic NS throughput of the whole job
(6 H W T K flops per matrix per step, summed, over the step time), in TFLOP/s;
``ms_per_step`` is the optimizer-step time. ``roofline`` compares the step with
the slower of its tensor time (6 H W T K at the bf16 dense peak) and its HBM
time (the bytes of G, M and W read and written once at the measured copy
bandwidth). ``secondary`` holds the other workloads measured in the same run
(GPT-2-small set, 4096^2 tile-size sweep, ragged shapes with the runtime tile
schedule), each with its own roofline, clocks and CPU baseline.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload instead.

Launch: ``python bench.py [--gpus N --steps K --warmup W]``. With N > 1 and no
torchrun environment the script starts N ranks itself through
``torch.distributed.run``; every rank runs the full layer set on its own GPU
(independent replicas, weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "HiMuon step ms & tiled-NS TFLOP/s vs bf16 tensor peak (8B layer set, T=128, K=5)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL = "ns_tc_kernel"

# Fused step bytes per parameter: G bf16 read (2), M fp32 read + write (8),
# W bf16 read + write (4).
STEP_BYTES_PER_PARAM = 14

WORKLOADS = {
    # name: (shapes fn, rank of the synthetic gradients, T, K, chunk bytes)
    "llama3_8b": ("llama3_8b_shapes", 16, 128, 5, 8 << 30),
    "gpt2_small": ("gpt2_small_shapes", 8, 128, 5, 0),
}

# The CPU baseline's sample, the same in both arms: one fused step of the
# oracle on one K-projection-shaped matrix (1024 x 4096, 256 tiles of T = 128).
CPU_SAMPLE_SHAPE = (1024, 4096)


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


# ---------------------------------------------------------------- distributed helpers

def dist_setup():
    """(rank, world, local_rank) from the torchrun environment; initialises the
    process group when world > 1 (nccl on GPUs, gloo otherwise)."""
    rank, world, local = env_int("RANK", 0), env_int("WORLD_SIZE", 1), env_int("LOCAL_RANK", 0)
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(x: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def relaunch_command(argv, nproc: int, port: int):
    """The torchrun command line that starts ``nproc`` ranks of this script."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={nproc}", "--master-addr=127.0.0.1", f"--master-port={port}",
            os.path.abspath(__file__), *argv]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


# ---------------------------------------------------------------- measurement helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def roofline(flops: float, nbytes: float, seconds: float, peaks, peak_src: str) -> dict:
    """Roofline of a measured region: the slower of the tensor time (flops at
    the burst bf16 peak) and the HBM time (bytes at the copy bandwidth) sets
    the bound; ``frac`` = that time / the measured time."""
    p_tc = float(peaks.get("bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"])
    p_hbm = float(peaks.get("hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"])
    t_tc = flops / (p_tc * 1e12)
    t_hbm = nbytes / (p_hbm * 1e9)
    if t_tc >= t_hbm:
        r = {"bound": "tensor", "achieved": round(flops / seconds / 1e12, 2), "peak": p_tc,
             "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": round(nbytes / seconds / 1e9, 1), "peak": p_hbm,
             "unit": "GB/s"}
    r["frac"] = round(r["achieved"] / r["peak"], 4)
    r["roofline_ms"] = round(max(t_tc, t_hbm) * 1e3, 4)
    r["tensor_ms"] = round(t_tc * 1e3, 4)
    r["hbm_ms"] = round(t_hbm * 1e3, 4)
    r["algorithmic_flops"] = flops
    r["algorithmic_bytes"] = nbytes
    r["peak_source"] = f"{peak_src}: bf16_tflops (burst) and hbm_gbs of MEASURED_PEAKS.json"
    return r


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def ncu_traffic(kernel_src_hash: str):
    """Per-launch DRAM bytes of the timed kernel from the committed ncu summary,
    if it was taken on the current kernel source (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
        if d.get("source_sha256") == kernel_src_hash:
            return d
    except Exception:
        pass
    return None


# The files the timed kernel and its launch plan are built from: a change to
# any of them makes the committed DRAM counters stale; a change elsewhere (the
# GEMM path, the fp32 path) does not.
KERNEL_SOURCES = ("tiled_newton_schulz_03_b300/csrc/api.cu",
                  "tiled_newton_schulz_03_b300/csrc/common.cuh",
                  "tiled_newton_schulz_03_b300/csrc/kernels.h",
                  "tiled_newton_schulz_03_b300/csrc/ns_tc.cu",
                  "tiled_newton_schulz_03_b300/csrc/ptx.cuh",
                  "tiled_newton_schulz_03_b300/csrc/tile_util.cuh",
                  "include/himuon.h")


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode() + f.read())
    return h.hexdigest()


# ---------------------------------------------------------------- workload

def workload_shapes(name):
    from tiled_newton_schulz_03_b300 import synth
    fn, rank, T, K, chunk = WORKLOADS[name]
    return getattr(synth, fn)(), rank, T, K, chunk


def step_flops(shapes, T, K):
    return sum(6.0 * H * W * min(T, max(H, W)) * K for H, W in shapes)


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 1) for i in threadpool_info()), default=os.cpu_count())
    except Exception:
        return os.cpu_count()


def cpu_oracle_step(H, W, T, K, seed, rank=16):
    """One fused step of the fp64 oracle on one seeded H x W matrix; returns
    (seconds, flops)."""
    import numpy as np

    import oracle
    from tiled_newton_schulz_03_b300 import synth

    G = synth.lowrank_noise(H, W, seed=seed, rank=rank).double().numpy()
    Wt = synth.gaussian(H, W, seed=seed + 50, std=0.02).double().numpy()
    M = np.zeros((H, W))
    t0 = time.perf_counter()
    oracle.himuon_step(Wt, G, M, T, K, lr=0.02, mu=0.95)
    return time.perf_counter() - t0, 6.0 * H * W * min(T, max(H, W)) * K


def cpu_oracle_ns(H, W, T, K, seed, rank=8):
    """The oracle's tiled NS map (or, for T >= max(H, W), the full-matrix map)
    on one seeded H x W matrix; returns (seconds, flops)."""
    import oracle
    from tiled_newton_schulz_03_b300 import synth

    G = synth.lowrank_noise(H, W, seed=seed, rank=rank).double().numpy()
    t0 = time.perf_counter()
    if T >= max(H, W):
        oracle.full_ns(G, K)
    else:
        oracle.tiled_ns(G, T, K)
    return time.perf_counter() - t0, 6.0 * H * W * min(T, max(H, W)) * K


def cpu_baseline(fn, budget_s: float, desc: str, min_runs: int = 1):
    """Repeats ``fn(i) -> (seconds, flops)`` until budget_s of CPU work has run."""
    spent, flops, n = 0.0, 0.0, 0
    while n < min_runs or spent < budget_s:
        s, f = fn(n)
        spent += s
        flops += f
        n += 1
    return {"value": round(flops / spent / 1e12, 6), "unit": UNIT, "cores": oracle_threads(),
            "kind": "oracle", "sample": f"{n} x {desc} in fp64 ({spent:.1f} s)"}, flops / spent


def headline_cpu_sample(i, T=128, K=5):
    H, W = CPU_SAMPLE_SHAPE
    return cpu_oracle_step(H, W, T, K, seed=900 + i)


# ---------------------------------------------------------------- our implementation

def run_ours(args):
    import torch

    import tiled_newton_schulz_03_b300 as hm
    from tiled_newton_schulz_03_b300 import build as hbuild, synth

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbuild.build()
    hm.load_library()
    handle = hm.Handle(dev)

    shapes, grank, T, K, chunk = workload_shapes(args.workload)
    flops = step_flops(shapes, T, K)
    nparams = sum(H * W for H, W in shapes)
    nbytes = nparams * STEP_BYTES_PER_PARAM

    # inputs resident in HBM: G bf16 (low-rank + noise), W bf16 ~ N(0, 0.02^2), M fp32 = 0
    Gs = [synth.lowrank_noise(H, W, seed=1000 * rank + i, rank=grank, device=dev)
          for i, (H, W) in enumerate(shapes)]
    Ws = [synth.gaussian(H, W, seed=500000 + i, std=0.02, dtype=torch.bfloat16, device=dev)
          for i, (H, W) in enumerate(shapes)]
    Ms = [torch.zeros(H, W, dtype=torch.float32, device=dev) for H, W in shapes]
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    def one_step():
        hm.step(Ws, Gs, Ms, T, K, lr=0.02, mu=0.95, nesterov=True, chunk_bytes=chunk,
                handle=handle, stream=stream)

    if args.mode == "sharded":
        # strong scaling: each rank steps the matrices it owns (balanced by NS
        # work) and the owners broadcast the new weights to every rank
        from tiled_newton_schulz_03_b300 import shard
        sharded = shard.ShardedStep(shapes, T, K, lambda W, G, M: hm.step(
            W, G, M, T, K, lr=0.02, mu=0.95, nesterov=True, chunk_bytes=chunk, handle=handle,
            stream=stream))

        def one_step():                       # noqa: F811
            sharded(Ws, Gs, Ms)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if hm.device_error(handle=handle) != 0:
        raise RuntimeError("device error during warm-up")

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local) as clk:
        dist_barrier(world)
        torch.cuda.synchronize()
        l0 = handle.launch_count()
        ev[0].record(stream)
        for i in range(args.steps):
            one_step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        dist_barrier(world)
        launches = handle.launch_count() - l0
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    total_ms = dist_max(total_ms, world, dev)
    if hm.device_error(handle=handle) != 0:
        raise RuntimeError("device error during the timed region")
    ms_per_step = total_ms / args.steps
    jobs = 1 if args.mode == "sharded" else world   # layer sets stepped per step, all ranks
    value = jobs * flops * args.steps / (total_ms * 1e-3) / 1e12

    # Roofline of the fused step kernel. Its launches run back to back on the
    # stream and are the whole step (ncu launch list), so the average launch
    # duration is the step time / launches per step, and per launch the
    # algorithmic work is the step's / launches per step: the ratio is the same.
    launches_per_step = launches / args.steps
    peaks, peak_src = load_peaks()
    med_s = statistics.median(step_ms) * 1e-3
    roof = roofline(flops, nbytes, med_s, peaks, peak_src)
    traffic_info = ncu_traffic(kernel_source_hash())
    traffic = None
    if traffic_info and traffic_info.get("workload") == args.workload:
        traffic = traffic_info.get("dram_bytes_per_launch")
    roof.update({
        "traffic": traffic, "kernel": KERNEL + "<128, step>",
        "launches_per_step": launches_per_step,
        "launch_ms_avg": round(statistics.median(step_ms) / max(launches_per_step, 1), 3),
        "algorithmic_bytes_per_launch": nbytes / max(launches_per_step, 1),
        "bytes_per_param": STEP_BYTES_PER_PARAM,
        "hbm_frac": round(roof["hbm_ms"] / (med_s * 1e3), 4),
        "tensor_frac": round(roof["tensor_ms"] / (med_s * 1e3), 4),
        "tensor_frac_of_sustained_peak": round(
            flops / med_s / 1e12 / float(peaks.get("bf16_tflops_sustained") or 1400.0), 4),
        "sustained_peak_note": "bf16_tflops_sustained was taken at a median SM clock of "
                               f"{peaks.get('clocks_under_load', {}).get('sm_mhz_median')} MHz "
                               "(cuBLAS under the power cap); reported for context only",
    })

    # end to end through the public API: G from pinned host memory, step, W back
    e2e = None
    if not args.no_e2e and args.mode == "replicas":
        e2e = run_e2e(hm, handle, Gs, Ws, Ms, shapes, T, K, chunk, flops, stream, args, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        H, W = CPU_SAMPLE_SHAPE
        cpu, rate = cpu_baseline(headline_cpu_sample, args.cpu_seconds,
                                 f"fused step of one {H}x{W} matrix ({H * W // (T * T)} tiles of "
                                 f"T={T}, K={K})")
        cpu["ms_per_step_extrapolated_full_workload"] = round(flops / rate * 1e3, 1)

    secondary = None
    if rank == 0 and world == 1 and args.secondary and args.workload == "llama3_8b":
        del Gs, Ws, Ms
        torch.cuda.empty_cache()
        secondary = run_secondary(hm, handle, dev, stream, peaks, peak_src, args)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "strong" if args.mode == "sharded" else "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded low-rank + noise gradients, N(0,0.02^2) weights, zero momentum)",
        "config": {"workload": f"{args.workload}: {len(shapes)} matrices, {nparams / 1e9:.2f} G params, "
                               f"T={T}, K={K}, fused momentum(0.95, Nesterov) + update(lr 0.02)",
                   "T": T, "K": K, "matrices": len(shapes), "params": nparams,
                   "chunk_bytes": chunk, "grad_dtype": "bf16", "weight_dtype": "bf16",
                   "momentum_dtype": "fp32", "l2": "inputs larger than L2 (G+M+W = "
                   f"{nbytes / 1e9:.0f} GB per step)",
                   "parallelism": (f"{args.mode} x{world}" if world > 1 else "single GPU")},
        "step_ms": {"median": round(statistics.median(step_ms), 3), "min": round(min(step_ms), 3),
                    "max": round(max(step_ms), 3)},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(launches), "clocks": clk.summary(),
    }
    if secondary is not None:
        line["secondary"] = secondary
    if rank == 0:
        print(json.dumps(line), flush=True)
    handle.close()


def run_e2e(hm, handle, Gs, Ws, Ms, shapes, T, K, chunk, flops, stream, args, world, dev):
    """The same step through the public API with the gradients coming from, and
    the weights going back to, pinned host memory every step. Layers are
    pipelined: layer l's gradients go up on one copy stream while layer l-1 is
    stepped on the compute stream and layer l-2's weights come down on another
    copy stream (events order each layer's copy, step and read-back)."""
    import torch
    try:
        hG = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in Gs]
        hW = [torch.empty(w.shape, dtype=w.dtype, pin_memory=True) for w in Ws]
    except Exception as exc:  # pinned memory exhausted on this host
        return {"value": None, "unit": UNIT, "error": f"pinned host buffers: {exc}"[:200]}
    for h, g in zip(hG, Gs):
        h.copy_(g)
    h2d = sum(g.numel() * g.element_size() for g in Gs)
    d2h = sum(w.numel() * w.element_size() for w in Ws)
    n = max(1, args.e2e_steps)
    per = max(1, len(Gs) // 32)           # one group per layer of the layer set
    groups = [list(range(i, min(len(Gs), i + per))) for i in range(0, len(Gs), per)]
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)

    def e2e_step():
        uploaded = []
        for gi, idx in enumerate(groups):
            with torch.cuda.stream(up):
                for i in idx:
                    Gs[i].copy_(hG[i], non_blocking=True)
                e = torch.cuda.Event()
                e.record(up)
            uploaded.append(e)
        stepped = []
        for gi, idx in enumerate(groups):
            stream.wait_event(uploaded[gi])
            hm.step([Ws[i] for i in idx], [Gs[i] for i in idx], [Ms[i] for i in idx], T, K,
                    lr=0.02, mu=0.95, nesterov=True, chunk_bytes=chunk, handle=handle,
                    stream=stream)
            e = torch.cuda.Event()
            e.record(stream)
            stepped.append(e)
        for gi, idx in enumerate(groups):
            down.wait_event(stepped[gi])
            with torch.cuda.stream(down):
                for i in idx:
                    hW[i].copy_(Ws[i], non_blocking=True)
        # the next step's uploads overwrite G: they wait for this step's kernels
        up.wait_event(stepped[-1])

    def copies_only():
        # the same copies on the same streams with no compute between them: the
        # floor the pipelined step can reach over this host link
        for idx in groups:
            with torch.cuda.stream(up):
                for i in idx:
                    Gs[i].copy_(hG[i], non_blocking=True)
            with torch.cuda.stream(down):
                for i in idx:
                    hW[i].copy_(Ws[i], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    dist_barrier(world)
    t0 = time.perf_counter()
    for _ in range(n):
        e2e_step()
    torch.cuda.synchronize()
    dt = dist_max(time.perf_counter() - t0, world, dev)
    copies_only()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    copies_only()
    torch.cuda.synchronize()
    floor = time.perf_counter() - t1
    return {"value": round(world * flops * n / dt / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(dt / n * 1e3, 2), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n,
            "pipeline": f"{len(groups)} layer groups; H2D, step and D2H on three streams",
            "copies_alone_ms": round(floor * 1e3, 2),
            "copies_alone_gbs_each_way": round(h2d / floor / 1e9, 1)}


# ---------------------------------------------------------------- secondary workloads

def _timed_b2b(fn, reps, stream):
    """CUDA-event times (ms) of fn over reps runs issued back to back (inputs
    larger than L2; the host work of one call overlaps the GPU work of the
    previous one, as in a training loop)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record(stream)
    for i in range(reps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]


def _timed(fn, reps, stream, flush=None):
    """CUDA-event times (ms) of fn over reps runs; L2 flushed before each when
    the inputs would fit in it."""
    import torch
    times = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    return times


def run_secondary(hm, handle, dev, stream, peaks, peak_src, args,
                  groups=("gpt2_small", "sweep4096", "ragged")):
    """Configs measured besides the headline: the GPT-2-small fused step, the
    4096 x 4096 tile-size sweep (tiled NS only) and the ragged set with the
    runtime tile schedule. Each entry carries its roofline, the clocks seen
    while it ran, its kernel launches and an oracle CPU baseline on a sample."""
    import torch
    out = []
    fns = {"gpt2_small": _sec_gpt2, "sweep4096": _sec_sweep, "ragged": _sec_ragged}
    for g in groups:
        out += fns[g](hm, handle, dev, stream, peaks, peak_src, args)
        torch.cuda.empty_cache()
    assert hm.device_error(handle=handle) == 0
    return out


def _sec_gpt2(hm, handle, dev, stream, peaks, peak_src, args):
    """GPT-2-small set, fused step, T = 128, K = 5."""
    import torch

    from tiled_newton_schulz_03_b300 import synth
    reps, cpu_s = max(5, args.secondary_reps), args.secondary_cpu_seconds
    shapes = synth.gpt2_small_shapes()
    Ws = [synth.gaussian(H, W, seed=10 + i, std=0.02, dtype=torch.bfloat16, device=dev) for i, (H, W) in enumerate(shapes)]
    Gs = [synth.lowrank_noise(H, W, seed=1 + 100 * i, rank=8, device=dev) for i, (H, W) in enumerate(shapes)]
    Ms = [torch.zeros(H, W, device=dev) for H, W in shapes]
    fn = lambda: hm.step(Ws, Gs, Ms, 128, 5, lr=0.02, mu=0.95, handle=handle, stream=stream)
    for _ in range(args.warmup):
        fn()
    with ClockSampler(dev.index) as clk:
        l0 = handle.launch_count()
        times = _timed_b2b(fn, reps * 8, stream)
        launches = handle.launch_count() - l0
    ms = statistics.median(times)
    # host time to issue one step call (72 matrices; tensor maps and the
    # descriptor image come from the handle's cache after the first call)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(20):
        fn()
    host_us = (time.perf_counter() - t0) / 20 * 1e6
    torch.cuda.synchronize()
    nparams = sum(H * W for H, W in shapes)
    flops = step_flops(shapes, 128, 5)
    cpu, _ = cpu_baseline(lambda i: cpu_oracle_step(768, 768, 128, 5, seed=40 + i, rank=8), cpu_s,
                          "fused step of one 768x768 matrix (36 tiles of T=128, K=5)")
    return [{"workload": f"gpt2_small: {len(shapes)} matrices, {nparams / 1e6:.1f} M params, "
                         "T=128, K=5, fused momentum(0.95, Nesterov) + update(lr 0.02)",
             "ms_per_step": round(ms, 4), "value": round(flops / (ms * 1e-3) / 1e12, 2),
             "unit": UNIT, "l2": f"inputs larger than L2 ({nparams * 14 / 1e9:.2f} GB per step); "
                                 "steps back to back",
             "roofline": roofline(flops, nparams * STEP_BYTES_PER_PARAM, ms * 1e-3, peaks, peak_src),
             "gpu_launches_per_run": launches / len(times), "clocks": clk.summary(),
             "host_us_per_call": round(host_us, 1), "cpu_baseline": cpu}]


def _sec_sweep(hm, handle, dev, stream, peaks, peak_src, args):
    """4096 x 4096 sweep, tiled NS only (bf16 in and out), K = 5."""
    import torch

    from tiled_newton_schulz_03_b300 import synth
    reps, cpu_s = max(5, args.secondary_reps), args.secondary_cpu_seconds
    out = []
    G = synth.lowrank_noise(4096, 4096, seed=3, rank=8, device=dev)
    o = torch.empty_like(G)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)   # 256 MB > L2
    for T in (32, 64, 128, 256, 4096):
        fn = lambda: hm.tiled_ns(G, T, 5, out=o, handle=handle, stream=stream)
        for _ in range(args.warmup):
            fn()
        with ClockSampler(dev.index) as clk:
            l0 = handle.launch_count()
            times = _timed(fn, reps * 4, stream, flush)
            launches = handle.launch_count() - l0
        ms = statistics.median(times)
        flops = 6.0 * 4096 * 4096 * min(T, 4096) * 5
        Hs = 1024 if T == 4096 else 512
        cpu, _ = cpu_baseline(lambda i: cpu_oracle_ns(Hs, 4096 if T != 4096 else Hs, T, 5, seed=70 + i),
                              cpu_s, (f"full-matrix map of one {Hs}x{Hs} matrix" if T == 4096 else
                                      f"tiled map of a {Hs}x4096 row band (T={T})") + ", K=5")
        out.append({"workload": f"sweep4096: one 4096x4096 bf16 matrix, T={T}, K=5, tiled NS "
                                "(bf16 out)" + (" = full-matrix map" if T == 4096 else ""),
                    "T": T, "ms_per_step": round(ms, 4), "value": round(flops / (ms * 1e-3) / 1e12, 2),
                    "unit": UNIT, "l2": "flushed before every run (256 MB write)",
                    "roofline": roofline(flops, 4.0 * 4096 * 4096, ms * 1e-3, peaks, peak_src),
                    "gpu_launches_per_run": launches / len(times), "clocks": clk.summary(),
                    "cpu_baseline": cpu})
    return out


def _sec_ragged(hm, handle, dev, stream, peaks, peak_src, args):
    """Ragged set, three fused steps with T = 64 -> 128 -> 256, K = 3 and 5."""
    import torch

    from tiled_newton_schulz_03_b300 import synth
    reps, cpu_s = max(5, args.secondary_reps), args.secondary_cpu_seconds
    out = []
    shapes = [(1000, 3000), (5120, 13824), (2048, 50257)]
    nparams = sum(H * W for H, W in shapes)
    sched = hm.TSchedule([(0, 64), (1, 128), (2, 256)])
    for K in (3, 5):
        Ws = [synth.gaussian(H, W, seed=10 + i, std=0.02, dtype=torch.bfloat16, device=dev) for i, (H, W) in enumerate(shapes)]
        Ms = [torch.zeros(H, W, device=dev) for H, W in shapes]
        for step in range(3):
            Gs = [synth.lowrank_noise(H, W, seed=100 * step + i, rank=8, device=dev) for i, (H, W) in enumerate(shapes)]
            T = sched(step)
            # time copies of the state, so that every timed run does the same step
            Wc = [w.clone() for w in Ws]
            Mc = [m.clone() for m in Ms]
            fn = lambda: hm.step(Wc, Gs, Mc, T, K, lr=0.02, mu=0.95, handle=handle, stream=stream)
            for _ in range(args.warmup):
                fn()
            with ClockSampler(dev.index) as clk:
                l0 = handle.launch_count()
                times = _timed_b2b(fn, reps, stream)
                launches = handle.launch_count() - l0
            hm.step(Ws, Gs, Ms, T, K, lr=0.02, mu=0.95, handle=handle, stream=stream)
            ms = statistics.median(times)
            flops = step_flops(shapes, T, K)
            cpu, _ = cpu_baseline(lambda i: cpu_oracle_step(256, 3000, T, K, seed=80 + i, rank=8),
                                  cpu_s / 2, f"fused step of a 256x3000 row band (T={T}, K={K})")
            out.append({"workload": f"ragged: 1000x3000, 5120x13824, 2048x50257 bf16, step {step} of the "
                                    f"T schedule 64->128->256, T={T}, K={K}, fused step",
                        "T": T, "K": K, "step": step, "ms_per_step": round(ms, 4),
                        "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
                        "l2": f"inputs larger than L2 ({nparams * 14 / 1e9:.2f} GB per step); "
                              "steps back to back",
                        "roofline": roofline(flops, nparams * STEP_BYTES_PER_PARAM, ms * 1e-3, peaks,
                                             peak_src),
                        "gpu_launches_per_run": launches / len(times), "clocks": clk.summary(),
                        "cpu_baseline": cpu})
            del Wc, Mc, Gs
        del Ws, Ms
    return out


# ---------------------------------------------------------------- reference arm: the oracle

def run_reference(args):
    rank, world = env_int("RANK", 0), env_int("WORLD_SIZE", 1)
    if rank != 0:
        return
    shapes, grank, T, K, chunk = workload_shapes(args.workload)
    flops = step_flops(shapes, T, K)
    nparams = sum(H * W for H, W in shapes)
    H, W = CPU_SAMPLE_SHAPE
    # each step: the oracle's fused step on the bounded sample (the same sample
    # as the GPU arm's cpu_baseline); warm-up steps untimed
    for i in range(args.warmup):
        headline_cpu_sample(i, T, K)
    secs, done = [], 0.0
    for i in range(args.steps):
        s, f = headline_cpu_sample(i, T, K)
        secs.append(s)
        done += f
    rate = done / sum(secs)
    value = rate / 1e12
    sample = (f"per step: fused step of one {H}x{W} matrix ({H * W // (T * T)} tiles of T={T}, "
              f"K={K}) in fp64; {args.steps} steps, {sum(secs):.1f} s")
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(secs) * 1e3, 1),
        "ms_per_step_measures": f"the bounded sample ({H}x{W}, one of the workload's 224 matrices)",
        "ms_per_step_extrapolated_full_workload": round(flops / rate * 1e3, 1),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded low-rank + noise gradients)",
        "config": {"workload": f"{args.workload}: {len(shapes)} matrices, {nparams / 1e9:.2f} G params, "
                               f"T={T}, K={K}, fused momentum(0.95, Nesterov) + update(lr 0.02)",
                   "T": T, "K": K, "matrices": len(shapes), "params": nparams,
                   "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- stand-alone sweeps

def run_sweep(args):
    """One secondary workload alone (``--workload sweep4096`` or ``ragged``):
    the same entries as in the headline line's ``secondary``, one JSON line
    each."""
    import torch

    import tiled_newton_schulz_03_b300 as hm
    from tiled_newton_schulz_03_b300 import build as hbuild
    hbuild.build()
    dev = torch.device("cuda", 0)
    handle = hm.Handle(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, src = load_peaks()
    args.secondary_cpu_seconds = 0.0
    for e in run_secondary(hm, handle, dev, stream, peaks, src, args, groups=(args.workload,)):
        print(json.dumps(e), flush=True)
    handle.close()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["sweep4096", "ragged"],
                    default="llama3_8b",
                    help="llama3_8b (headline) or gpt2_small: the fused step, one JSON line; "
                         "sweep4096 / ragged: the secondary entries alone, one line each")
    ap.add_argument("--mode", choices=["replicas", "sharded"], default="replicas",
                    help="N > 1: replicas (every rank steps the whole layer set; weak scaling) or "
                         "sharded (each rank steps its share, owners broadcast W; strong scaling)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-secondary", dest="secondary", action="store_false",
                    help="skip the secondary workloads after the headline")
    ap.add_argument("--secondary-reps", type=int, default=10)
    ap.add_argument("--secondary-cpu-seconds", type=float, default=2.0)
    args = ap.parse_args()

    world = env_int("WORLD_SIZE", 0)
    if args.gpus > 1 and world == 0:
        # not under torchrun: start one rank per GPU and pass the exit code on
        cmd = relaunch_command(sys.argv[1:], args.gpus, _free_port())
        sys.exit(subprocess.call(cmd))
    if world and args.gpus != world:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; running WORLD_SIZE ranks",
              file=sys.stderr)

    if args.workload in ("sweep4096", "ragged") and args.impl == "ours":
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
