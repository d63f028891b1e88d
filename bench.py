"""Benchmark of the HiMuon hot path on B300: one fused optimizer step (momentum,
tiled Newton-Schulz with T = 128 and K = 5, weight update) over the 2-D weights
of a Llama-3-8B-shaped model (32 layers x {Q, O 4096^2; K, V 1024 x 4096; gate,
up 14336 x 4096; down 4096 x 14336}: 224 matrices, 6.98 G parameters), with
synthetic low-rank-plus-noise gradients resident in HBM.

Prints one JSON line. ``value`` is the algorithmic NS throughput of the whole job
(6 H W T K flops per matrix per step, summed, over the step time), in TFLOP/s;
``ms_per_step`` is the optimizer-step time. ``--impl reference`` times the fp64
CPU oracle on a bounded sample of the same workload instead.

Launch: ``python bench.py [--gpus 1 --steps K --warmup W]``; for N > 1 under
``torch.distributed.run`` every rank runs the full layer set on its own GPU
(independent replicas, weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import json
import math
import os
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

WORKLOADS = {
    # name: (shapes fn, rank of the synthetic gradients, T, K, chunk bytes)
    "llama3_8b": ("llama3_8b_shapes", 16, 128, 5, 8 << 30),
    "gpt2_small": ("gpt2_small_shapes", 8, 128, 5, 0),
}


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


# ---------------------------------------------------------------- measurement helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


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
    return sum(6.0 * H * W * T * K for H, W in shapes)


def cpu_oracle_rate(shapes, T, K, budget_s: float, max_tiles: int | None = None):
    """Times the fp64 oracle's fused step on whole sample matrices of the
    workload until ``budget_s`` seconds of CPU work have run. Returns
    (flops/s, description, threads)."""
    import numpy as np
    import torch

    import oracle
    from tiled_newton_schulz_03_b300 import synth

    try:
        from threadpoolctl import threadpool_info
        threads = max((i.get("num_threads", 1) for i in threadpool_info()), default=os.cpu_count())
    except Exception:
        threads = os.cpu_count()
    # sample: the K-projection shape (1024 x 4096), or a row band of a matrix
    H, W = min(shapes, key=lambda s: s[0] * s[1])
    rows = H
    if max_tiles is not None:
        rows = max(T, min(H, (max_tiles // max(1, math.ceil(W / T))) * T))
    done_flops, spent, n = 0.0, 0.0, 0
    while spent < budget_s or n == 0:
        G = synth.lowrank_noise(rows, W, seed=900 + n, rank=16).double().numpy()
        Wt = synth.gaussian(rows, W, seed=950 + n, std=0.02).double().numpy()
        M = np.zeros((rows, W))
        t0 = time.perf_counter()
        oracle.himuon_step(Wt, G, M, T, K, lr=0.02, mu=0.95)
        spent += time.perf_counter() - t0
        done_flops += 6.0 * rows * W * T * K
        n += 1
        if max_tiles is not None:
            break
    del torch
    desc = (f"{n} x fused step of one {rows}x{W} matrix ({rows * W // (T * T)} tiles of "
            f"T={T}, K={K}) in fp64, {spent:.1f} s")
    return done_flops / spent, desc, threads, spent


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
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12

    # roofline of the fused step kernel: its launches are back to back on the
    # stream and make up the step; achieved = step flops / step time.
    launches_per_step = launches / args.steps
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained") or FALLBACK_PEAKS["bf16_tflops_sustained"])
    achieved = flops / (statistics.median(step_ms) * 1e-3) / 1e12
    traffic_info = ncu_traffic(kernel_source_hash())
    traffic = None
    if traffic_info and traffic_info.get("workload") == args.workload:
        traffic = traffic_info.get("dram_bytes_per_launch")
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_kind": f"bf16_tflops_sustained ({peak_src})",
                "frac_of_burst": round(achieved / float(peaks.get("bf16_tflops") or 1800.0), 4),
                "kernel": KERNEL + "<step>", "launches_per_step": launches_per_step,
                "hbm_bytes_per_step_algorithmic": nparams * (2 + 8 + 4),
                "hbm_frac_of_step": round(nparams * 14 / (statistics.median(step_ms) * 1e-3) /
                                          (float(peaks.get("hbm_gbs") or 6400.0) * 1e9), 4)}

    # end to end through the public API: G from pinned host memory, step, W back
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(hm, handle, Gs, Ws, Ms, shapes, T, K, chunk, flops, stream, args, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, threads, _ = cpu_oracle_rate(shapes, T, K, args.cpu_seconds)
        cpu = {"value": round(rate / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": desc, "ms_per_step_extrapolated": round(flops / rate * 1e3, 1)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded low-rank + noise gradients, N(0,0.02^2) weights, zero momentum)",
        "config": {"workload": f"{args.workload}: {len(shapes)} matrices, {nparams / 1e9:.2f} G params, "
                               f"T={T}, K={K}, fused momentum(0.95, Nesterov) + update(lr 0.02)",
                   "T": T, "K": K, "matrices": len(shapes), "params": nparams,
                   "chunk_bytes": chunk, "grad_dtype": "bf16", "weight_dtype": "bf16",
                   "momentum_dtype": "fp32", "l2": "inputs larger than L2 (G+M+W = "
                   f"{nparams * 14 / 1e9:.0f} GB per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "step_ms": {"median": round(statistics.median(step_ms), 3), "min": round(min(step_ms), 3),
                    "max": round(max(step_ms), 3)},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(launches), "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    handle.close()


def run_e2e(hm, handle, Gs, Ws, Ms, shapes, T, K, chunk, flops, stream, args, world, dev):
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

    def e2e_step():
        for h, g in zip(hG, Gs):
            g.copy_(h, non_blocking=True)
        hm.step(Ws, Gs, Ms, T, K, lr=0.02, mu=0.95, nesterov=True, chunk_bytes=chunk,
                handle=handle, stream=stream)
        for h, w in zip(hW, Ws):
            h.copy_(w, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    dist_barrier(world)
    t0 = time.perf_counter()
    for _ in range(n):
        e2e_step()
    torch.cuda.synchronize()
    dt = dist_max(time.perf_counter() - t0, world, dev)
    return {"value": round(world * flops * n / dt / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(dt / n * 1e3, 2), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n}


# ---------------------------------------------------------------- reference arm: the oracle

def run_reference(args):
    rank, world, _ = env_int("RANK", 0), env_int("WORLD_SIZE", 1), env_int("LOCAL_RANK", 0)
    if rank != 0:
        return
    shapes, grank, T, K, chunk = workload_shapes(args.workload)
    flops = step_flops(shapes, T, K)
    nparams = sum(H * W for H, W in shapes)
    # each step: the oracle's fused step on a bounded sample (a row band of
    # the smallest matrix shape, <= 64 tiles); warm-up steps untimed.
    for _ in range(args.warmup):
        cpu_oracle_rate(shapes, T, K, 0.0, max_tiles=16)
    rates, spent, desc, threads = [], 0.0, "", 1
    for _ in range(args.steps):
        r, desc, threads, s = cpu_oracle_rate(shapes, T, K, 0.0, max_tiles=64)
        rates.append(r)
        spent += s
    rate = len(rates) / sum(1.0 / r for r in rates)    # total flops / total time
    value = rate / 1e12
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(flops / rate * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded low-rank + noise gradients)",
        "config": {"workload": f"{args.workload}: {len(shapes)} matrices, {nparams / 1e9:.2f} G params, "
                               f"T={T}, K={K}, fused momentum(0.95, Nesterov) + update(lr 0.02)",
                   "T": T, "K": K, "matrices": len(shapes), "params": nparams,
                   "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}; ms_per_step extrapolated to the full "
                                   f"workload by flops ({spent:.1f} s total)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- secondary workloads

def _timed(fn, reps, flush, stream):
    """Median CUDA-event time (ms) of fn over reps runs, L2 flushed before each."""
    import torch
    times = []
    for _ in range(reps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    return statistics.median(times)


def run_sweep(args):
    """Tile-size sweep on one 4096 x 4096 bf16 matrix (rank-8 + noise), K = 5:
    tiled NS only, one JSON line per T (T = 4096 is the full-matrix map). The
    matrix fits in L2, so L2 is flushed (a 256 MB write) before every run."""
    import torch

    import tiled_newton_schulz_03_b300 as hm
    from tiled_newton_schulz_03_b300 import build as hbuild, synth
    hbuild.build()
    dev = torch.device("cuda", 0)
    handle = hm.Handle(dev)
    stream = torch.cuda.current_stream(dev)
    G = synth.lowrank_noise(4096, 4096, seed=3, rank=8, device=dev)
    out = torch.empty_like(G)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    peaks, src = load_peaks()
    for T in (32, 64, 128, 256, 4096):
        fn = lambda: hm.tiled_ns(G, T, 5, out=out, handle=handle, stream=stream)
        for _ in range(args.warmup):
            fn()
        ms = _timed(fn, args.steps, flush, stream)
        flops = 6.0 * 4096 * 4096 * min(T, 4096) * 5
        tf = flops / (ms * 1e-3) / 1e12
        hbm_ms = 4.0 * 4096 * 4096 / (float(peaks.get("hbm_gbs", 6400.0)) * 1e9) * 1e3
        print(json.dumps({"workload": "sweep4096", "T": T, "K": 5, "ms": round(ms, 4),
                          "tflops": round(tf, 2), "frac_of_burst_bf16": round(tf / float(peaks.get("bf16_tflops", 1800.0)), 4),
                          "roofline_ms": round(max(flops / (float(peaks.get("bf16_tflops", 1800.0)) * 1e12) * 1e3, hbm_ms), 4),
                          "peak_source": src}), flush=True)
    assert hm.device_error(handle=handle) == 0
    handle.close()


def run_ragged(args):
    """Ragged shapes and the runtime tile schedule: 1000x3000, 5120x13824 and
    2048x50257 bf16 (rank-8 + noise), three successive fused steps with T = 64,
    128, 256, for K = 3 and 5; one JSON line per (K, step)."""
    import torch

    import tiled_newton_schulz_03_b300 as hm
    from tiled_newton_schulz_03_b300 import build as hbuild, synth
    hbuild.build()
    dev = torch.device("cuda", 0)
    handle = hm.Handle(dev)
    stream = torch.cuda.current_stream(dev)
    shapes = [(1000, 3000), (5120, 13824), (2048, 50257)]
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
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
            ms = _timed(fn, args.steps, flush, stream)
            hm.step(Ws, Gs, Ms, T, K, lr=0.02, mu=0.95, handle=handle, stream=stream)
            flops = sum(6.0 * H * W * T * K for H, W in shapes)
            print(json.dumps({"workload": "ragged", "K": K, "step": step, "T": T, "ms": round(ms, 4),
                              "tflops": round(flops / (ms * 1e-3) / 1e12, 2)}), flush=True)
    assert hm.device_error(handle=handle) == 0
    handle.close()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["sweep4096", "ragged"],
                    default="llama3_8b",
                    help="llama3_8b (headline) or gpt2_small: the fused step, one JSON line; "
                         "sweep4096 / ragged: secondary per-configuration timings")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.workload == "sweep4096" and args.impl == "ours":
        run_sweep(args)
    elif args.workload == "ragged" and args.impl == "ours":
        run_ragged(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
