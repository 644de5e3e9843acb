"""Benchmark of the KDA prefill chunk solver on GB300.

One step = one call of the solver (every chunk-head of one batch: task decode,
tile loads, the four diagonal inverses, the merge and the stores; on the split
path also the workspace round trip) on the packed workload of 16 requests x
512 tokens, 64 heads, fp32 in and out (the 8192-token x 64-head solve the
metric is quoted on).  Inputs are synthetic (seeded KDA-style A).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  N > 1 runs one independent replica per GPU
(no collective on the data path); the value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import kda_inputs as ki  # noqa: E402

METRIC = "solve ms & achieved HBM GB/s (vs ~8 TB/s) at 8192 tok x 64 heads, 1 GB300"
WORKLOAD = "packed_16x512_h64_f32"
FALLBACK_HBM_GBS = 6800.0
DTYPE_NAME = {"f32": "f32", "bf16": "bf16", "f16": "f16"}
ELT = {"f32": 4, "bf16": 2, "f16": 2}


# ------------------------------------------------------------ byte models
def sector_read_bytes(n: int, elt: int) -> int:
    """Bytes of 32-byte sectors covering the strictly lower part of an n-row chunk."""
    return sum(-(-(i * elt) // 32) * 32 for i in range(n))


def algorithmic_bytes(inp: ki.SolverInput, in_elt: int, out_elt: int) -> int:
    """Minimum HBM bytes of one solve: the strictly lower part of A (sector granular)
    plus the full output rows (incl. the structural zeros and ones)."""
    per_n = {}
    tot = 0
    for _, n in inp.chunks():
        if n not in per_n:
            per_n[n] = sector_read_bytes(n, in_elt) + n * 64 * out_elt
        tot += per_n[n]
    return tot * inp.H


def full_tensor_bytes(inp: ki.SolverInput, in_elt: int, out_elt: int) -> int:
    return inp.A.numel() * (in_elt + out_elt)


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        # one-second timestamp resolution: keep samples within the timed window +- 1 s
        sel = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0] or rows
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in sel:
            for name, v in zip(names[1:], r[3][1:]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": sorted(reasons), "samples": len(sel)}


# -------------------------------------------------------------- peaks etc.
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_chunked_02_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it was
    taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
    except (OSError, ValueError):
        return None
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ ranks
def dist_setup(nccl: bool):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if nccl else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(ms_local: float, bytes_per_rank: int, world: int, device) -> tuple:
    """Weak scaling over independent replicas: every rank solves its own copy of the
    workload; the job takes as long as the slowest rank.  Returns (ms, GB/s of the
    whole job)."""
    ms = max_over_ranks(ms_local, world, device)
    return ms, world * bytes_per_rank / (ms / 1e3) / 1e9


# ------------------------------------------------------------- CPU oracle
def time_oracle(inp: ki.SolverInput, seconds: float, alg_bytes: int, max_reps: int = 10 ** 9):
    import oracle
    orc = oracle.get()
    A64 = oracle.to_f64(inp.A)
    cu = inp.cu_seqlens.numpy() if inp.cu_seqlens is not None else None
    reps = 0
    t0 = time.perf_counter()
    while True:
        orc.solve_tril(A64, cu)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= max_reps:
            break
    return alg_bytes * reps / el / 1e9, reps, el, orc.num_threads()


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores: the reference arm."""
    if rank != 0:
        return
    wl = ki.WORKLOADS[args.workload]
    inp = ki.build(wl)
    ine, oute = ELT[wl.in_dtype], ELT[wl.out_dtype]
    alg = algorithmic_bytes(inp, ine, oute)
    import oracle
    orc = oracle.get()
    A64 = oracle.to_f64(inp.A)
    cu = inp.cu_seqlens.numpy() if inp.cu_seqlens is not None else None
    for _ in range(args.warmup):
        orc.solve_tril(A64, cu)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.solve_tril(A64, cu)
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    v = alg / (ms / 1e3) / 1e9
    sample = f"the full workload ({len(inp.chunks()) * inp.H} chunk-heads) per step, fp64 oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(inp, "oracle (CPU)"),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(inp: ki.SolverInput, path: str):
    wl = inp.workload
    return {"workload": wl.name, "layout": wl.layout, "tokens": inp.B * inp.T,
            "requests": len(inp.seqlens), "heads": inp.H, "in_dtype": wl.in_dtype,
            "out_dtype": wl.out_dtype, "path": path,
            "l2": "input+output %.0f MB > 129 MB L2; no flush between steps"
                  % (full_tensor_bytes(inp, ELT[wl.in_dtype], ELT[wl.out_dtype]) / 1e6)}


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import linear_attention_chunked_02_gb300 as kda
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = ki.WORKLOADS[args.workload]
    inp = ki.build(wl)
    in_dtype, out_dtype = ki.torch_dtype(wl.in_dtype), ki.torch_dtype(wl.out_dtype)
    ine, oute = ELT[wl.in_dtype], ELT[wl.out_dtype]
    A = inp.A.to(dev)
    cu = inp.cu_seqlens.to(dev) if inp.cu_seqlens is not None else None
    nseq = 0 if cu is None else cu.numel() - 1
    out = torch.empty(A.shape, dtype=out_dtype, device=dev)
    need = kda.workspace_size(inp.B, inp.T, inp.H, nseq)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return kda.solve_tril(A, cu, out_dtype=out_dtype, path=args.path, out=out, workspace=ws,
                              stream=stream, return_path=True)

    _, taken = step()
    launches_per_step = 2 if taken == "split" else 1
    alg = algorithmic_bytes(inp, ine, oute)
    full = full_tensor_bytes(inp, ine, oute)

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier(world)
    ms, value = whole_job_gbs(ev0.elapsed_time(ev1) / args.steps, alg, world, dev)
    if rank == 0:
        sampler.stop()
        clocks = sampler.summary(t0, t1)

    # end to end: pinned host buffers, copies inside the timed region (C-ABI host entry)
    A_host = inp.A.pin_memory()
    cu_host = inp.cu_seqlens.pin_memory() if inp.cu_seqlens is not None else None
    Ai_host = torch.empty(A.shape, dtype=out_dtype).pin_memory()
    cu_dev = torch.empty_like(cu) if cu is not None else None
    A_dev = torch.empty_like(A)
    e2e_steps = max(3, min(args.steps, 200))
    for _ in range(2):
        kda.solve_tril_host(A_host, Ai_host, A_dev, out, cu_host, cu_dev, ws, stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        kda.solve_tril_host(A_host, Ai_host, A_dev, out, cu_host, cu_dev, ws, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms, e2e_value = whole_job_gbs(e0.elapsed_time(e1) / e2e_steps, alg, world, dev)

    if rank != 0:
        return
    peak, peak_kind = hbm_peak()
    kernel = "kda_tril_kernel<MODE_FUSED>" if taken == "single" else "kda_tril_kernel<MODE_MERGE>"
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.in_dtype, "data": "synthetic",
        "config": config_dict(inp, taken),
        "effective_gbs": full / (ms / 1e3) / 1e9,
        "chunk_heads_per_s": len(inp.chunks()) * inp.H / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": ncu_traffic(kernel, wl.name), "kernel": kernel,
                     "algorithmic_bytes_per_launch": alg},
        "e2e": {"value": e2e_value, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": inp.A.numel() * ine + (0 if cu is None else cu.numel() * 4),
                "d2h_bytes_per_step": inp.A.numel() * oute},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        v, reps, el, cores = time_oracle(inp, args.cpu_seconds, alg)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": f"{reps} solves of the full workload in {el:.1f} s"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(ki.WORKLOADS))
    ap.add_argument("--path", default="auto", choices=["auto", "single", "split"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        world, rank, _ = dist_setup(nccl=False)
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(nccl=True)
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
