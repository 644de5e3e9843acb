"""Benchmark of the KDA prefill chunk solver on GB300.

One step = one call of the solver (every chunk-head of one batch: task decode,
tile loads, the four diagonal inverses, the merge and the stores; on the split
path also the workspace round trip) on the packed workload of 16 requests x
512 tokens, 64 heads, fp32 in and out (the 8192-token x 64-head solve the
metric is quoted on).  Inputs are synthetic (seeded KDA-style A).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--bt 16|32|64]

``--bt`` times the solver's 16- or 32-token branch on the workload's shape.

Prints one JSON line (rank 0).  N > 1 runs one independent replica per GPU
(no collective on the data path); the value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_inputs as ki  # noqa: E402

METRIC = "solve ms & achieved HBM GB/s (vs ~8 TB/s) at 8192 tok x 64 heads, 1 GB300"
WORKLOAD = "packed_16x512_h64_f32"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10 ** 6
KERNEL = {64: "kda_tril_kernel<MODE_FUSED>", 32: "kda_bt32_kernel", 16: "kda_bt16_kernel"}
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
            per_n[n] = sector_read_bytes(n, in_elt) + n * inp.bt * out_elt
        tot += per_n[n]
    return tot * inp.H


def full_tensor_bytes(inp: ki.SolverInput, in_elt: int, out_elt: int) -> int:
    return inp.A.numel() * (in_elt + out_elt)


# ----------------------------------------------------------------- clocks
def parse_smi_time(text: str) -> float:
    """Seconds since the epoch of an nvidia-smi timestamp ("2026/12/03 09:40:26.123", local time)."""
    whole, _, frac = text.strip().partition(".")
    return time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + (float("0." + frac) if frac.isdigit() else 0.0)


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
                rows.append((parse_smi_time(parts[0]), float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        # the samples taken during the timed region; if it was too short to hold
        # three, the window is widened (and says so)
        window = "timed region"
        sel = [r for r in rows if t0 <= r[0] <= t1]
        if len(sel) < 3:
            window = "timed region +- 0.25 s"
            sel = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in sel:
            for name, v in zip(names[1:], r[3][1:]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": sorted(reasons), "samples": len(sel), "window": window}


# -------------------------------------------------------------- peaks etc.
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# sources that define each kernel family and its launch
_COMMON_SOURCES = ["kda_kernels.cuh", "kda_launch.cuh", "kda_api.cu", "kda_inst_f32.cu",
                   "kda_inst_bf16.cu", "kda_inst_f16.cu"]
KERNEL_SOURCES = {"kda_tril_kernel": _COMMON_SOURCES, "kda_bt": _COMMON_SOURCES + ["kda_small.cuh"],
                  "kda_kgb": _COMMON_SOURCES + ["kda_small.cuh", "kda_kgb.cuh"]}
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed: what a traffic
    capture depends on."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str) -> str:
    files = next(v for k, v in KERNEL_SOURCES.items() if kernel.startswith(k))
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_chunked_02_gb300", "csrc")
    for f in files:
        h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


ROTATE_MIN_BYTES = 16 << 20


def l2_policy(inp: ki.SolverInput):
    """How steps stay out of L2: ("none", 1) when the footprint is at least twice the
    L2; ("rotate", R) from 16 MiB up: R copies of the input and output, step i using
    copy i % R, so that a copy is R - 1 >= 2 L2 / footprint solves old when it is used
    again and the steps run back to back; ("flush", 1) below 16 MiB: a 256 MB write
    between steps, each step timed alone."""
    wl = inp.workload
    fp = full_tensor_bytes(inp, ELT[wl.in_dtype], ELT[wl.out_dtype])
    if fp >= 2 * L2_BYTES:
        return "none", 1
    if fp >= ROTATE_MIN_BYTES:
        return "rotate", -(-2 * L2_BYTES // fp) + 1
    return "flush", 1


def flushes_l2(inp: ki.SolverInput) -> bool:
    return l2_policy(inp)[0] == "flush"


def workload_key(wl: ki.Workload) -> str:
    return wl.name if wl.bt == 64 else f"{wl.name}_bt{wl.bt}"


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it was
    taken on the current kernel sources."""
    try:
        d = json.load(open(TRAFFIC_JSON))
    except (OSError, ValueError):
        return None
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


_UNIT = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}


def record_traffic(csv_path: str, workload: str, kernel: str, command: str) -> dict:
    """Store the per-launch DRAM bytes of the launches captured in an ncu --csv log
    (metrics dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum)
    under (workload, kernel): the mean over the captured launches.  Captured as
    consecutive launches with --cache-control none, each launch's write figure
    includes the previous launch's output lines that it evicts from L2, so in the
    steady state the mean is the whole per-launch traffic."""
    import csv
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    vals = {}
    for r in csv.DictReader(lines):
        name = r.get("Metric Name")
        if name in ("dram__bytes_read.sum", "dram__bytes_write.sum", "gpu__time_duration.sum"):
            v = float(r["Metric Value"].replace(",", ""))
            vals.setdefault(r["ID"], {})[name] = v * _UNIT.get(r.get("Metric Unit", "byte"), 1.0)
    if not vals:
        raise ValueError(f"no captured launch in {csv_path}")
    n = len(vals)
    mean = {k: sum(v[k] for v in vals.values()) / n
            for k in ("dram__bytes_read.sum", "dram__bytes_write.sum", "gpu__time_duration.sum")}
    rd, wr, ns = mean["dram__bytes_read.sum"], mean["dram__bytes_write.sum"], mean["gpu__time_duration.sum"]
    entry = {"source_hash": kernel_source_hash(kernel),
             "dram_bytes_per_launch": int(rd + wr), "dram_read": int(rd), "dram_write": int(wr),
             "launches": n, "ncu_us_per_launch": ns / 1e3,
             "physical_gbs": (rd + wr) / ns,
             "note": f"mean over {n} consecutive launches: {command}"}
    try:
        d = json.load(open(TRAFFIC_JSON))
    except (OSError, ValueError):
        d = {}
    d.setdefault(workload, {})[kernel] = entry
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(d, f, indent=1)
        f.write("\n")
    return entry


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


REFERENCE_BUDGET_S = 90.0       # timed seconds the reference arm aims for at any --steps


def sample_input(inp: ki.SolverInput, units: int, heads: int) -> ki.SolverInput:
    """The first `units` requests (packed) or batch rows (dense) of `inp`, first `heads` heads."""
    if inp.cu_seqlens is None:
        return ki.SolverInput(inp.workload, inp.A[:units, :, :heads].contiguous(), None, inp.seqlens[:units])
    cu = inp.cu_seqlens[:units + 1].clone()
    rows = int(cu[-1])
    return ki.SolverInput(inp.workload, inp.A[:, :rows, :heads].contiguous(), cu, inp.seqlens[:units])


def reference_sample(full, steps: int, time_of):
    """(units, heads) of the sample a reference step solves: the full workload, or
    halved (heads first, then requests or batch rows) while `steps` solves of it
    would take more than REFERENCE_BUDGET_S.  time_of(units, heads) times one solve
    of a candidate; halving stops early once it no longer pays (a solve's fixed
    cost dominates), so the sample stays as large as that allows."""
    units = full.B if full.cu_seqlens is None else len(full.seqlens)
    heads = full.H
    t = time_of(units, heads)
    while steps * t > REFERENCE_BUDGET_S and (heads > 1 or units > 1):
        nu, nh = (units, heads // 2) if heads > 1 else (units // 2, heads)
        nt = time_of(nu, nh)
        if nt > 0.75 * t:
            break
        units, heads, t = nu, nh, nt
    return units, heads


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores: the reference arm.  Each step
    solves a bounded sample of the workload (all of it when --steps allows), sized
    so that the timed steps take about REFERENCE_BUDGET_S."""
    if rank != 0:
        return
    wl = ki.WORKLOADS[args.workload].with_(bt=args.bt)
    full = ki.build(wl)
    ine, oute = ELT[wl.in_dtype], ELT[wl.out_dtype]
    import oracle
    orc = oracle.get()
    cu_of = lambda x: x.cu_seqlens.numpy() if x.cu_seqlens is not None else None

    def time_of(units, heads):
        x = sample_input(full, units, heads)
        A64, cu = oracle.to_f64(x.A), cu_of(x)
        t0 = time.perf_counter()
        orc.solve_tril(A64, cu)
        return time.perf_counter() - t0

    units, heads = reference_sample(full, args.steps, time_of)
    inp = sample_input(full, units, heads)
    alg = algorithmic_bytes(inp, ine, oute)
    A64 = oracle.to_f64(inp.A)
    cu = cu_of(inp)
    for _ in range(args.warmup):
        orc.solve_tril(A64, cu)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.solve_tril(A64, cu)
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    v = alg / (ms / 1e3) / 1e9
    what = "requests" if full.cu_seqlens is not None else "batch rows"
    sample = (f"{len(inp.chunks()) * inp.H} of the workload's {len(full.chunks()) * full.H} chunk-heads per step "
              f"(the first {units} {what}, first {heads} of {full.H} heads), fp64 oracle")
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
    mb = full_tensor_bytes(inp, ELT[wl.in_dtype], ELT[wl.out_dtype]) / 1e6
    kind, r = l2_policy(inp)
    l2 = {"flush": f"input+output {mb:.0f} MB < 2 x 129 MB L2: 256 MB written between steps, each step timed alone",
          "rotate": f"input+output {mb:.0f} MB x {r} copies used in turn ({mb * r:.0f} MB > 2 x 129 MB L2), "
                    "back to back",
          "none": f"input+output {mb:.0f} MB > 129 MB L2; no flush between steps"}[kind]
    return {"workload": workload_key(wl), "layout": wl.layout, "tokens": inp.B * inp.T,
            "requests": len(inp.seqlens), "heads": inp.H, "chunk": wl.bt, "in_dtype": wl.in_dtype,
            "out_dtype": wl.out_dtype, "path": path, "l2": l2}


# ---------------------------------------------------------------- our arm
def timed_calls(n, run, stream, dev, flush):
    """Device ms of n calls of run(): one event pair around all of them, or, with
    an L2 flush buffer, one pair per call with the flush outside it."""
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for e0, e1 in pairs:
        flush.zero_()
        e0.record(stream)
        run()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return sum(e0.elapsed_time(e1) for e0, e1 in pairs)


# ------------------------------------------- fused construction + solve (kgb)
KGB_KERNEL = "kda_kgb_kernel"


def kgb_bytes(x: ki.KgbInput, in_elt: int, out_elt: int) -> int:
    """Minimum HBM bytes of one fused solve: every row's keys, decays and beta, and
    the chunks' output rows."""
    rows = x.B * x.T
    return rows * x.H * (x.K * in_elt + x.K * 4 + in_elt) + sum(n for _, n in x.chunks()) * x.H * 64 * out_elt


def kgb_config(x: ki.KgbInput):
    wl = x.workload
    mb = kgb_bytes(x, ELT[wl.in_dtype], ELT[wl.out_dtype]) / 1e6
    return {"workload": f"{wl.name}_kgb", "layout": wl.layout, "tokens": x.B * x.T, "requests": len(x.seqlens),
            "heads": x.H, "key_dim": x.K, "chunk": 64, "in_dtype": wl.in_dtype, "out_dtype": wl.out_dtype,
            "op": "chunk matrix from k, g, beta fused with the solve",
            "l2": f"inputs+output {mb:.0f} MB > 129 MB L2; no flush between steps"}


def time_oracle_kgb(x: ki.KgbInput, seconds: float, alg_bytes: int):
    import oracle
    orc = oracle.get()
    k, g, b = (oracle.to_f64(t) for t in (x.k, x.g, x.beta))
    cu = x.cu_seqlens.numpy() if x.cu_seqlens is not None else None
    reps = 0
    t0 = time.perf_counter()
    while True:
        orc.solve_kgb(k, g, b, cu)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return alg_bytes * reps / el / 1e9, reps, el, orc.num_threads()


def run_ours_kgb(args, world, rank, local):
    import linear_attention_chunked_02_gb300 as kda
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = ki.WORKLOADS[args.workload]
    x = ki.build_kgb(wl)
    out_dtype = ki.torch_dtype(wl.out_dtype)
    ine, oute = ELT[wl.in_dtype], ELT[wl.out_dtype]
    k, g, b = x.k.to(dev), x.g.to(dev), x.beta.to(dev)
    cu = x.cu_seqlens.to(dev) if x.cu_seqlens is not None else None
    out = torch.empty((x.B, x.T, x.H, 64), dtype=out_dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.solve_tril_kgb(k, g, b, cu, out_dtype=out_dtype, out=out, stream=stream)

    alg = kgb_bytes(x, ine, oute)
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.time()
    total = timed_calls(args.steps, step, stream, dev, None)
    t1 = time.time()
    barrier(world)
    ms, value = whole_job_gbs(total / args.steps, alg, world, dev)
    if rank == 0:
        sampler.stop()
        clocks = sampler.summary(t0, t1)

    # end to end: pinned host inputs copied in and the output copied back every step
    hk, hg, hb = x.k.pin_memory(), x.g.pin_memory(), x.beta.pin_memory()
    hcu = x.cu_seqlens.pin_memory() if x.cu_seqlens is not None else None
    hout = torch.empty(out.shape, dtype=out_dtype).pin_memory()
    dk, dg, db = torch.empty_like(k), torch.empty_like(g), torch.empty_like(b)
    dcu = torch.empty_like(cu) if cu is not None else None

    def e2e_step():
        with torch.cuda.stream(stream):
            dk.copy_(hk, non_blocking=True)
            dg.copy_(hg, non_blocking=True)
            db.copy_(hb, non_blocking=True)
            if dcu is not None:
                dcu.copy_(hcu, non_blocking=True)
            kda.solve_tril_kgb(dk, dg, db, dcu, out_dtype=out_dtype, out=out, stream=stream)
            hout.copy_(out, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 100))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms, e2e_value = whole_job_gbs(timed_calls(e2e_steps, e2e_step, stream, dev, None) / e2e_steps, alg,
                                      world, dev)
    if rank != 0:
        return
    peak, peak_kind = hbm_peak()
    achieved = alg / (ms / 1e3) / 1e9
    key = f"{wl.name}_kgb"
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.in_dtype, "data": "synthetic", "config": kgb_config(x),
        "chunk_heads_per_s": len(x.chunks()) * x.H / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": ncu_traffic(KGB_KERNEL, key), "kernel": KGB_KERNEL,
                     "algorithmic_bytes_per_launch": alg},
        "e2e": {"value": e2e_value, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": x.k.numel() * ine + x.g.numel() * 4 + x.beta.numel() * ine
                + (0 if cu is None else cu.numel() * 4),
                "d2h_bytes_per_step": out.numel() * oute},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        v, reps, el, cores = time_oracle_kgb(x, args.cpu_seconds, alg)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": f"{reps} solves of the full workload in {el:.1f} s"}
    print(json.dumps(line), flush=True)


def sample_kgb(x: ki.KgbInput, units: int, heads: int) -> ki.KgbInput:
    """The first `units` requests (packed) or batch rows (dense) of `x`, first `heads` heads."""
    if x.cu_seqlens is None:
        cut = lambda t: t[:units, :, :heads].contiguous()
        return ki.KgbInput(x.workload, cut(x.k), cut(x.g), cut(x.beta), None, x.seqlens[:units])
    cu = x.cu_seqlens[:units + 1].clone()
    rows = int(cu[-1])
    cut = lambda t: t[:, :rows, :heads].contiguous()
    return ki.KgbInput(x.workload, cut(x.k), cut(x.g), cut(x.beta), cu, x.seqlens[:units])


def run_reference_kgb(args, world, rank):
    """The oracle of the fused path, as it stands, on the host cores, on a bounded
    sample per step (as run_reference)."""
    if rank != 0:
        return
    wl = ki.WORKLOADS[args.workload]
    full = ki.build_kgb(wl)
    import oracle
    orc = oracle.get()
    f64 = lambda y: [oracle.to_f64(t) for t in (y.k, y.g, y.beta)]
    cu_of = lambda y: y.cu_seqlens.numpy() if y.cu_seqlens is not None else None

    def time_of(units, heads):
        y = sample_kgb(full, units, heads)
        args_, cu = f64(y), cu_of(y)
        t0 = time.perf_counter()
        orc.solve_kgb(*args_, cu)
        return time.perf_counter() - t0

    units, heads = reference_sample(full, args.steps, time_of)
    x = sample_kgb(full, units, heads)
    alg = kgb_bytes(x, ELT[wl.in_dtype], ELT[wl.out_dtype])
    k, g, b = f64(x)
    cu = cu_of(x)
    for _ in range(args.warmup):
        orc.solve_kgb(k, g, b, cu)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.solve_kgb(k, g, b, cu)
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    v = alg / (ms / 1e3) / 1e9
    what = "requests" if full.cu_seqlens is not None else "batch rows"
    sample = (f"{len(x.chunks()) * x.H} of the workload's {len(full.chunks()) * full.H} chunk-heads per step "
              f"(the first {units} {what}, first {heads} of {full.H} heads), fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": kgb_config(full),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def copy_probe(nbytes: int = 134217728) -> dict:
    """Pinned host <-> device copy rates of one GPU: each direction alone and both at
    once on two streams (the floor of the end-to-end leg, which moves A in and Ai out)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, reps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def both():
        cur = torch.cuda.current_stream()
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)
        cur.wait_stream(s1)
        cur.wait_stream(s2)

    h2d = timed(lambda: d_in.copy_(h_in, non_blocking=True))
    d2h = timed(lambda: h_out.copy_(d_out, non_blocking=True))
    bi = timed(both)
    return {"bytes_each_way": nbytes, "h2d_ms": h2d, "h2d_gbs": nbytes / h2d / 1e6, "d2h_ms": d2h,
            "d2h_gbs": nbytes / d2h / 1e6, "both_ms": bi, "both_gbs_total": 2 * nbytes / bi / 1e6}


def run_ours(args, world, rank, local):
    import linear_attention_chunked_02_gb300 as kda
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = ki.WORKLOADS[args.workload].with_(bt=args.bt)
    inp = ki.build(wl)
    in_dtype, out_dtype = ki.torch_dtype(wl.in_dtype), ki.torch_dtype(wl.out_dtype)
    ine, oute = ELT[wl.in_dtype], ELT[wl.out_dtype]
    A = inp.A.to(dev)
    cu = inp.cu_seqlens.to(dev) if inp.cu_seqlens is not None else None
    nseq = 0 if cu is None else cu.numel() - 1
    out = torch.empty(A.shape, dtype=out_dtype, device=dev)
    need = kda.workspace_size(inp.B, inp.T, inp.H, nseq) if wl.bt == 64 else 0
    tf32 = args.precision == "tf32"
    if tf32 and (wl.bt != 64 or args.path == "split"):
        raise SystemExit("--precision tf32 is the 64-token single pass")
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev) if wl.bt == 64 and not tf32 else None
    stream = torch.cuda.current_stream(dev)
    kind, copies = l2_policy(inp)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if kind == "flush" else None
    As = [A] + [A.clone() for _ in range(copies - 1)]
    outs = [out] + [torch.empty_like(out) for _ in range(copies - 1)]
    turn = [0]

    def step():
        i = turn[0] % copies
        turn[0] += 1
        return kda.solve_tril(As[i], cu, out_dtype=out_dtype, path=args.path, out=outs[i], workspace=ws,
                              stream=stream, return_path=True, precision=args.precision)

    def timed_steps(n, run):
        return timed_calls(n, run, stream, dev, flush)

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
    t0 = time.time()
    total_ms = timed_steps(args.steps, step)
    t1 = time.time()
    barrier(world)
    ms, value = whole_job_gbs(total_ms / args.steps, alg, world, dev)
    if rank == 0:
        sampler.stop()
        clocks = sampler.summary(t0, t1)

    # end to end: pinned host buffers, copies inside the timed region (the C-ABI host
    # entry for 64-token chunks; copies on the stream around solve_tril otherwise)
    A_host = inp.A.pin_memory()
    cu_host = inp.cu_seqlens.pin_memory() if inp.cu_seqlens is not None else None
    Ai_host = torch.empty(A.shape, dtype=out_dtype).pin_memory()
    cu_dev = torch.empty_like(cu) if cu is not None else None
    A_dev = torch.empty_like(A)

    def e2e_step():
        if wl.bt == 64 and not tf32:
            kda.solve_tril_host(A_host, Ai_host, A_dev, out, cu_host, cu_dev, ws, stream)
            return
        with torch.cuda.stream(stream):
            A_dev.copy_(A_host, non_blocking=True)
            if cu_dev is not None:
                cu_dev.copy_(cu_host, non_blocking=True)
            kda.solve_tril(A_dev, cu_dev, out_dtype=out_dtype, out=out, stream=stream, precision=args.precision)
            Ai_host.copy_(out, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 200))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_total = timed_steps(e2e_steps, e2e_step)
    barrier(world)
    e2e_ms, e2e_value = whole_job_gbs(e2e_total / e2e_steps, alg, world, dev)

    if rank != 0:
        return
    peak, peak_kind = hbm_peak()
    kernel = KERNEL[wl.bt] if taken == "single" else "kda_tril_kernel<MODE_MERGE>"
    if tf32:
        kernel = "kda_tril_kernel<MODE_FUSED, TF32>"
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.in_dtype, "data": "synthetic",
        "config": dict(config_dict(inp, taken), **({"precision": "tf32"} if tf32 else {})),
        "effective_gbs": full / (ms / 1e3) / 1e9,
        "chunk_heads_per_s": len(inp.chunks()) * inp.H / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": ncu_traffic(kernel, workload_key(wl)), "kernel": kernel,
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
    # 20000 steps: the 8192-token solve's timed region lasts about 0.8 s, so the
    # 50 ms clock samples fall inside it
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(ki.WORKLOADS))
    ap.add_argument("--path", default="auto", choices=["auto", "single", "split"])
    ap.add_argument("--precision", default="ieee", choices=["ieee", "tf32"],
                    help="tf32: the 64-token single pass with plain TF32 merge products")
    ap.add_argument("--bt", type=int, default=64, choices=[16, 32, 64],
                    help="chunk length (16 and 32: the solver's shorter branches)")
    ap.add_argument("--op", default="solve", choices=["solve", "kgb"],
                    help="kgb: the chunk matrix built from keys, decays and betas (128 channels) "
                         "fused with the 64-token solve")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="store the DRAM traffic of the launch captured in this ncu --csv log "
                         "for --workload/--bt in profiles/traffic.json, then exit")
    ap.add_argument("--ncu-command", default="", help="the command the capture ran (recorded)")
    ap.add_argument("--copy-probe", action="store_true",
                    help="print pinned host <-> device copy rates (the end-to-end floor) and exit")
    args = ap.parse_args()
    if args.copy_probe:
        print(json.dumps(copy_probe()))
        return
    if args.record_traffic:
        wl = ki.WORKLOADS[args.workload].with_(bt=args.bt)
        key, kernel = ((f"{wl.name}_kgb", KGB_KERNEL) if args.op == "kgb" else (workload_key(wl), KERNEL[args.bt]))
        print(json.dumps(record_traffic(args.record_traffic, key, kernel, args.ncu_command)))
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        world, rank, _ = dist_setup(nccl=False)
        (run_reference_kgb if args.op == "kgb" else run_reference)(args, world, rank)
        return
    world, rank, local = dist_setup(nccl=True)
    (run_ours_kgb if args.op == "kgb" else run_ours)(args, world, rank, local)


if __name__ == "__main__":
    main()
