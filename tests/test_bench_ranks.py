"""The multi-rank path of bench.py on CPU (gloo, world size 2).

On this pool every rank solves its own replica of the workload; the only
cross-rank operations are the barriers around the timed region and the
maximum of the per-rank times.  These tests run them with two gloo ranks.
"""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r took (1 + r) ms for 1e9 bytes: the job is as slow as the slowest rank
        ms, gbs = bench.whole_job_gbs(1.0 + rank, 10 ** 9, world, "cpu")
        q.put((rank, ms, gbs))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_whole_job_time_is_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, gbs in got:
        assert ms == 2.0
        assert abs(gbs - 2 * 1e9 / 2e-3 / 1e9) < 1e-9       # two replicas of 1 GB in 2 ms


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_gbs(4.0, 2 * 10 ** 9, 1, "cpu") == (4.0, 500.0)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched on two ranks: rank 0 alone prints its line."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_fused_op():
    """`bench.py --impl reference --op kgb`: the oracle of the fused path on the host."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--op", "kgb", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "packed_16x512_h64_f32_kgb"
    assert d["config"]["key_dim"] == 128 and d["cpu_baseline"]["kind"] == "oracle"
