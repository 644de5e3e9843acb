"""The reference arm of bench.py (the oracle on the host cores, CPU only).

`bench.py --impl reference` times the oracle on a bounded sample of the
workload.  These tests check that a sample is a genuine sub-workload (the
oracle's answer on it is the matching slice of its answer on the whole), that
the sample size follows the time budget, and that the arm prints its JSON line.
"""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

import numpy as np
import pytest

import bench
import kda_inputs as ki
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _solve(x):
    cu = x.cu_seqlens.numpy() if x.cu_seqlens is not None else None
    return oracle.get().solve_tril(oracle.to_f64(x.A), cu)


def test_packed_sample_is_a_sub_workload():
    full = ki.build(ki.Workload("s", "packed", H=4, in_dtype="f32", out_dtype="f32", seed=5,
                                seqlens=(64, 50, 128, 7)))
    part = bench.sample_input(full, 2, 3)
    rows = int(full.cu_seqlens[2])
    assert part.A.shape == (1, rows, 3, 64) and list(part.seqlens) == [64, 50]
    np.testing.assert_array_equal(_solve(part), _solve(full)[:, :rows, :3])


def test_dense_sample_is_a_sub_workload():
    full = ki.build(ki.Workload("s", "dense", H=4, in_dtype="bf16", out_dtype="f32", seed=6, B=3, T=70))
    part = bench.sample_input(full, 2, 1)
    assert part.A.shape == (2, 70, 1, 64)
    np.testing.assert_array_equal(_solve(part), _solve(full)[:2, :, :1])


def test_kgb_sample_is_a_sub_workload():
    full = ki.build_kgb(ki.Workload("s", "packed", H=3, in_dtype="f32", out_dtype="f32", seed=7,
                                    seqlens=(40, 64, 90)), K=32)
    part = bench.sample_kgb(full, 2, 2)
    rows = int(full.cu_seqlens[2])
    orc = oracle.get()
    got = orc.solve_kgb(*(oracle.to_f64(t) for t in (part.k, part.g, part.beta)), part.cu_seqlens.numpy())
    ref = orc.solve_kgb(*(oracle.to_f64(t) for t in (full.k, full.g, full.beta)), full.cu_seqlens.numpy())
    np.testing.assert_array_equal(got, ref[:, :rows, :2])


def _full(units, heads, packed=True):
    return SimpleNamespace(B=units, H=heads, cu_seqlens=object() if packed else None,
                           seqlens=list(range(units)))


def test_reference_sample_halves_heads_then_units():
    seen = []

    def time_of(u, h):                        # 10 ms per request and head
        seen.append((u, h))
        return 0.01 * u * h

    units, heads = bench.reference_sample(_full(16, 64), 1000, time_of)
    # heads halve 64 -> 1 first (1000 steps x 0.16 s still over 90 s), then requests 16 -> 8
    assert (units, heads) == (8, 1)
    assert 1000 * 0.01 * units * heads <= bench.REFERENCE_BUDGET_S
    assert seen[:3] == [(16, 64), (16, 32), (16, 16)]


def test_reference_sample_keeps_the_whole_workload_when_it_fits():
    assert bench.reference_sample(_full(4, 8, packed=False), 3, lambda u, h: 1.0) == (4, 8)


def test_reference_sample_stops_when_halving_no_longer_pays():
    # a fixed 1 s per solve dominates: halving the heads saves under a quarter
    units, heads = bench.reference_sample(_full(16, 64), 1000, lambda u, h: 1.0 + 1e-4 * u * h)
    assert (units, heads) == (16, 64)


def _reference_line(*extra):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "dense_1x64_h4_f32",
                        "--steps", "3", "--warmup", "3", *extra],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("extra", [(), ("--op", "kgb")], ids=["solve", "kgb"])
def test_reference_arm_prints_its_line(extra):
    d = _reference_line(*extra)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("dense_1x64_h4_f32")
