"""Stream order of back-to-back launches (GPU).

The single-pass, short-chunk and fused kernels are launched with programmatic
stream serialization: each may be scheduled while the previous kernel of the
stream is still running, and waits (griddepcontrol.wait) before its first global
memory access (the split path's kernels are ordinary launches).  These
tests check the orderings that wait must give, against the same calls with a
device synchronisation between them (the kernels are deterministic, so the
results must be bitwise equal):

* read after write: a solve that reads the previous solve's output;
* write after read: a solve that overwrites the buffer the previous one reads;
* the same sequences captured in a CUDA graph and replayed.
"""
from __future__ import annotations

import pytest
import torch

import kda_inputs as ki

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_chunked_02_gb300 import build as kbuild
    kbuild.build()
    import linear_attention_chunked_02_gb300 as k
    return k


def _input(bt: int):
    wl = ki.WORKLOADS["packed_16x512_h64_f32"].with_(bt=bt)
    inp = ki.build(wl)
    return inp.A.to(DEV), inp.cu_seqlens.to(DEV)


def _chain(kda, A, cu, n, sync):
    """n solves, each reading the previous one's output as its input."""
    outs = []
    x = A
    for _ in range(n):
        x = kda.solve_tril(x, cu, out_dtype=torch.float32, path="single")
        if sync:
            torch.cuda.synchronize()
        outs.append(x)
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("bt", [16, 32, 64])
def test_read_after_write(kda, bt):
    A, cu = _input(bt)
    ref = _chain(kda, A, cu, 3, sync=True)
    assert all(bool(torch.isfinite(r).all()) for r in ref)
    for _ in range(3):
        got = _chain(kda, A, cu, 3, sync=False)
        for r, g in zip(ref, got):
            assert torch.equal(r, g)


@pytest.mark.parametrize("bt", [16, 32, 64])
def test_write_after_read(kda, bt):
    A, cu = _input(bt)
    A2 = A * 0.5                                        # another input of the same shape
    ref1 = kda.solve_tril(A, cu, out_dtype=torch.float32, path="single")
    ref2 = kda.solve_tril(A2, cu, out_dtype=torch.float32, path="single")
    torch.cuda.synchronize()
    for _ in range(3):
        src = A.clone()
        torch.cuda.synchronize()
        out1 = torch.empty_like(ref1)
        kda.solve_tril(src, cu, out_dtype=torch.float32, path="single", out=out1)
        # the next solve writes into the buffer the previous one reads
        kda.solve_tril(A2, cu, out_dtype=torch.float32, path="single", out=src)
        torch.cuda.synchronize()
        assert torch.equal(out1, ref1)
        assert torch.equal(src, ref2)


def test_split_path_kernels_in_order(kda):
    """The split path's merge kernel reads the workspace its diagonal kernel writes."""
    A, cu = _input(64)
    single = kda.solve_tril(A, cu, out_dtype=torch.float32, path="single")
    for _ in range(3):
        split = kda.solve_tril(A, cu, out_dtype=torch.float32, path="split")
        torch.cuda.synchronize()
        assert torch.equal(split, single)


def test_fused_construction_then_solve(kda):
    """The fused construction's output feeds a solve launched right behind it."""
    wl = ki.WORKLOADS["packed_16x512_h64_f32"]
    x = ki.build_kgb(wl)
    k, g, b = x.k.to(DEV), x.g.to(DEV), x.beta.to(DEV)
    cu = x.cu_seqlens.to(DEV)
    Ai = kda.solve_tril_kgb(k, g, b, cu)
    torch.cuda.synchronize()
    ref = kda.solve_tril(Ai, cu, out_dtype=torch.float32, path="single")
    torch.cuda.synchronize()
    for _ in range(3):
        Ai2 = kda.solve_tril_kgb(k, g, b, cu)
        got = kda.solve_tril(Ai2, cu, out_dtype=torch.float32, path="single")
        torch.cuda.synchronize()
        assert torch.equal(Ai2, Ai)
        assert torch.equal(got, ref)


@pytest.mark.parametrize("bt", [16, 64])
def test_graph_replay(kda, bt):
    A, cu = _input(bt)
    ref = _chain(kda, A, cu, 2, sync=True)
    s = torch.cuda.Stream()
    o1 = torch.empty_like(ref[0])
    o2 = torch.empty_like(ref[1])
    with torch.cuda.stream(s):
        kda.solve_tril(A, cu, out_dtype=torch.float32, path="single", out=o1, stream=s)   # set-up outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            kda.solve_tril(A, cu, out_dtype=torch.float32, path="single", out=o1, stream=s)
            kda.solve_tril(o1, cu, out_dtype=torch.float32, path="single", out=o2, stream=s)
    torch.cuda.synchronize()
    for _ in range(3):
        o1.zero_()
        o2.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o1, ref[0])
        assert torch.equal(o2, ref[1])
