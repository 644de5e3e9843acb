"""Negative controls for the parity checker, on CPU: mistakes a kernel could make
must fail oracle.parity.check_solution, the verdict every GPU parity test uses.

The two planted mistakes are a zeroed off-diagonal output block and a chunk
boundary shifted by one token.  On KDA-style inputs the decay makes the far
blocks of the inverse tiny, so the zeroed-block mistake is checked on the two
stress kinds (no decay, Gaussian A), and the last test records that on KDA inputs
alone it would go unseen.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
import oracle.parity as parity

BLOCKS = [(1, 0), (2, 0), (3, 0), (2, 1), (3, 1), (3, 2)]
F32 = torch.float32


def _case(kind, seqlens=(64, 64, 64)):
    inp = ki.build(ki.Workload("ctl", "packed", H=2, in_dtype="f32", out_dtype="f32", seed=31,
                               seqlens=seqlens, kind=kind))
    ref = oracle.get().solve_tril(oracle.to_f64(inp.A), inp.cu_seqlens.numpy()).reshape(-1, inp.H, 64)
    return inp, ref


def _verdict(inp, got, ref):
    return parity.check_solution(got, ref, inp.chunks(), 64, inp.A.dtype, F32)[0]


def _zero_block(inp, out, I, J):
    bad = out.copy()
    for row0, n in inp.chunks():
        bad[row0 + 16 * I:row0 + min(n, 16 * I + 16), :, 16 * J:16 * J + 16] = 0.0
    return bad


@pytest.mark.parametrize("blk", BLOCKS, ids=str)
@pytest.mark.parametrize("kind", ["gauss", "nodecay"])
def test_zeroed_block_fails_on_stress_inputs(kind, blk):
    inp, ref = _case(kind)
    good = ref.astype(np.float32).astype(np.float64)        # a correctly rounded fp32 result
    assert _verdict(inp, good, ref)
    assert not _verdict(inp, _zero_block(inp, good, *blk), ref)


def test_shifted_chunk_boundary_fails():
    for kind in ("gauss", "kda"):
        inp, ref = _case(kind, seqlens=(50, 70, 64))
        cu = inp.cu_seqlens.numpy().copy()
        cu[1] += 1                                           # the second request starts a token late
        wrong = oracle.get().solve_tril(oracle.to_f64(inp.A), cu).reshape(-1, inp.H, 64)
        assert not _verdict(inp, wrong.astype(np.float32).astype(np.float64), ref), kind


def test_far_block_is_invisible_on_kda_inputs_alone():
    """Why the stress kinds exist: on KDA inputs block (3,0) of the inverse is so small
    that zeroing it stays within the tolerance."""
    inp, ref = _case("kda")
    good = ref.astype(np.float32).astype(np.float64)
    assert np.abs(ref.reshape(-1, 2, 64)[48:64, :, :16]).max() < 1e-6
    assert _verdict(inp, _zero_block(inp, good, 3, 0), ref)


@pytest.mark.parametrize("layout", ["dense", "packed"])
def test_parts_cover_the_input_and_agree_with_the_whole(layout):
    """The part-by-part comparison of the large workloads sees every chunk exactly
    once, and the oracle run on the parts equals the oracle run on the whole."""
    if layout == "dense":
        wl = ki.Workload("p", "dense", H=3, in_dtype="f32", out_dtype="f32", seed=4, B=5, T=130, kind="gauss")
    else:
        wl = ki.Workload("p", "packed", H=3, in_dtype="bf16", out_dtype="f32", seed=4,
                         seqlens=(1, 200, 0, 64, 65, 7, 300), kind="gauss")
    inp = ki.build(wl)
    orc = oracle.get()
    whole = orc.solve_tril(oracle.to_f64(inp.A), inp.cu_seqlens.numpy() if inp.cu_seqlens is not None else None)
    whole = whole.reshape(-1, inp.H, 64)
    seen = []
    nparts = 0
    for r0, nrows, A_sub, cu_sub, sub in parity.parts(inp, limit=7):
        nparts += 1
        ref = orc.solve_tril(oracle.to_f64(A_sub), cu_sub.numpy() if cu_sub is not None else None)
        assert np.array_equal(ref.reshape(-1, inp.H, 64), whole[r0:r0 + nrows])
        seen += [(r0 + a, n) for (a, n) in sub]
        ok, msg = parity.check_solution(whole[r0:r0 + nrows], ref.reshape(-1, inp.H, 64), sub, 64, inp.A.dtype, F32)
        assert ok, msg
    assert seen == inp.chunks() and nparts > 2
