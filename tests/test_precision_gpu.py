"""The TF32 precision mode of the 64-token solve against the fp64 oracle (GPU).

kda_solve_tril_prec(..., KDA_PREC_TF32) keeps the diagonal inverses in FP32 and
forms each merge product as one TF32 tensor-core product.  Its error bound is
derived from that arithmetic (oracle.parity.tf32_bounds, pinned on the CPU by
tests/test_tf32_bound.py); structural entries must still be exact.  The IEEE mode
of the same entry must equal kda_solve_tril_ex's single pass bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
import oracle.parity as parity

pytestmark = pytest.mark.gpu

F32, BF16, F16 = torch.float32, torch.bfloat16, torch.float16
NAMES = {F32: "f32", BF16: "bf16", F16: "f16"}
DEV = "cuda:0"


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_chunked_02_gb300 import build as kbuild
    kbuild.build()
    import linear_attention_chunked_02_gb300 as k
    return k


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def run(kda, inp, out_dtype, precision):
    A = inp.A.to(DEV)
    cu = inp.cu_seqlens.to(DEV) if inp.cu_seqlens is not None else None
    out = kda.solve_tril(A, cu, out_dtype=out_dtype, path="single", precision=precision)
    torch.cuda.synchronize()
    return out


def check_tf32(inp, got_t, ref, out_dtype, label):
    H, bt = inp.H, inp.bt
    got = got_t.to(torch.float64).cpu().numpy().reshape(-1, H, bt)
    A = oracle.to_f64(inp.A).reshape(-1, H, bt)
    ok, msg, worst = parity.check_solution_tf32(got, ref.reshape(-1, H, bt), A, inp.chunks(), bt, out_dtype)
    assert ok, f"{label}: {msg}"
    return worst


def oracle_ref(orc, inp):
    return orc.solve_tril(oracle.to_f64(inp.A), inp.cu_seqlens.numpy() if inp.cu_seqlens is not None else None)


@pytest.mark.parametrize("in_dtype", [F32, BF16, F16], ids=str)
@pytest.mark.parametrize("out_dtype", [F32, BF16], ids=str)
@pytest.mark.parametrize("kind", ["kda", "gauss", "nodecay"])
def test_tf32_mode_within_its_bound(kda, orc, in_dtype, out_dtype, kind):
    inp = ki.build(ki.Workload("prec", "packed", H=4, in_dtype=NAMES[in_dtype], out_dtype=NAMES[out_dtype],
                               seed=23, seqlens=(1, 63, 64, 65, 200, 0, 128, 7), kind=kind))
    ref = oracle_ref(orc, inp)
    got = run(kda, inp, out_dtype, "tf32")
    check_tf32(inp, got, ref, out_dtype, f"{in_dtype}->{out_dtype} {kind}")
    ieee = run(kda, inp, out_dtype, "ieee")
    single = kda.solve_tril(inp.A.to(DEV), inp.cu_seqlens.to(DEV), out_dtype=out_dtype, path="single")
    torch.cuda.synchronize()
    assert torch.equal(ieee, single)                   # the IEEE mode is the single pass
    if out_dtype == F32:
        assert not torch.equal(got, ieee)              # the TF32 mode really computes in TF32


@pytest.mark.parametrize("T", [1, 17, 64, 65, 130])
def test_tf32_mode_dense_edges(kda, orc, T):
    inp = ki.build(ki.Workload("pe", "dense", H=3, in_dtype="f32", out_dtype="f32", seed=T, B=2, T=T,
                               kind="gauss"))
    check_tf32(inp, run(kda, inp, F32, "tf32"), oracle_ref(orc, inp), F32, f"T={T}")


def test_tf32_mode_block_diagonal_input_is_exact(kda):
    """With the off-diagonal blocks zero the merge products are zero in any
    precision: the TF32 mode must equal the IEEE mode bit for bit."""
    inp = ki.build(ki.Workload("bd", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=3, B=1, T=128,
                               kind="gauss"))
    A = inp.A.clone()
    for c0 in range(0, 128, 64):
        for i in range(64):
            A[0, c0 + i, :, : 16 * (i // 16)] = 0.0
    Ad = A.to(DEV)
    tf = kda.solve_tril(Ad, out_dtype=F32, path="single", precision="tf32")
    ie = kda.solve_tril(Ad, out_dtype=F32, path="single", precision="ieee")
    torch.cuda.synchronize()
    assert torch.equal(tf, ie)


def test_tf32_mode_full_size_every_element(kda, orc):
    """The 8192-token x 64-head workload, every element against the bound."""
    inp = ki.build(ki.WORKLOADS["packed_16x512_h64_f32"])
    ref = oracle_ref(orc, inp)
    worst = check_tf32(inp, run(kda, inp, F32, "tf32"), ref, F32, "16x512")
    assert worst < 0.5, worst


def test_tf32_mode_rejects_what_it_does_not_do(kda):
    A = torch.zeros(1, 64, 1, 64, device=DEV)
    with pytest.raises(ValueError):
        kda.solve_tril(A, path="split", precision="tf32")
    with pytest.raises(ValueError):
        kda.solve_tril(torch.zeros(1, 32, 1, 32, device=DEV), precision="tf32")
