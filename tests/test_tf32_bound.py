"""Where the TF32 precision mode's tolerance comes from (CPU only).

The TF32 mode of the 64-token solve keeps the four diagonal 16x16 inverses in
FP32 and forms every merge product (level A: X10 = -X11 A10 X00, X32 = -X33 A32
X22; level B: T = A_BL X_TL, X_BL = -X_BR T) from operands truncated to TF32 with
FP32 accumulation.  This test runs that arithmetic in numpy and checks, against
the fp64 oracle on the same rounded inputs, that its error stays inside
oracle.parity.tf32_bounds() -- with room -- on KDA, Gaussian and no-decay
inputs, and that planted mistakes in the merge (a wrong sign, a dropped term, a
transposed operand) land outside it.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
import oracle.parity as parity

BT = 64


def _tf32(x):
    return (np.asarray(x, np.float32).view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32).astype(np.float64)


def _prod(P, Q):
    """One TF32 tensor-core product: operands truncated, FP32 result."""
    return (_tf32(P) @ _tf32(Q)).astype(np.float32).astype(np.float64)


def _tf32_solve(A, n, plant=None):
    """The TF32 mode's arithmetic on one chunk-head's n x n strictly lower A."""
    L = np.zeros((BT, BT))
    L[:n, :n] = np.tril(A[:n, :n], -1)
    L = L.astype(np.float32).astype(np.float64)
    X = np.zeros((BT, BT))
    blk = lambda M, i, j: M[16 * i:16 * i + 16, 16 * j:16 * j + 16]
    for b in range(4):                                   # FP32 diagonal inverses
        D = np.linalg.inv(np.eye(16) + blk(L, b, b)).astype(np.float32).astype(np.float64)
        X[16 * b:16 * b + 16, 16 * b:16 * b + 16] = D
    for (i, j) in ((1, 0), (3, 2)):                      # level A
        T = _prod(blk(L, i, j), blk(X, j, j))
        if plant == "transpose":
            T = _prod(blk(L, i, j).T, blk(X, j, j))
        X[16 * i:16 * i + 16, 16 * j:16 * j + 16] = -_prod(blk(X, i, i), T)
    # level B: T = A_BL X_TL, then X_BL = -X_BR T, block by block
    T = {}
    for i in (2, 3):
        for j in (0, 1):
            acc = _prod(blk(L, i, 0), blk(X, 0, j)) + (_prod(blk(L, i, 1), blk(X, 1, j)) if plant != "drop" else 0)
            T[i, j] = acc.astype(np.float32).astype(np.float64)
    for i in (2, 3):
        for j in (0, 1):
            acc = _prod(blk(X, i, 2), T[2, j]) + _prod(blk(X, i, 3), T[3, j])
            sign = 1.0 if (plant == "sign" and (i, j) == (3, 0)) else -1.0
            X[16 * i:16 * i + 16, 16 * j:16 * j + 16] = sign * acc.astype(np.float32).astype(np.float64)
    out = np.zeros((n, BT))
    out[:, :n] = X[:n, :n]
    return out


def _worst(kind, plant=None, in_dtype="f32"):
    wl = ki.Workload("tf32", "packed", H=2, in_dtype=in_dtype, out_dtype="f32", seed=11,
                     seqlens=(64, 64, 50, 64), kind=kind)
    inp = ki.build(wl)
    A = oracle.to_f64(inp.A)[0]
    ref = oracle.get().solve_tril(oracle.to_f64(inp.A), inp.cu_seqlens.numpy())[0]
    got = np.zeros_like(ref)
    for row0, n in inp.chunks():
        for h in range(inp.H):
            got[row0:row0 + n, h] = _tf32_solve(A[row0:row0 + n, h], n, plant)
    ok, msg, worst = parity.check_solution_tf32(got, ref, A, inp.chunks(), BT, torch.float32)
    return ok, worst


@pytest.mark.parametrize("kind", ["kda", "gauss", "nodecay"])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_tf32_arithmetic_is_inside_the_bound_with_room(kind, in_dtype):
    ok, worst = _worst(kind, in_dtype=in_dtype)
    assert ok and worst < 0.25, worst


@pytest.mark.parametrize("plant", ["sign", "drop", "transpose"])
def test_planted_merge_mistakes_exceed_the_bound(plant):
    ok, worst = _worst("kda", plant)
    assert not ok and worst > 1.0, (plant, worst)
