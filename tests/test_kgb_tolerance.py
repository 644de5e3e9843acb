"""Where the fused path's tolerance comes from (CPU only).

The fused kernel builds each chunk's matrix in FP32 from keys, decays and betas:
per 16-row block a reference row, Q = k exp(g - g_ref), P = k exp(g_ref - g), a
per-channel factor exp(g_rI - g_rJ) between blocks, FP32 products, then the FP32
solve.  This test runs that arithmetic in numpy float32 and compares it with the
fp64 oracle on the same rounded inputs: the worst error must sit far inside the
2e-5 * (1 + |ref|) the GPU parity tests use for every input dtype.
"""
import numpy as np
import pytest

import kda_inputs as ki
import oracle

BT, BS = 64, 16


def _fp32_construction(k, g, beta, n):
    """FP32 A [n, n] of one chunk-head by the reference-row factorisation."""
    f32 = np.float32
    K = k.shape[1]
    kp = np.zeros((BT, K), f32)
    gp = np.zeros((BT, K), f32)
    kp[:n], gp[:n] = k, g
    A = np.zeros((BT, BT), f32)
    for I in range(4):
        rI = BS * I
        if rI >= n:
            continue
        QI = kp[rI:rI + BS] * np.exp(gp[rI:rI + BS] - gp[rI]).astype(f32)
        for J in range(I + 1):
            rJ = BS * J
            f = np.exp(gp[rI] - gp[rJ]).astype(f32) if I > J else np.ones(K, f32)
            PJ = kp[rJ:rJ + BS] * np.exp(gp[rJ] - gp[rJ:rJ + BS]).astype(f32)
            live_i = (np.arange(BS) + rI < n)[:, None]
            live_j = (np.arange(BS) + rJ < n)[:, None]
            A[rI:rI + BS, rJ:rJ + BS] = np.where(live_i, QI * f, 0).astype(f32) @ np.where(live_j, PJ, 0).astype(f32).T
    return (np.tril(A, -1)[:n, :n] * np.asarray(beta[:n], f32)[:, None]).astype(f32)


def _fp32_solve(A):
    n = A.shape[0]
    X = np.zeros((n, n), np.float32)
    for j in range(n):
        X[j, j] = 1.0
        for i in range(j + 1, n):
            X[i, j] = -np.float32(np.dot(A[i, j:i], X[j:i, j]))
    return X


@pytest.mark.parametrize("kind", ["kda", "nodecay"])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_fp32_construction_is_far_inside_the_tolerance(kind, in_dtype):
    wl = ki.Workload("tol", "packed", H=3, in_dtype=in_dtype, out_dtype="f32", seed=5,
                     seqlens=(64, 64, 40), kind=kind)
    x = ki.build_kgb(wl)
    k, g, b = (oracle.to_f64(t) for t in (x.k, x.g, x.beta))
    ref = oracle.get().solve_kgb(k, g, b, x.cu_seqlens.numpy())[0]
    worst = 0.0
    for row0, n in x.chunks():
        for h in range(x.H):
            A = _fp32_construction(k[0, row0:row0 + n, h].astype(np.float32),
                                   g[0, row0:row0 + n, h].astype(np.float32), b[0, row0:row0 + n, h], n)
            X = _fp32_solve(A)
            R = ref[row0:row0 + n, h, :n]
            worst = max(worst, float(np.max(np.abs(X - R) / (1 + np.abs(R)))))
    assert worst <= 2e-5 / 100, worst
