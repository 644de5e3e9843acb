"""Where the fused path's tolerance comes from (CPU only).

The fused kernel builds each chunk's matrix in FP32 from keys, decays and betas.
Per 16-row block I with first row rI and last live row eI:

* Q_I = k exp(g - g_rI) and P_I = k exp(g_eI - g): every exponent is <= 0 for
  a non-increasing g, so neither factor can overflow;
* block (I, J), I > J: (Q_I * exp(g_rI - g_eJ)) P_J^T, again with a
  non-positive exponent;
* diagonal block (I, I): (Q_I * exp(g_rI - g_eI)) P_I^T for the channels whose
  decay over the block stays within a safe span; the channels that fall
  further are left out of that product and their terms are added one by one as
  k_i k_j exp(g_i - g_j).

This test runs that arithmetic in numpy float32 and compares it with the fp64
oracle on the same rounded inputs: the worst error must sit far inside the
2e-5 * (1 + |ref|) the GPU parity tests use for every input dtype, on KDA
decays, on no decay, and on steep decays (per-token drops of 3 to 20 nats and
cliffs of 100 nats, so that blocks fall by far more than FP32's exponent range).
A planted copy that factors through the block's first row alone (the form that
overflows) must fail on the steep inputs.
"""
import numpy as np
import pytest

import kda_inputs as ki
import oracle

BT, BS = 64, 16
SAFE_SPAN = 32.0          # nats of decay over a diagonal block that its product still takes


def _fp32_construction(k, g, beta, n, first_row_only=False):
    """FP32 A [n, n] of one chunk-head by the block-reference factorisation."""
    f32 = np.float32
    K = k.shape[1]
    kp = np.zeros((BT, K), f32)
    gp = np.zeros((BT, K), f32)
    kp[:n], gp[:n] = k, g
    A = np.zeros((BT, BT), f32)
    live = (np.arange(BT) < n)[:, None]
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        for I in range(4):
            rI = BS * I
            if rI >= n:
                continue
            eI = min(rI + BS - 1, n - 1)
            QI = np.where(live[rI:rI + BS], kp[rI:rI + BS] * np.exp(gp[rI:rI + BS] - gp[rI]), 0).astype(f32)
            for J in range(I + 1):
                rJ = BS * J
                eJ = min(rJ + BS - 1, n - 1)
                if first_row_only:          # P_J = k exp(g_rJ - g): a positive exponent
                    PJ = kp[rJ:rJ + BS] * np.exp(gp[rJ] - gp[rJ:rJ + BS])
                    f = np.exp(gp[rI] - gp[rJ]) if I > J else np.ones(K, f32)
                else:
                    PJ = kp[rJ:rJ + BS] * np.exp(gp[eJ] - gp[rJ:rJ + BS])
                    f = np.exp(gp[rI] - gp[eJ])
                PJ = np.where(live[rJ:rJ + BS], PJ, 0).astype(f32)
                f = f.astype(f32)
                steep = np.zeros(K, bool)
                if I == J and not first_row_only:
                    steep = (gp[rI] - gp[eI]) > SAFE_SPAN
                    f = np.where(steep, f32(0), f).astype(f32)
                blk = (QI * f).astype(f32) @ PJ.T
                for d in np.nonzero(steep)[0]:          # the steep channels, term by term
                    kc, gc = kp[rI:rI + BS, d], gp[rI:rI + BS, d]
                    t = (kc[:, None] * kc[None, :]) * np.exp(gc[:, None] - gc[None, :]).astype(f32)
                    ok = live[rI:rI + BS] & live[rI:rI + BS].T & np.tri(BS, k=-1, dtype=bool)
                    blk = (blk + np.where(ok, t, 0)).astype(f32)
                A[rI:rI + BS, rJ:rJ + BS] = blk
    return (np.tril(A, -1)[:n, :n] * np.asarray(beta[:n], f32)[:, None]).astype(f32)


def _fp32_solve(A):
    n = A.shape[0]
    X = np.zeros((n, n), np.float32)
    for j in range(n):
        X[j, j] = 1.0
        for i in range(j + 1, n):
            X[i, j] = -np.float32(np.dot(A[i, j:i], X[j:i, j]))
    return X


def _worst(kind, in_dtype, first_row_only=False):
    wl = ki.Workload("tol", "packed", H=3, in_dtype=in_dtype, out_dtype="f32", seed=5,
                     seqlens=(64, 64, 40), kind=kind)
    x = ki.build_kgb(wl)
    k, g, b = (oracle.to_f64(t) for t in (x.k, x.g, x.beta))
    ref = oracle.get().solve_kgb(k, g, b, x.cu_seqlens.numpy())[0]
    worst = 0.0
    with np.errstate(invalid="ignore", over="ignore"):
        for row0, n in x.chunks():
            for h in range(x.H):
                A = _fp32_construction(k[0, row0:row0 + n, h].astype(np.float32),
                                       g[0, row0:row0 + n, h].astype(np.float32), b[0, row0:row0 + n, h], n,
                                       first_row_only)
                X = _fp32_solve(A)
                R = ref[row0:row0 + n, h, :n]
                err = np.abs(X - R) / (1 + np.abs(R))
                worst = max(worst, float(np.inf if not np.all(np.isfinite(err)) else np.max(err)))
    return worst


@pytest.mark.parametrize("kind", ["kda", "nodecay", "steep"])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_fp32_construction_is_far_inside_the_tolerance(kind, in_dtype):
    worst = _worst(kind, in_dtype)
    assert worst <= 2e-5 / 100, worst


def test_first_row_factorisation_fails_on_steep_decays():
    assert _worst("steep", "f32", first_row_only=True) > 2e-5
