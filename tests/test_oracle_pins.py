"""Pins for the fp64 oracle: facts fixed by mathematics, not by the oracle itself.

Each ``check_*`` raises AssertionError on a mismatch and takes an oracle
handle, so the negative controls at the bottom can run the same checks on
copies of the oracle compiled with a deliberate mistake.

Operation (LightLLM PR #1703, PR description): per 64-token chunk and head,
``(I + A)^-1`` for the strictly lower-triangular chunk matrix ``A``; chunks
restart at every request start (packed) or batch row (dense).
"""
from __future__ import annotations

import itertools
import os
from fractions import Fraction

import numpy as np
import pytest

import kda_inputs as ki
import oracle as orc_mod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_cases.txt")
BT = 64


def _series_inverse(M: np.ndarray) -> np.ndarray:
    """(I + M)^-1 = sum_{k=0}^{n-1} (-M)^k, exact for nilpotent (strictly lower) M."""
    n = M.shape[0]
    term = np.eye(n)
    acc = np.eye(n)
    for _ in range(1, n):
        term = term @ (-M)
        acc = acc + term
    return acc


def _strict(M: np.ndarray, n: int) -> np.ndarray:
    out = np.tril(np.asarray(M, dtype=np.float64)[:n, :n], -1)
    return out


def _load_golden():
    cases = []
    lines = [l.strip() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    i = 0
    while i < len(lines):
        assert lines[i].startswith("case")
        name = lines[i].split()[1]
        n = int(lines[i + 1].split()[1])
        assert lines[i + 2] == "M"
        M = np.array([[float(x) for x in lines[i + 3 + r].split()] for r in range(n)])
        assert lines[i + 3 + n] == "X"
        X = np.array([[float(x) for x in lines[i + 4 + n + r].split()] for r in range(n)])
        assert lines[i + 4 + 2 * n] == "end"
        cases.append((name, n, M, X))
        i += 5 + 2 * n
    return cases


# ---------------------------------------------------------------- the checks

def check_golden(orc):
    """Hand-worked cases from tests/golden/worked_cases.txt, bit-exact."""
    for name, n, M, X in _load_golden():
        got = orc.invert_chunk(M, n)
        assert np.array_equal(got[:n, :n], X), name
        assert np.array_equal(got[n:, n:], np.eye(BT - n)), name


def check_worked_small(orc):
    """2x2 [[0,0],[a,0]] -> [[1,0],[-a,1]]; 4x4 bidiagonal a=2 -> (-2)^(i-j)."""
    for a in (0.5, -3.0, 7.25):
        got = orc.invert_chunk(np.array([[0.0, 0.0], [a, 0.0]]), 2)
        assert np.array_equal(got[:2, :2], np.array([[1.0, 0.0], [-a, 1.0]]))
    M = np.diag([2.0] * 3, -1)
    got = orc.invert_chunk(M, 4)
    want = np.array([[(-2.0) ** (i - j) if j <= i else 0.0 for j in range(4)] for i in range(4)])
    assert np.array_equal(got[:4, :4], want)


def _cofactor_inverse(L):
    """Exact inverse of an integer unit lower-triangular matrix via cofactors (Leibniz)."""
    n = len(L)

    def det(m):
        k = len(m)
        if k == 0:
            return Fraction(1)
        tot = Fraction(0)
        for perm in itertools.permutations(range(k)):
            inv = sum(1 for a in range(k) for b in range(a + 1, k) if perm[a] > perm[b])
            p = Fraction(-1 if inv % 2 else 1)
            for r in range(k):
                p *= m[r][perm[r]]
                if p == 0:
                    break
            tot += p
        return tot

    d = det(L)
    X = [[Fraction(0)] * n for _ in range(n)]
    for i in range(n):
        for j in range(n):
            minor = [[L[r][c] for c in range(n) if c != i] for r in range(n) if r != j]
            X[i][j] = (-1) ** (i + j) * det(minor) / d
    return X


def check_rational(orc):
    """Small-integer cases, n <= 6, equal exactly to the cofactor inverse in rationals."""
    rng = np.random.default_rng(1234)
    for n in range(1, 7):
        for _ in range(3):
            M = np.tril(rng.integers(-3, 4, size=(n, n)), -1).astype(np.float64)
            L = [[Fraction(int(M[r][c])) + (1 if r == c else 0) for c in range(n)] for r in range(n)]
            X = _cofactor_inverse(L)
            want = np.array([[float(x) for x in row] for row in X])
            got = orc.invert_chunk(M, n)
            assert np.array_equal(got[:n, :n], want), (n, M)


def check_closed_form(orc):
    """Config-style, no-decay and Gaussian chunks against the nilpotent series, 1e-12."""
    for kind, seed in (("kda", 11), ("nodecay", 12), ("gauss", 13)):
        wl = ki.Workload("pin", "packed", H=2, in_dtype="f32", out_dtype="f32", seed=seed,
                         seqlens=(64, 40, 17), kind=kind)
        inp = ki.build(wl)
        A = orc_mod.to_f64(inp.A)[0]
        for row0, n in inp.chunks():
            for h in range(inp.H):
                M = _strict(A[row0:row0 + n, h, :], n)
                want = _series_inverse(M)
                got = orc.invert_chunk(A[row0:row0 + n, h, :], n)[:n, :n]
                err = np.abs(got - want) / (1.0 + np.abs(want))
                assert err.max() <= 1e-12, (kind, row0, n, h, err.max())


def check_exact_64(orc):
    """64x64 structures whose inverse is exact in floating point."""
    Z = np.zeros((BT, BT))
    I = np.eye(BT)
    assert np.array_equal(orc.invert_chunk(Z, BT), I)
    ones = np.tril(np.ones((BT, BT)), -1)
    assert np.array_equal(orc.invert_chunk(ones, BT), I - np.diag(np.ones(BT - 1), -1))
    bi = np.diag(np.full(BT - 1, 0.5), -1)
    want = np.array([[(-0.5) ** (i - j) if j <= i else 0.0 for j in range(BT)] for i in range(BT)])
    assert np.array_equal(orc.invert_chunk(bi, BT), want)
    rng = np.random.default_rng(7)
    # nonzeros only in the four diagonal 16x16 blocks: off-diagonal blocks stay exactly 0
    M = np.zeros((BT, BT))
    for b in range(4):
        s = slice(16 * b, 16 * b + 16)
        M[s, s] = np.tril(rng.standard_normal((16, 16)) * 0.3, -1)
    X = orc.invert_chunk(M, BT)
    for bi_ in range(4):
        for bj in range(4):
            blk = X[16 * bi_:16 * bi_ + 16, 16 * bj:16 * bj + 16]
            if bi_ != bj:
                assert np.all(blk == 0.0)
            else:
                want = _series_inverse(M[16 * bi_:16 * bi_ + 16, 16 * bi_:16 * bi_ + 16])
                assert np.abs(blk - want).max() <= 1e-13
    # nonzeros only in one off-diagonal block: A^2 = 0, so the inverse is I - A exactly
    for p in range(4):
        for q in range(p):
            M = np.zeros((BT, BT))
            M[16 * p:16 * p + 16, 16 * q:16 * q + 16] = rng.standard_normal((16, 16))
            assert np.array_equal(orc.invert_chunk(M, BT), I - M), (p, q)
    # chains of blocks with power-of-two entries: I - A + A^2 - A^3 exactly
    for chain in ([(1, 0), (2, 1)], [(1, 0), (2, 1), (3, 2)], [(2, 1), (3, 2)], [(3, 1), (1, 0)]):
        M = np.zeros((BT, BT))
        for p, q in chain:
            M[16 * p:16 * p + 16, 16 * q:16 * q + 16] = (
                rng.integers(-1, 2, size=(16, 16)) * 2.0 ** -rng.integers(0, 4, size=(16, 16)))
        want = I - M + M @ M - M @ M @ M
        assert np.array_equal(orc.invert_chunk(M, BT), want), chain


def check_similarity(orc):
    """Power-of-two diagonal similarity: for D = diag(2^e), (I + D M D^-1)^-1 =
    D (I + M)^-1 D^-1, exactly -- every term of row i, column j of the forward
    substitution scales by the same 2^(e_i - e_j).  An index that takes a row or
    column other than the term's own (M[i-1][k], X[k][j+1]) breaks it."""
    rng = np.random.default_rng(17)
    for n in (64, 37):
        M = np.tril(rng.standard_normal((n, n)) * 0.2, -1)
        e = rng.integers(-3, 4, n)
        D = np.ldexp(1.0, e)
        Ms = M * D[:, None] / D[None, :]
        X = orc.invert_chunk(M, n)[:n, :n]
        Xs = orc.invert_chunk(Ms, n)[:n, :n]
        assert np.array_equal(Xs, X * D[:, None] / D[None, :]), n


def check_residual(orc):
    """||(I + M) X - I||_max <= 1e-12 on config-style chunks, full and partial."""
    wl = ki.Workload("pin", "dense", H=3, in_dtype="f32", out_dtype="f32", seed=21, B=2, T=100)
    inp = ki.build(wl)
    A = orc_mod.to_f64(inp.A).reshape(-1, inp.H, BT)
    for row0, n in inp.chunks():
        for h in range(inp.H):
            M = _strict(A[row0:row0 + n, h, :], n)
            X = orc.invert_chunk(A[row0:row0 + n, h, :], n)[:n, :n]
            assert np.abs((np.eye(n) + M) @ X - np.eye(n)).max() <= 1e-12


def _expected_layout(A64, chunks, H):
    """Per-chunk placement written out independently of the oracle's own enumeration."""
    out = np.zeros_like(A64)
    for row0, n in chunks:
        for h in range(H):
            M = _strict(A64[row0:row0 + n, h, :], n)
            X = _series_inverse(M)
            out[row0:row0 + n, h, :n] = X
    return out


def check_layout(orc):
    """Chunk boundaries: packed restarts at each request, dense at each batch row."""
    wl = ki.Workload("pin", "packed", H=2, in_dtype="f32", out_dtype="f32", seed=31,
                     seqlens=(5, 70, 64, 0, 130, 1), kind="gauss")
    inp = ki.build(wl)
    A = orc_mod.to_f64(inp.A)
    got = orc.solve_tril(A, inp.cu_seqlens.numpy())[0]
    want = _expected_layout(A[0], inp.chunks(), inp.H)
    assert np.abs(got - want).max() <= 1e-12
    # each request solved alone as a dense row gives the same bits
    cu = inp.cu_seqlens.tolist()
    for s in range(len(cu) - 1):
        if cu[s + 1] == cu[s]:
            continue
        dense = orc.solve_tril(A[:, cu[s]:cu[s + 1]])
        assert np.array_equal(dense[0], got[cu[s]:cu[s + 1]])
    wl = ki.Workload("pin", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=32, B=3, T=77,
                     kind="gauss")
    inp = ki.build(wl)
    A = orc_mod.to_f64(inp.A)
    got = orc.solve_tril(A).reshape(-1, inp.H, BT)
    want = _expected_layout(A.reshape(-1, inp.H, BT), inp.chunks(), inp.H)
    assert np.abs(got - want).max() <= 1e-12


def check_poison(orc):
    """NaN written into every ignored element changes nothing."""
    wl = ki.Workload("pin", "packed", H=2, in_dtype="f32", out_dtype="f32", seed=41,
                     seqlens=(3, 64, 100))
    clean = ki.build(wl)
    dirty = ki.build(wl, poison=True)
    assert torch_isnan_any(dirty.A)
    a = orc.solve_tril(orc_mod.to_f64(clean.A), clean.cu_seqlens.numpy())
    b = orc.solve_tril(orc_mod.to_f64(dirty.A), dirty.cu_seqlens.numpy())
    assert np.array_equal(a, b)


def torch_isnan_any(t) -> bool:
    import torch
    return bool(torch.isnan(t.float()).any())


# ------------------------------- chunk matrices from keys, betas and decays
KGB_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kgb_cases.txt")


def _load_kgb_golden():
    lines = [l.strip() for l in open(KGB_GOLDEN) if l.strip() and not l.startswith("#")]
    cases, i = [], 0
    while i < len(lines):
        name = lines[i].split()[1]
        _, n, _, K = lines[i + 1].split()
        n, K = int(n), int(K)
        i += 2
        blocks = {}
        for key, rows in (("k", n), ("g", n), ("beta", 1), ("X", n)):
            assert lines[i] == key, (name, lines[i])
            blocks[key] = np.array([[float(x) for x in lines[i + 1 + r].split()] for r in range(rows)])
            i += 1 + rows
        assert lines[i] == "end"
        i += 1
        cases.append((name, n, K, blocks))
    return cases


def _kgb_one(orc, k, g, beta, cu=None):
    """k, g: [T, K]; beta: [T] for one head of one batch row."""
    k = np.asarray(k, dtype=np.float64)[None, :, None, :]
    g = np.asarray(g, dtype=np.float64)[None, :, None, :]
    beta = np.asarray(beta, dtype=np.float64).reshape(1, -1, 1)
    Ai, A = orc.solve_kgb(k, g, beta, cu, return_A=True)
    return Ai[0, :, 0, :], A[0, :, 0, :]


def check_kgb_golden(orc):
    """Hand-worked (k, g, beta) -> X cases (tests/golden/kgb_cases.txt)."""
    for name, n, K, b in _load_kgb_golden():
        Ai, _ = _kgb_one(orc, b["k"], b["g"], b["beta"][0])
        assert np.abs(Ai[:n, :n] - b["X"]).max() <= 1e-15, name
        assert np.all(Ai[:n, n:] == 0), name


def check_kgb_nodecay(orc):
    """g = 0: A is beta_i (K K^T)_ij below the diagonal (a plain matrix product)."""
    rng = np.random.default_rng(7)
    for T, K in ((64, 128), (50, 32), (130, 8)):
        k = rng.standard_normal((T, K))
        beta = rng.uniform(0.1, 1.0, T)
        _, A = _kgb_one(orc, k, np.zeros((T, K)), beta)
        for t0 in range(0, T, BT):
            n = min(BT, T - t0)
            kc = k[t0:t0 + n]
            want = np.tril(beta[t0:t0 + n, None] * (kc @ kc.T), -1)
            assert np.abs(A[t0:t0 + n, :n] - want).max() <= 1e-12 * max(1.0, np.abs(want).max())
            assert np.all(A[t0:t0 + n, n:] == 0)


def check_kgb_decay_closed_form(orc):
    """One-hot keys, beta = 1, g_t = -lam * t on every channel: A[i][j] = r^(i-j)
    with r = exp(-lam), so I + A = (I - r S)^-1 and the inverse is I - r S
    (S = ones on the subdiagonal), in every chunk, full or partial."""
    for lam, T, K in ((0.3, 64, 4), (1.0, 100, 1), (0.05, 37, 16)):
        k = np.zeros((T, K))
        k[:, 0] = 1.0
        g = -lam * np.arange(T, dtype=np.float64)[:, None] * np.ones((1, K))
        Ai, _ = _kgb_one(orc, k, g, np.ones(T))
        r = np.exp(-lam)
        for t0 in range(0, T, BT):
            n = min(BT, T - t0)
            want = np.eye(n) - r * np.eye(n, k=-1)
            assert np.abs(Ai[t0:t0 + n, :n] - want).max() <= 1e-13, (lam, t0)


def check_kgb_shift_invariance(orc):
    """Only differences of g inside a chunk enter: g + c (c per channel) changes nothing."""
    wl = ki.Workload("pin", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=43, B=1, T=90)
    x = ki.build_kgb(wl, K=16)
    k, g, beta = (orc_mod.to_f64(t) for t in (x.k, x.g, x.beta))
    c = np.random.default_rng(3).uniform(-5, 5, (1, 1, 2, 16))
    a = orc.solve_kgb(k, g, beta)
    b = orc.solve_kgb(k, g + c, beta)
    assert np.abs(a - b).max() <= 1e-12


def check_kgb_generator(orc):
    """The oracle's per-term definition against the generator's factorised matrix
    product (exp(g_i) and exp(-g_j) split) on the same fp64 draws, and the solve
    against the plain solver oracle on that matrix."""
    for kind in ("kda", "nodecay"):
        rng = np.random.default_rng(11)
        L, H = 150, 2
        k, beta, g = ki._draw_kgb(rng, L, H, kind)
        A_gen = ki._slab(np.random.default_rng(11), L, H, kind)
        Ai, A = orc.solve_kgb(k[None], g[None], beta[None], return_A=True)
        assert np.abs(A[0] - A_gen).max() <= 1e-12, kind
        Ai2 = orc.solve_tril(A_gen[None])
        assert np.abs(Ai - Ai2).max() <= 1e-11, kind


KGB_CHECKS = [check_kgb_golden, check_kgb_nodecay, check_kgb_decay_closed_form,
              check_kgb_shift_invariance, check_kgb_generator]

ALL_CHECKS = [check_golden, check_worked_small, check_rational, check_closed_form,
              check_exact_64, check_similarity, check_residual, check_layout, check_poison] + KGB_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check, oracle_lib):
    assert oracle_lib.planted() == 0
    check(oracle_lib)


# ------------------------------------------------------- negative controls
# A copy of the oracle compiled with one deliberate mistake must fail the pins
# named here; otherwise the pins would not be able to see that mistake.
PLANTS = {
    1: ("drops the last term of each row sum", ["check_golden", "check_rational",
                                                 "check_closed_form", "check_exact_64"]),
    2: ("wrong sign of the off-diagonal entries", ["check_golden", "check_worked_small",
                                                    "check_rational", "check_closed_form"]),
    3: ("packed chunk boundary shifted by one token", ["check_layout"]),
    4: ("decay exponent reversed", ["check_kgb_golden", "check_kgb_decay_closed_form",
                                    "check_kgb_generator"]),
    5: ("beta of the column instead of the row", ["check_kgb_golden", "check_kgb_nodecay",
                                                   "check_kgb_generator"]),
}


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_planted_mistake_is_caught(plant, tmp_path):
    path = orc_mod.compile_oracle(str(tmp_path / f"planted{plant}.so"), plant=plant, openmp=False)
    bad = orc_mod.Oracle(path)
    assert bad.planted() == plant
    _, must_fail = PLANTS[plant]
    for check in ALL_CHECKS:
        if check.__name__ in must_fail:
            with pytest.raises(AssertionError):
                check(bad)


def test_oracle_threads(oracle_lib):
    assert oracle_lib.num_threads() >= 1


# ------------------------------------------- the 32- and 16-token branches
@pytest.mark.parametrize("bt", [16, 32])
def test_small_chunk_branches(oracle_lib, bt):
    """Chunk length bt: nilpotent series per chunk, placement in both layouts, and
    the hand-worked cases embedded in a bt x bt identity."""
    orc = oracle_lib
    for name, n, M, X in _load_golden():
        got = orc.invert_chunk(M, n, bt=bt)
        assert got.shape == (bt, bt)
        assert np.array_equal(got[:n, :n], X) and np.array_equal(got[n:, n:], np.eye(bt - n)), name
    for kind, layout in (("gauss", "packed"), ("kda", "dense"), ("nodecay", "packed")):
        if layout == "packed":
            wl = ki.Workload("pin", "packed", H=2, in_dtype="f32", out_dtype="f32", seed=50 + bt,
                             seqlens=(5, 2 * bt + 3, 0, bt, 1), kind=kind, bt=bt)
        else:
            wl = ki.Workload("pin", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=60 + bt,
                             B=2, T=3 * bt - 5, kind=kind, bt=bt)
        inp = ki.build(wl)
        assert inp.A.shape[3] == bt
        A = orc_mod.to_f64(inp.A)
        got = orc.solve_tril(A, inp.cu_seqlens.numpy() if inp.cu_seqlens is not None else None)
        got = got.reshape(-1, inp.H, bt)
        want = _expected_layout(A.reshape(-1, inp.H, bt), inp.chunks(), inp.H)
        assert np.abs(got - want).max() <= 1e-12, (kind, layout)
