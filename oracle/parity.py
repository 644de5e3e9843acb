"""Parity criteria between the CUDA path and the fp64 oracle -- TEST INFRASTRUCTURE.

Tolerances (stated for this solver): against the exact inverse of the rounded
input, max |got - ref| <= tol * (1 + |ref|) with tol = 2e-5 for fp32 input and
1e-3 for bf16/fp16 input.  When the output itself is bf16/fp16 the reference
is first rounded to that dtype and one unit in its last place is added to the
bound (a correctly rounded bf16 value in [0.5, 1) can sit 2^-9 from the exact
value, more than 1e-3 * 1.5).  Structural entries -- the unit diagonal, the
zero upper triangle and the zero columns past a partial chunk's length -- must
be exact.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_IN = {torch.float32: 2e-5, torch.bfloat16: 1e-3, torch.float16: 1e-3}
MANT_BITS = {torch.bfloat16: 7, torch.float16: 10}
MIN_EXP = {torch.bfloat16: -126, torch.float16: -14}


def round_to(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """fp64 -> fp32 -> dtype, round to nearest even at each step, back to fp64."""
    return torch.from_numpy(ref.astype(np.float32)).to(dtype).to(torch.float64).numpy()


def ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Spacing of `dtype` numbers at |x| (subnormal spacing near zero)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, np.finfo(np.float64).tiny)))
    e = np.maximum(e, MIN_EXP[dtype])
    return np.ldexp(1.0, (e - MANT_BITS[dtype]).astype(np.int64))


def bound(ref: np.ndarray, in_dtype: torch.dtype, out_dtype: torch.dtype):
    """(reference to compare with, elementwise allowed |difference|)."""
    tol = TOL_IN[in_dtype] * (1.0 + np.abs(ref))
    if out_dtype == torch.float32:
        return ref, tol
    return round_to(ref, out_dtype), tol + ulp(ref, out_dtype)


def structure_mask(n: int, bt: int = 64) -> np.ndarray:
    """[n, bt] True where the output is structurally fixed (diagonal, j > i, j >= n)."""
    i = np.arange(n)[:, None]
    j = np.arange(bt)[None, :]
    return j >= i


def check_tile(got: np.ndarray, ref: np.ndarray, n: int, in_dtype, out_dtype):
    """got, ref: [n, bt] of one chunk-head of chunk length bt.  Returns (ok, max_excess, where)."""
    want, tol = bound(ref, in_dtype, out_dtype)
    st = structure_mask(n, got.shape[1])
    if not np.array_equal(got[st], ref[st]):
        return False, float("inf"), "structure"
    diff = np.abs(got - want)
    excess = diff - tol
    worst = float(np.max(excess)) if excess.size else -1.0
    if not np.all(np.isfinite(got)):
        return False, float("inf"), "non-finite"
    return worst <= 0.0, worst, "value"


def residual(M: np.ndarray, X: np.ndarray) -> float:
    """||(I + strict_lower(M)) X - I||_max for one n x n chunk."""
    n = X.shape[0]
    L = np.eye(n) + np.tril(M[:n, :n], -1)
    return float(np.abs(L @ X - np.eye(n)).max()) if n else 0.0


def residual_bound(M: np.ndarray, X: np.ndarray, out_dtype: torch.dtype) -> float:
    """1e-4 for fp32 output.  A bf16/fp16 output also carries its own rounding:
    each entry of X is off by up to half an ulp of the output dtype, which moves
    the residual by up to ||I + M||_inf * max(ulp(X)) / 2 (the exact inverse
    rounded to bf16 already exceeds 1e-4 on KDA inputs, and fp16 does so on
    inputs whose inverse has entries of order one)."""
    if out_dtype == torch.float32:
        return 1e-4
    n = X.shape[0]
    L = np.eye(n) + np.tril(M[:n, :n], -1)
    return 1e-4 + float(np.abs(L).sum(1).max()) * 0.5 * float(ulp(X, out_dtype).max())


def check_solution(got: np.ndarray, ref: np.ndarray, chunks, bt: int, in_dtype, out_dtype):
    """Whole-output verdict.  got, ref: [rows, H, bt] fp64 (the output as computed and
    the oracle's); chunks: (row0, n) of every chunk.  Rows in no chunk are not
    compared; in the others the structural entries (diagonal, above it, columns at
    or past n) must be equal exactly and every value finite and within bound().
    Returns (ok, message)."""
    rows = got.shape[0]
    i_in = np.full(rows, -1)
    for row0, n in chunks:
        i_in[row0:row0 + n] = np.arange(n)
    cov = i_in >= 0
    got, ref, i_in = got[cov], ref[cov], i_in[cov]
    struct = np.broadcast_to(np.arange(bt)[None, None, :] >= i_in[:, None, None], got.shape)
    if not np.array_equal(got[struct], ref[struct]):
        return False, "structural entries differ"
    if not np.all(np.isfinite(got)):
        return False, "non-finite output"
    want, tol = bound(ref, in_dtype, out_dtype)
    excess = np.abs(got - want) - tol
    if excess.size and excess.max() > 0:
        k = np.unravel_index(np.argmax(excess), excess.shape)
        return False, f"max excess {excess.max():.3g} at {k}: got {got[k]!r} ref {ref[k]!r}"
    return True, ""


def parts(inp, limit: int):
    """Independent parts of a solver input (a kda_inputs.SolverInput), each of at
    most `limit` chunk-heads where the layout allows: whole batch rows (dense) or
    whole requests (packed), so that the fp64 reference of one part fits in host
    memory.  Yields (first row, row count, A of the part, its cu_seqlens or None,
    its chunks as (row0, n) relative to the part)."""
    H, bt = inp.H, inp.bt
    chunks = inp.chunks()
    if inp.cu_seqlens is None:
        per_row = -(-inp.T // bt) * H if inp.T > 0 else 1
        step = max(1, limit // per_row)
        for b0 in range(0, inp.B, step):
            b1 = min(inp.B, b0 + step)
            lo, hi = b0 * inp.T, b1 * inp.T
            yield lo, hi - lo, inp.A[b0:b1], None, [(r0 - lo, n) for (r0, n) in chunks if lo <= r0 < hi]
        return
    cu = inp.cu_seqlens.tolist()
    s0 = 0
    while s0 < len(cu) - 1:
        s1, tasks = s0, 0
        while s1 < len(cu) - 1:
            t = -(-(cu[s1 + 1] - cu[s1]) // bt) * H
            if s1 > s0 and tasks + t > limit:
                break
            tasks += t
            s1 += 1
        lo, hi = cu[s0], cu[s1]
        sub_cu = torch.tensor([c - lo for c in cu[s0:s1 + 1]], dtype=torch.int32)
        yield lo, hi - lo, inp.A[:, lo:hi], sub_cu, [(r0 - lo, n) for (r0, n) in chunks if lo <= r0 < hi]
        s0 = s1


# ------------------------------------------------ TF32 precision mode bound
TF32_BOUND_SCALE = 2.0 ** -6


def tf32_bounds(A: np.ndarray, X: np.ndarray, chunks, bt: int = 64) -> np.ndarray:
    """Elementwise error bound of the TF32 precision mode, [rows, H, bt] fp64.

    A: the rounded input widened to fp64, X: the exact inverse (the oracle's), both
    [rows, H, bt]; chunks: (row0, n) of every chunk.  In that mode every 16x16
    merge product P Q is formed from P and Q truncated to TF32 (relative error below
    2^-10 each) with FP32 accumulation (16 terms), so it is off by at most
    (2^-9 + 2^-18 + 16 * 2^-24) |P| |Q| < 2^-8.9 |P| |Q|.  Every off-diagonal block of
    X is a chain of two such products (level A: X10 = -X11 A10 X00; level B:
    X_BL = -X_BR A_BL X_TL, whose factors X_TL and X_BR carry level A's error);
    to first order the error is at most 2 * 2^-8.9 (|X| |L| |X|) + 4 * 2^-8.9
    (|X| |L| |X| |L| |X|) elementwise, L the strictly lower A, which
    2^-6 * (M + M2) covers with room for the FP32 diagonal inverses.  Structural
    entries are not bounded here (they must be exact)."""
    rows, H, _ = A.shape
    out = np.zeros((rows, H, bt))
    for row0, n in chunks:
        if n == 0:
            continue
        La = np.abs(np.tril(A[row0:row0 + n, :, :n].transpose(1, 0, 2), -1))   # [H, n, n]
        Xa = np.abs(X[row0:row0 + n, :, :n].transpose(1, 0, 2))
        M = Xa @ La @ Xa
        M2 = M @ La @ Xa
        out[row0:row0 + n, :, :n] = (TF32_BOUND_SCALE * (M + M2)).transpose(1, 0, 2)
    return out


def check_solution_tf32(got: np.ndarray, ref: np.ndarray, A: np.ndarray, chunks, bt: int, out_dtype):
    """TF32-mode verdict: structural entries exact, values finite and within
    tf32_bounds() (plus the output dtype's rounding for bf16/fp16 output).
    Returns (ok, message, worst |got - ref| / bound)."""
    rows = got.shape[0]
    i_in = np.full(rows, -1)
    for row0, n in chunks:
        i_in[row0:row0 + n] = np.arange(n)
    cov = i_in >= 0
    tb = tf32_bounds(A, ref, chunks, bt)
    g, r, t, ii = got[cov], ref[cov], tb[cov], i_in[cov]
    struct = np.broadcast_to(np.arange(bt)[None, None, :] >= ii[:, None, None], g.shape)
    if not np.array_equal(g[struct], r[struct]):
        return False, "structural entries differ", float("inf")
    if not np.all(np.isfinite(g)):
        return False, "non-finite output", float("inf")
    want = r if out_dtype == torch.float32 else round_to(r, out_dtype)
    tol = t + (0.0 if out_dtype == torch.float32 else ulp(r, out_dtype)) + 1e-12
    ratio = np.abs(g - want) / tol
    worst = float(ratio[~struct].max()) if (~struct).any() else 0.0
    if worst > 1.0:
        k = np.unravel_index(np.argmax(np.where(struct, 0, ratio)), ratio.shape)
        return False, f"error {worst:.3g} x the bound at {k}: got {g[k]!r} ref {r[k]!r}", worst
    return True, "", worst
