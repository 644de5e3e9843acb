"""Where the fused path's tolerance comes from (CPU only).

The fused kernel builds each chunk's matrix in FP32 from keys, decays and betas
with one reference value c_d per channel (g of the chunk's middle live row):

* Q = k 2^{(g - c) log2 e} and P = k 2^{(c - g) log2 e}, the difference g - c
  taken first and then scaled, so the exponent's error grows with its size but
  not with |g|;
* A = beta * strict_lower(Q P^T), the product taken in split TF32 on the tensor
  cores (Qh Ph^T + Qh Pl^T + Ql Ph^T, FP32 sums): the hi parts truncated to
  TF32, the lo parts the exact FP32 remainders, which the tensor cores read as
  TF32 (modelled both truncated and rounded to nearest);
* a channel whose g leaves [c - 48, c + 48] over the chunk's live rows is left
  out of the product and its terms k_i k_j exp(g_i - g_j) are added one by one.

This test runs that arithmetic in numpy float32 and compares it with the fp64
oracle on the same rounded inputs: the worst error must sit far inside the
2e-5 * (1 + |ref|) the GPU parity tests use for every input dtype, on KDA
decays, on no decay, and on steep decays (per-token drops of 3 to 20 nats and
cliffs of 100 nats), and on decays that take the factors' exponents near the
largest the product accepts.  A planted copy without the steep channels' slow
path must fail on the steep inputs.
"""
import numpy as np
import pytest

import kda_inputs as ki
import oracle

BT = 64
SAFE = 48.0               # nats of g from the channel's reference that the product takes
L2E = 1.4426950408889634


def _tf32(x):
    """Truncate float32 values to TF32 (10 explicit mantissa bits)."""
    return (np.asarray(x, np.float32).view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)


def _tf32_rn(x):
    """Round float32 values to the nearest TF32 value (ties to even)."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0xFFF) + ((b >> np.uint64(13)) & np.uint64(1))) & np.uint64(0xFFFFE000)
    return b.astype(np.uint32).view(np.float32)


def _fp32_construction(k, g, beta, n, steep_path=True, lo_read=_tf32):
    """FP32 A [n, n] of one chunk-head by the single-reference factorisation."""
    f32 = np.float32
    k = k.astype(f32)
    g = g.astype(f32)
    ref = g[(n - 1) // 2]
    keep = ((g[0] - ref) * f32(L2E) <= f32(SAFE * L2E)) & ((ref - g[n - 1]) * f32(L2E) <= f32(SAFE * L2E))
    if not steep_path:
        keep = np.ones_like(keep)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        e = ((g - ref).astype(f32) * f32(L2E)).astype(f32)
        Q = np.where(keep, k * np.exp2(e), 0).astype(f32)
        P = np.where(keep, k * np.exp2(-e), 0).astype(f32)
        Qh, Ph = _tf32(Q), _tf32(P)
        Ql, Pl = lo_read((Q - Qh).astype(f32)), lo_read((P - Ph).astype(f32))
        D = (Qh.astype(np.float64) @ Ph.T.astype(np.float64) + Qh.astype(np.float64) @ Pl.T.astype(np.float64)
             + Ql.astype(np.float64) @ Ph.T.astype(np.float64)).astype(f32)
        for dch in np.nonzero(~keep)[0]:
            kc, gc = k[:, dch], g[:, dch]
            D = (D + (kc[:, None] * kc[None, :]) * np.exp((gc[:, None] - gc[None, :]).astype(f32)).astype(f32)
                 ).astype(f32)
    return (np.tril(D, -1) * np.asarray(beta[:n], f32)[:, None]).astype(f32)


def _fp32_solve(A):
    n = A.shape[0]
    X = np.zeros((n, n), np.float32)
    for j in range(n):
        X[j, j] = 1.0
        for i in range(j + 1, n):
            X[i, j] = -np.float32(np.dot(A[i, j:i], X[j:i, j]))
    return X


def _worst(kind, in_dtype, **kw):
    wl = ki.Workload("tol", "packed", H=3, in_dtype=in_dtype, out_dtype="f32", seed=5,
                     seqlens=(64, 64, 40, 7), kind=kind)
    x = ki.build_kgb(wl)
    k, g, b = (oracle.to_f64(t) for t in (x.k, x.g, x.beta))
    ref = oracle.get().solve_kgb(k, g, b, x.cu_seqlens.numpy())[0]
    worst = 0.0
    with np.errstate(invalid="ignore", over="ignore"):
        for row0, n in x.chunks():
            for h in range(x.H):
                A = _fp32_construction(k[0, row0:row0 + n, h], g[0, row0:row0 + n, h], b[0, row0:row0 + n, h], n,
                                       **kw)
                X = _fp32_solve(A)
                R = ref[row0:row0 + n, h, :n]
                err = np.abs(X - R) / (1 + np.abs(R))
                worst = max(worst, float(np.inf if not np.all(np.isfinite(err)) else np.max(err)))
    return worst


@pytest.mark.parametrize("kind", ["kda", "nodecay", "steep"])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lo_read", [_tf32, _tf32_rn], ids=["lo_truncated", "lo_rounded"])
def test_fp32_construction_is_far_inside_the_tolerance(kind, in_dtype, lo_read):
    worst = _worst(kind, in_dtype, lo_read=lo_read)
    assert worst <= 2e-5 / 100, worst


def test_tf32_rounding_helpers():
    x = np.array([1.0, 1.0 + 2.0 ** -10, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -12,
                  -1.5 - 2.0 ** -11, 1.0 + 2.0 ** -11 + 2.0 ** -13], np.float32)
    assert _tf32(x).tolist() == [1.0, 1.0 + 2.0 ** -10, 1.0, 1.0 + 2.0 ** -10, 1.0, -1.5, 1.0]
    # ties go to the even TF32 neighbour; below half rounds down, above half up
    assert _tf32_rn(x).tolist() == [1.0, 1.0 + 2.0 ** -10, 1.0, 1.0 + 2.0 ** -9, 1.0, -1.5, 1.0 + 2.0 ** -10]


def test_steep_channels_need_their_slow_path():
    assert _worst("steep", "f32", steep_path=False) > 2e-5


def test_decays_near_the_safe_span():
    """Every channel decaying about 1.45 nats per token: g reaches about 46 nats from
    the reference at the chunk's ends, near the span the product takes (some
    channels just past it take the slow path), so the factors carry exponents
    near their largest."""
    rng = np.random.default_rng(1)
    orc = oracle.get()
    worst = 0.0
    for _ in range(4):
        k = rng.standard_normal((64, 128))
        k /= np.linalg.norm(k, axis=1, keepdims=True)
        k = k.astype(np.float32).astype(np.float64)
        g = (-1.45 * np.arange(64)[:, None] * rng.uniform(0.9, 1.1, (1, 128))).astype(np.float32).astype(np.float64)
        b = (1 / (1 + np.exp(-rng.standard_normal(64)))).astype(np.float32).astype(np.float64)
        ref = orc.solve_kgb(k[None, :, None], g[None, :, None], b[None, :, None])[0][:, 0, :]
        X = _fp32_solve(_fp32_construction(k, g, b, 64))
        worst = max(worst, float(np.max(np.abs(X - ref) / (1 + np.abs(ref)))))
    assert worst <= 2e-5 / 100, worst
