"""The fused path (chunk matrix built on chip from keys, betas and decays, then
solved) against the fp64 oracle, element by element, through the C ABI.

Tolerance: 2e-5 * (1 + |ref|) for every input dtype (the oracle runs on the same
rounded k, g, beta), compared after rounding the reference to the output dtype
with one output ulp of slack; the structural entries (unit diagonal, zeros above
it and past a partial chunk's end) exactly.
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
DTYPES = [F32, BF16, F16]
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


def run(kda, x, out_dtype=F32, out=None):
    cu = x.cu_seqlens.to(DEV) if x.cu_seqlens is not None else None
    o = kda.solve_tril_kgb(x.k.to(DEV), x.g.to(DEV), x.beta.to(DEV), cu, out_dtype=out_dtype, out=out)
    torch.cuda.synchronize()
    return o


def reference(orc, x, return_A=False):
    return orc.solve_kgb(oracle.to_f64(x.k), oracle.to_f64(x.g), oracle.to_f64(x.beta),
                         x.cu_seqlens.numpy() if x.cu_seqlens is not None else None, return_A=return_A)


def check(x, got_t, ref, out_dtype, label):
    got = got_t.to(torch.float64).cpu().numpy().reshape(-1, x.H, 64)
    ok, msg = parity.check_solution(got, ref.reshape(-1, x.H, 64), x.chunks(), 64, F32, out_dtype)
    assert ok, f"{label}: {msg}"


@pytest.mark.parametrize("T", [1, 15, 16, 17, 33, 63, 64, 65, 130])
@pytest.mark.parametrize("H", [1, 3])
def test_kgb_dense_edges(kda, orc, T, H):
    x = ki.build_kgb(ki.Workload("e", "dense", H=H, in_dtype="f32", out_dtype="f32", seed=T * 5 + H, B=2, T=T))
    check(x, run(kda, x), reference(orc, x), F32, f"T={T} H={H}")


@pytest.mark.parametrize("in_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("out_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("kind", ["kda", "nodecay"])
def test_kgb_dtype_matrix_packed(kda, orc, in_dtype, out_dtype, kind):
    x = ki.build_kgb(ki.Workload("dt", "packed", H=4, in_dtype=NAMES[in_dtype], out_dtype=NAMES[out_dtype],
                                 seed=19, seqlens=(1, 63, 64, 65, 200, 0, 128, 7), kind=kind))
    check(x, run(kda, x, out_dtype), reference(orc, x), out_dtype, f"{in_dtype}->{out_dtype} {kind}")


@pytest.mark.parametrize("K", [32, 64, 96])
def test_kgb_key_dims(kda, orc, K):
    x = ki.build_kgb(ki.Workload("kd", "packed", H=3, in_dtype="bf16", out_dtype="f32", seed=K,
                                 seqlens=(70, 64, 5)), K=K)
    check(x, run(kda, x), reference(orc, x), F32, f"K={K}")


def test_kgb_decay_closed_form(kda):
    """One-hot keys, beta = 1, g_t = -lam t: (I + A)^-1 = I - exp(-lam) S in every chunk."""
    lam, T, H, K = 0.4, 150, 2, 128
    k = torch.zeros(1, T, H, K)
    k[..., 0] = 1.0
    g = (-lam * torch.arange(T, dtype=torch.float64)).float()[None, :, None, None].expand(1, T, H, K).contiguous()
    beta = torch.ones(1, T, H)
    out = kda.solve_tril_kgb(k.to(DEV), g.to(DEV), beta.to(DEV))
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()[0]
    r = np.exp(-lam)
    for t0 in range(0, T, 64):
        n = min(64, T - t0)
        want = np.eye(n) - r * np.eye(n, k=-1)
        for h in range(H):
            assert np.abs(got[t0:t0 + n, h, :n] - want).max() <= 2e-6, (t0, h)
            assert np.all(got[t0:t0 + n, h, n:] == 0)


def test_kgb_large_decay_offset(kda, orc):
    """g may run on across chunks: a large per-channel offset (rounded to fp32 in
    the input the oracle also sees) changes nothing beyond the tolerance."""
    x = ki.build_kgb(ki.Workload("off", "packed", H=3, in_dtype="f32", out_dtype="f32", seed=12,
                                 seqlens=(64, 100, 17)))
    off = torch.from_numpy(np.random.default_rng(5).uniform(-900, -300, (1, 1, 3, 128)).astype(np.float32))
    y = ki.KgbInput(x.workload, x.k, (x.g + off).contiguous(), x.beta, x.cu_seqlens, x.seqlens)
    check(y, run(kda, y), reference(orc, y), F32, "offset")


def _block_spans(x):
    """Per-channel fall of g over every 16-row block of every chunk (nats)."""
    g = x.g.double().numpy().reshape(-1, x.H, x.K)
    spans = []
    for row0, n in x.chunks():
        for r in range(0, n, 16):
            e = min(r + 15, n - 1)
            spans.append(g[row0 + r] - g[row0 + e])
    return np.stack(spans)


STEEP_CASES = {
    "packed": dict(layout="packed", seqlens=(1, 17, 64, 100, 0, 130, 33)),
    "dense": dict(layout="dense", B=2, T=130),
}


@pytest.mark.parametrize("in_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", list(STEEP_CASES))
def test_kgb_steep_decays(kda, orc, in_dtype, case):
    """Decays that fall 3 to 20 nats per token, and cliffs of 100 nats: blocks fall
    far past FP32's exponent range (a factorisation through one reference row
    overflows there), while the terms of nearby rows stay large."""
    wl = ki.Workload("steep", H=3, in_dtype=NAMES[in_dtype], out_dtype="f32", seed=23, kind="steep",
                     **STEEP_CASES[case])
    x = ki.build_kgb(wl)
    spans = _block_spans(x)
    assert spans.max() > 400 and np.mean(spans > 80) > 0.4        # the inputs do what they claim
    out = run(kda, x)
    assert torch.isfinite(out).all()
    check(x, out, reference(orc, x), F32, f"steep {case} {in_dtype}")


@pytest.mark.parametrize("out_dtype", DTYPES, ids=str)
def test_kgb_steep_decays_full_size(kda, orc, out_dtype):
    """The 16 x 512-token, 64-head shape with steep decays, every element."""
    wl = ki.WORKLOADS["packed_16x512_h64_f32"].with_(kind="steep", out_dtype=NAMES[out_dtype], seed=29)
    x = ki.build_kgb(wl)
    check(x, run(kda, x, out_dtype), reference(orc, x), out_dtype, f"steep full size -> {out_dtype}")


def test_kgb_decays_near_the_safe_span(kda, orc):
    """Every channel decaying about 1.45 nats per token, so that g reaches about 46
    nats from the chunk's middle at its ends: the tensor-core product's factors
    carry exponents near the largest it accepts (channels just past it take the
    slow path)."""
    T, H, K = 200, 3, 128
    rng = np.random.default_rng(17)
    k = rng.standard_normal((1, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    t = np.arange(T) % 64
    g = -1.45 * t[None, :, None, None] * rng.uniform(0.9, 1.1, (1, 1, H, K))
    beta = 1 / (1 + np.exp(-rng.standard_normal((1, T, H))))
    wl = ki.Workload("near", "dense", H=H, in_dtype="f32", out_dtype="f32", seed=0, B=1, T=T)
    x = ki.KgbInput(wl, torch.from_numpy(k.astype(np.float32)), torch.from_numpy(g.astype(np.float32)),
                    torch.from_numpy(beta.astype(np.float32)), None, [T])
    check(x, run(kda, x), reference(orc, x), F32, "near the safe span")


def test_kgb_residual(kda, orc):
    x = ki.build_kgb(ki.Workload("res", "packed", H=4, in_dtype="f32", out_dtype="f32", seed=31,
                                 seqlens=(64, 100, 33)))
    got = run(kda, x).double().cpu().numpy().reshape(-1, x.H, 64)
    _, A = reference(orc, x, return_A=True)
    A = A.reshape(-1, x.H, 64)
    for row0, n in x.chunks():
        for h in range(x.H):
            M = A[row0:row0 + n, h, :n]
            X = got[row0:row0 + n, h, :n]
            assert parity.residual(M, X) <= parity.residual_bound(M, X, F32), (row0, h)


SENTINEL = {F32: 0x7FC0DEAD, BF16: 0x7FDE, F16: 0x7EAD}
INT_VIEW = {F32: torch.int32, BF16: torch.int16, F16: torch.int16}


@pytest.mark.parametrize("out_dtype", DTYPES, ids=str)
def test_kgb_guard_band_canaries(kda, out_dtype):
    x = ki.build_kgb(ki.Workload("c", "packed", H=3, in_dtype="f32", out_dtype="f32", seed=3,
                                 seqlens=(7, 64, 90, 0, 1)))
    pad = 4096
    n = x.B * x.T * x.H * 64
    buf = torch.full((pad + n + pad,), SENTINEL[out_dtype], dtype=INT_VIEW[out_dtype], device=DEV)
    out = buf[pad:pad + n].view(out_dtype).view(x.B, x.T, x.H, 64)
    run(kda, x, out_dtype, out=out)
    assert torch.all(buf[:pad] == SENTINEL[out_dtype]) and torch.all(buf[pad + n:] == SENTINEL[out_dtype])
    assert not torch.any(buf[pad:pad + n] == SENTINEL[out_dtype])


def test_kgb_packed_equals_dense_and_deterministic(kda):
    lens = (5, 64, 130, 1, 77)
    wl = ki.Workload("pd", "packed", H=4, in_dtype="bf16", out_dtype="f32", seed=8, seqlens=lens)
    x = ki.build_kgb(wl)
    out = run(kda, x)
    for _ in range(2):
        assert torch.equal(out, run(kda, x))
    cu = x.cu_seqlens.tolist()
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        d = ki.KgbInput(wl.with_(layout="dense", T=lens[s]), x.k[:, sl].contiguous(), x.g[:, sl].contiguous(),
                        x.beta[:, sl].contiguous(), None, [lens[s]])
        assert torch.equal(run(kda, d)[0], out[0, sl]), s


@pytest.mark.parametrize("name", ["packed_16x512_h64_f32", "packed_ragged37_h32_bf16"])
def test_kgb_specified_shapes(kda, orc, name):
    """The specified workloads' shapes with keys of 128 channels, every element."""
    wl = ki.WORKLOADS[name]
    x = ki.build_kgb(wl)
    out_dtype = ki.torch_dtype(wl.out_dtype)
    check(x, run(kda, x, out_dtype), reference(orc, x), out_dtype, name)


def test_kgb_argument_errors(kda):
    x = ki.build_kgb(ki.Workload("a", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=1, B=1, T=64), K=32)
    k, g, b = x.k.to(DEV), x.g.to(DEV), x.beta.to(DEV)
    with pytest.raises(ValueError):
        kda.solve_tril_kgb(k, g.half(), b)                     # g must be float32
    with pytest.raises(ValueError):
        kda.solve_tril_kgb(k, g, b.half())                     # beta's dtype must match k's
    with pytest.raises(kda.KdaError) as e:
        kda.solve_tril_kgb(k[..., :16].contiguous(), g[..., :16].contiguous(), b)
    assert e.value.status == 2


def test_kgb_no_device_error_recorded(kda):
    """No bounded wait of the fused kernel ran out during this module."""
    assert kda.device_error(0) == 0
