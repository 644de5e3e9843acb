"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Axes (LightLLM PR #1703 regression-tests the layouts, the dtypes, the precision
modes and the fallbacks): layout {dense, packed} x input
dtype x output dtype x path {auto, split, single}, shape edges, the specified
workloads at full size, exact structures, NaN poisoning of ignored elements,
guard-band canaries, and bitwise equalities between paths and layouts.
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


DEV = "cuda:0"


def to_dev(inp):
    A = inp.A.to(DEV)
    cu = inp.cu_seqlens.to(DEV) if inp.cu_seqlens is not None else None
    return A, cu


def row_geometry(inp):
    """Per flattened row: (row index inside its chunk, chunk length); -1 for rows in no chunk."""
    rows = inp.B * inp.T
    i_in = np.full(rows, -1, dtype=np.int64)
    n_of = np.zeros(rows, dtype=np.int64)
    for row0, n in inp.chunks():
        i_in[row0:row0 + n] = np.arange(n)
        n_of[row0:row0 + n] = n
    return i_in, n_of


def check_full(inp, got_t, ref, out_dtype, label=""):
    """Every output element against the oracle (oracle.parity.check_solution)."""
    H, bt = inp.H, inp.bt
    got = got_t.to(torch.float64).cpu().numpy().reshape(-1, H, bt)
    ok, msg = parity.check_solution(got, ref.reshape(-1, H, bt), inp.chunks(), bt, inp.A.dtype, out_dtype)
    assert ok, f"{label}: {msg}"


def check_residuals(inp, got_t, out_dtype, limit=2048, seed=0):
    """||(I + M) X - I||_max per chunk-head on up to `limit` sampled chunk-heads."""
    H, bt = inp.H, inp.bt
    A = oracle.to_f64(inp.A).reshape(-1, H, bt)
    got = got_t.to(torch.float64).cpu().numpy().reshape(-1, H, bt)
    tasks = [(r, n, h) for (r, n) in inp.chunks() for h in range(H)]
    rng = np.random.default_rng(seed)
    if len(tasks) > limit:
        tasks = [tasks[i] for i in rng.choice(len(tasks), limit, replace=False)]
    for r, n, h in tasks:
        M = A[r:r + n, h, :n]
        X = got[r:r + n, h, :n]
        assert parity.residual(M, X) <= parity.residual_bound(M, X, out_dtype), (r, n, h)


def solve(kda, inp, out_dtype, path):
    A, cu = to_dev(inp)
    out, taken = kda.solve_tril(A, cu, out_dtype=out_dtype, path=path, return_path=True)
    torch.cuda.synchronize()
    return out, taken


def oracle_ref(orc, inp):
    return orc.solve_tril(oracle.to_f64(inp.A), inp.cu_seqlens.numpy() if inp.cu_seqlens is not None else None)


# ------------------------------------------------------------ small shapes

EDGE_T = [1, 15, 16, 17, 31, 33, 48, 63, 64, 65, 127, 128, 130]


@pytest.mark.parametrize("T", EDGE_T)
@pytest.mark.parametrize("H", [1, 3])
def test_dense_edges(kda, orc, T, H):
    inp = ki.build(ki.Workload("edge", "dense", H=H, in_dtype="f32", out_dtype="f32", seed=T * 7 + H,
                               B=2, T=T, kind="gauss"))
    ref = oracle_ref(orc, inp)
    outs = {}
    for path in ("single", "split"):
        out, taken = solve(kda, inp, F32, path)
        assert taken == path
        check_full(inp, out, ref, F32, f"T={T} H={H} {path}")
        outs[path] = out
    assert torch.equal(outs["single"], outs["split"])


DTYPES = [F32, BF16, F16]


@pytest.mark.parametrize("in_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("out_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("kind", ["kda", "gauss", "nodecay"])
def test_dtype_matrix_packed(kda, orc, in_dtype, out_dtype, kind):
    names = {F32: "f32", BF16: "bf16", F16: "f16"}
    inp = ki.build(ki.Workload("dt", "packed", H=4, in_dtype=names[in_dtype], out_dtype=names[out_dtype],
                               seed=17, seqlens=(1, 63, 64, 65, 200, 0, 128, 7), kind=kind))
    ref = oracle_ref(orc, inp)
    outs = {}
    for path in ("single", "split"):
        out, taken = solve(kda, inp, out_dtype, path)
        check_full(inp, out, ref, out_dtype, f"{in_dtype}->{out_dtype} {kind} {path}")
        outs[path] = out
    assert torch.equal(outs["single"], outs["split"])
    check_residuals(inp, outs["single"], out_dtype)


@pytest.mark.parametrize("lens", [
    (0, 0, 5, 0),                      # zero-length requests
    (1,) * 40,                         # all requests one row long
    (3000,),                           # one long request
    tuple(range(1, 70)),               # every partial length
])
def test_packed_edges(kda, orc, lens):
    inp = ki.build(ki.Workload("pe", "packed", H=2, in_dtype="bf16", out_dtype="f32", seed=len(lens),
                               seqlens=lens, kind="gauss"))
    ref = oracle_ref(orc, inp)
    for path in ("single", "split", "auto"):
        out, _ = solve(kda, inp, F32, path)
        check_full(inp, out, ref, F32, f"{lens[:4]} {path}")


# ------------------------------------------------- exact structures (bitwise)

def _exact_inputs():
    rng = np.random.default_rng(5)
    cases = {}
    I = np.eye(64)
    cases["zero"] = np.zeros((64, 64))
    cases["ones"] = np.tril(np.ones((64, 64)), -1)
    cases["bidiag_half"] = np.diag(np.full(63, 0.5), -1)
    bd = np.zeros((64, 64))
    for b in range(4):
        bd[16 * b:16 * b + 16, 16 * b:16 * b + 16] = np.tril(rng.integers(-2, 3, (16, 16)) * 0.25, -1)
    cases["blockdiag"] = bd
    for p in range(4):
        for q in range(p):
            M = np.zeros((64, 64))
            M[16 * p:16 * p + 16, 16 * q:16 * q + 16] = rng.integers(-3, 4, (16, 16)) * 0.5
            cases[f"block{p}{q}"] = M
    for chain in ([(1, 0), (2, 1)], [(2, 1), (3, 2)], [(1, 0), (2, 1), (3, 2)], [(3, 1), (1, 0)],
                  [(2, 0), (3, 2)]):
        M = np.zeros((64, 64))
        for p, q in chain:
            M[16 * p:16 * p + 16, 16 * q:16 * q + 16] = (
                rng.integers(-1, 2, (16, 16)) * 2.0 ** -rng.integers(0, 3, (16, 16)))
        cases["chain" + "".join(f"{p}{q}" for p, q in chain)] = M
    del I
    return cases


EXACT = _exact_inputs()


@pytest.mark.parametrize("name", sorted(EXACT))
def test_exact_structures_bitwise(kda, orc, name):
    M = EXACT[name]
    A = torch.from_numpy(M.astype(np.float32)).reshape(1, 64, 1, 64).contiguous()
    inp = ki.SolverInput(ki.Workload("exact", "dense", H=1, in_dtype="f32", out_dtype="f32", seed=0, T=64),
                         A, None, [64])
    ref = oracle_ref(orc, inp)[0, :, 0, :]
    for path in ("single", "split"):
        out, _ = solve(kda, inp, F32, path)
        got = out.cpu().numpy()[0, :, 0, :].astype(np.float64)
        assert np.array_equal(got, ref), (name, path, np.abs(got - ref).max())


# ------------------------------------------------------ robustness checks

def test_poisoned_ignored_elements(kda):
    wl = ki.Workload("poison", "packed", H=3, in_dtype="f32", out_dtype="f32", seed=23,
                     seqlens=(5, 64, 100, 1, 70))
    clean, dirty = ki.build(wl), ki.build(wl, poison=True)
    for path in ("single", "split"):
        a, _ = solve(kda, clean, F32, path)
        b, _ = solve(kda, dirty, F32, path)
        assert torch.equal(a, b), path
    wl = wl.with_(layout="dense", seqlens=None, B=2, T=77, in_dtype="bf16")
    clean, dirty = ki.build(wl), ki.build(wl, poison=True)
    for path in ("single", "split"):
        a, _ = solve(kda, clean, F32, path)
        b, _ = solve(kda, dirty, F32, path)
        assert torch.equal(a, b), path


SENTINEL = {F32: 0x7FC0DEAD, BF16: 0x7FDE, F16: 0x7EAD}
INT_VIEW = {F32: torch.int32, BF16: torch.int16, F16: torch.int16}


@pytest.mark.parametrize("out_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("layout", ["dense", "packed"])
def test_guard_band_canaries(kda, out_dtype, layout):
    """Output and workspace between sentinel-filled guard bands: nothing outside is
    written, everything inside is."""
    if layout == "dense":
        wl = ki.Workload("canary", "dense", H=3, in_dtype="f32", out_dtype="f32", seed=3, B=2, T=81)
    else:
        wl = ki.Workload("canary", "packed", H=3, in_dtype="f32", out_dtype="f32", seed=3,
                         seqlens=(7, 64, 90, 0, 1))
    inp = ki.build(wl)
    A, cu = to_dev(inp)
    pad = 4096
    n = A.numel()
    iv = INT_VIEW[out_dtype]
    buf = torch.full((pad + n + pad,), SENTINEL[out_dtype], dtype=iv, device=DEV)
    out = buf[pad:pad + n].view(out_dtype).view(A.shape)
    need = kda.workspace_size(inp.B, inp.T, inp.H, 0 if cu is None else cu.numel() - 1)
    wpad = 4096
    wbuf = torch.full((wpad + need + wpad,), 0x5A, dtype=torch.uint8, device=DEV)
    ws = wbuf[wpad:wpad + need]
    for path in ("single", "split"):
        buf[pad:pad + n] = SENTINEL[out_dtype]
        kda.solve_tril(A, cu, out_dtype=out_dtype, path=path, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == SENTINEL[out_dtype]) and torch.all(buf[pad + n:] == SENTINEL[out_dtype])
        assert not torch.any(buf[pad:pad + n] == SENTINEL[out_dtype]), path
        assert torch.all(wbuf[:wpad] == 0x5A) and torch.all(wbuf[wpad + need:] == 0x5A)


def test_packed_equals_dense_per_request(kda):
    lens = (5, 64, 130, 1, 77)
    wl = ki.Workload("pd", "packed", H=4, in_dtype="bf16", out_dtype="f32", seed=8, seqlens=lens)
    inp = ki.build(wl)
    out, _ = solve(kda, inp, F32, "single")
    cu = inp.cu_seqlens.tolist()
    for s in range(len(lens)):
        sub = inp.A[:, cu[s]:cu[s + 1]].contiguous()
        d = ki.SolverInput(wl.with_(layout="dense", T=lens[s]), sub, None, [lens[s]])
        o, _ = solve(kda, d, F32, "single")
        assert torch.equal(o[0], out[0, cu[s]:cu[s + 1]]), s


def test_deterministic_repeats(kda):
    inp = ki.build(ki.Workload("det", "packed", H=8, in_dtype="f16", out_dtype="bf16", seed=9,
                               seqlens=(300, 64, 17, 1000)))
    a, _ = solve(kda, inp, BF16, "single")
    for _ in range(3):
        b, _ = solve(kda, inp, BF16, "single")
        assert torch.equal(a, b)
        c, _ = solve(kda, inp, BF16, "split")
        assert torch.equal(a, c)


def test_selector_fallbacks(kda):
    # many tiny requests: the workspace would exceed the FP32 input -> single pass
    lens = tuple(int(x) for x in np.random.default_rng(1).integers(1, 9, size=512))
    inp = ki.build(ki.Workload("tiny", "packed", H=4, in_dtype="bf16", out_dtype="f32", seed=1, seqlens=lens))
    out, taken = solve(kda, inp, F32, "auto")
    assert taken == "single"
    # forced split with a too-small workspace is an error, not a silent fallback
    A, cu = to_dev(inp)
    small = torch.empty(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(kda.KdaError) as e:
        kda.solve_tril(A, cu, path="split", workspace=small)
    assert e.value.status == 3
    # auto with an insufficient workspace falls back to single pass
    out2, taken = kda.solve_tril(A, cu, path="auto", workspace=small, return_path=True)
    torch.cuda.synchronize()
    assert taken == "single" and torch.equal(out, out2)


def test_host_entry_point(kda):
    inp = ki.build(ki.Workload("host", "packed", H=4, in_dtype="bf16", out_dtype="f32", seed=12,
                               seqlens=(100, 64, 3)))
    A, cu = to_dev(inp)
    ref, _ = solve(kda, inp, F32, "auto")
    A_host = inp.A.pin_memory()
    cu_host = inp.cu_seqlens.pin_memory()
    Ai_host = torch.empty(inp.A.shape, dtype=F32).pin_memory()
    A_dev = torch.empty_like(A)
    Ai_dev = torch.empty(inp.A.shape, dtype=F32, device=DEV)
    cu_dev = torch.empty_like(cu)
    kda.solve_tril_host(A_host, Ai_host, A_dev, Ai_dev, cu_host, cu_dev)
    torch.cuda.synchronize()
    assert torch.equal(Ai_host, ref.cpu())


HOST_PIPELINE_CASES = {
    # > 32 MiB of copies: cut into pieces at request / batch-row / 64-row boundaries
    "packed_16x512_f32": ki.WORKLOADS["packed_16x512_h64_f32"],
    "packed_zero_len": ki.Workload("hp", "packed", H=64, in_dtype="f32", out_dtype="f32", seed=31,
                                   seqlens=(0, 700, 1, 0, 2500, 64, 0, 999, 1500, 3)),
    "dense_b1_f16": ki.Workload("hd1", "dense", H=64, in_dtype="f16", out_dtype="bf16", seed=32, B=1, T=8000),
    "dense_b3_f32": ki.Workload("hd3", "dense", H=32, in_dtype="f32", out_dtype="f32", seed=33, B=3, T=4000),
}


@pytest.mark.parametrize("name", sorted(HOST_PIPELINE_CASES))
def test_host_entry_point_pipelined(kda, name):
    wl = HOST_PIPELINE_CASES[name]
    inp = ki.build(wl)
    out_dtype = ki.torch_dtype(wl.out_dtype)
    ref, _ = solve(kda, inp, out_dtype, "auto")
    A, cu = to_dev(inp)
    A_host = inp.A.pin_memory()
    cu_host = inp.cu_seqlens.pin_memory() if cu is not None else None
    for _ in range(2):                                   # reused copy streams and events
        Ai_host = torch.full(inp.A.shape, float("nan"), dtype=out_dtype).pin_memory()
        A_dev = torch.empty_like(A)
        Ai_dev = torch.empty(inp.A.shape, dtype=out_dtype, device=DEV)
        cu_dev = torch.empty_like(cu) if cu is not None else None
        kda.solve_tril_host(A_host, Ai_host, A_dev, Ai_dev, cu_host, cu_dev)
        torch.cuda.current_stream().synchronize()       # the caller's stream covers the whole call
        assert torch.equal(Ai_host, ref.cpu()), name


def test_no_device_error_recorded(kda):
    assert kda.device_error(0) == 0


# ------------------------------------------------- the specified workloads

_CACHE = {}


def workload_input(name):
    if name not in _CACHE:
        _CACHE.clear()
        _CACHE[name] = ki.build(ki.WORKLOADS[name])
    return _CACHE[name]


EXPECTED_AUTO = {name: "single" for name in ki.WORKLOADS}     # split never paid on GB300


@pytest.mark.parametrize("name", list(ki.WORKLOADS))
def test_specified_workloads(kda, orc, name):
    inp = workload_input(name)
    wl = inp.workload
    out_dtype = ki.torch_dtype(wl.out_dtype)
    outs = {}
    for path in ("auto", "single", "split"):
        out, taken = solve(kda, inp, out_dtype, path)
        if path == "auto":
            assert taken == EXPECTED_AUTO[name]
        outs[path] = out
    assert torch.equal(outs["single"], outs["split"])
    assert torch.equal(outs["auto"], outs["single"])
    check_large(orc, inp, outs["auto"], out_dtype, name)


def check_large(orc, inp, got, out_dtype, name, slab_limit=40000):
    """Every output element against the oracle, run part by part (whole batch rows
    or whole requests of at most `slab_limit` chunk-heads) so that the fp64
    reference of a part fits in host memory; and residuals of sampled chunk-heads."""
    H, bt = inp.H, inp.bt
    g = got.view(-1, H, bt)
    for r0, nrows, A_sub, cu_sub, sub_chunks in parity.parts(inp, slab_limit):
        ref = orc.solve_tril(oracle.to_f64(A_sub), cu_sub.numpy() if cu_sub is not None else None)
        got_sub = g[r0:r0 + nrows].to(torch.float64).cpu().numpy()
        ok, msg = parity.check_solution(got_sub, ref.reshape(-1, H, bt), sub_chunks, bt, inp.A.dtype, out_dtype)
        assert ok, f"{name} rows {r0}..{r0 + nrows}: {msg}"
        del ref, got_sub
    check_residuals(inp, got, out_dtype, limit=1024)


# ------------------------------------------- 16- and 32-token chunk lengths

SMALL_BT = [16, 32]
SMALL_EDGE_T = [1, 2, 15, 16, 17, 31, 32, 33, 47, 48, 63, 64, 65, 100]
NAMES = {F32: "f32", BF16: "bf16", F16: "f16"}


@pytest.mark.parametrize("bt", SMALL_BT)
@pytest.mark.parametrize("T", SMALL_EDGE_T)
@pytest.mark.parametrize("H", [1, 3])
def test_small_chunks_dense_edges(kda, orc, bt, T, H):
    inp = ki.build(ki.Workload("edge", "dense", H=H, in_dtype="f32", out_dtype="f32", seed=T * 11 + H + bt,
                               B=2, T=T, kind="gauss", bt=bt))
    ref = oracle_ref(orc, inp)
    out, taken = solve(kda, inp, F32, "auto")
    assert taken == "single"
    check_full(inp, out, ref, F32, f"bt={bt} T={T} H={H}")
    check_residuals(inp, out, F32)


@pytest.mark.parametrize("bt", SMALL_BT)
@pytest.mark.parametrize("in_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("out_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("kind", ["kda", "gauss", "nodecay"])
def test_small_chunks_dtype_matrix_packed(kda, orc, bt, in_dtype, out_dtype, kind):
    inp = ki.build(ki.Workload("dt", "packed", H=4, in_dtype=NAMES[in_dtype], out_dtype=NAMES[out_dtype],
                               seed=29 + bt, seqlens=(1, 15, 16, 17, 31, 32, 33, 200, 0, 7), kind=kind, bt=bt))
    ref = oracle_ref(orc, inp)
    out, _ = solve(kda, inp, out_dtype, "single")
    check_full(inp, out, ref, out_dtype, f"bt={bt} {in_dtype}->{out_dtype} {kind}")
    check_residuals(inp, out, out_dtype)


@pytest.mark.parametrize("bt", SMALL_BT)
@pytest.mark.parametrize("kind", ["identity", "unit_subdiag"])
def test_small_chunks_exact_structures(kda, orc, bt, kind):
    """A = 0 gives exactly I; A = unit subdiagonal gives exactly (-1)^(i-j) below
    the diagonal (integers, exact in every dtype and in split TF32)."""
    T = 3 * bt - 5
    a = torch.zeros(1, T, 2, bt, dtype=torch.float32)
    if kind == "unit_subdiag":
        for r in range(T):
            i = r % bt
            if i > 0:
                a[0, r, :, i - 1] = 1.0
    for dt in DTYPES:
        wl = ki.Workload("exact", "dense", H=2, in_dtype=NAMES[dt], out_dtype="f32", seed=0, B=1, T=T, bt=bt)
        inp = ki.SolverInput(wl, a.to(dt).contiguous(), None, [T])
        ref = oracle_ref(orc, inp)
        out, _ = solve(kda, inp, F32, "single")
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref), (bt, kind, dt)


@pytest.mark.parametrize("bt", SMALL_BT)
def test_small_chunks_poisoned_ignored_elements(kda, bt):
    for layout, kw in (("packed", dict(seqlens=(5, bt, 3 * bt + 1, 1, 70))), ("dense", dict(B=2, T=77))):
        for ind in ("f32", "bf16"):
            wl = ki.Workload("poison", layout, H=3, in_dtype=ind, out_dtype="f32", seed=23, bt=bt, **kw)
            clean, dirty = ki.build(wl), ki.build(wl, poison=True)
            a, _ = solve(kda, clean, F32, "single")
            b, _ = solve(kda, dirty, F32, "single")
            assert torch.equal(a, b), (layout, ind)


@pytest.mark.parametrize("bt", SMALL_BT)
@pytest.mark.parametrize("out_dtype", DTYPES, ids=str)
@pytest.mark.parametrize("layout", ["dense", "packed"])
def test_small_chunks_guard_band_canaries(kda, bt, out_dtype, layout):
    if layout == "dense":
        wl = ki.Workload("canary", "dense", H=3, in_dtype="f32", out_dtype="f32", seed=3, B=2, T=81, bt=bt)
    else:
        wl = ki.Workload("canary", "packed", H=3, in_dtype="f32", out_dtype="f32", seed=3,
                         seqlens=(7, 64, 90, 0, 1), bt=bt)
    inp = ki.build(wl)
    A, cu = to_dev(inp)
    pad = 4096
    n = A.numel()
    buf = torch.full((pad + n + pad,), SENTINEL[out_dtype], dtype=INT_VIEW[out_dtype], device=DEV)
    out = buf[pad:pad + n].view(out_dtype).view(A.shape)
    kda.solve_tril(A, cu, out_dtype=out_dtype, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == SENTINEL[out_dtype]) and torch.all(buf[pad + n:] == SENTINEL[out_dtype])
    assert not torch.any(buf[pad:pad + n] == SENTINEL[out_dtype])


@pytest.mark.parametrize("bt", SMALL_BT)
def test_small_chunks_packed_equals_dense_and_deterministic(kda, bt):
    lens = (5, 64, 130, 1, 77)
    wl = ki.Workload("pd", "packed", H=4, in_dtype="bf16", out_dtype="f32", seed=8, seqlens=lens, bt=bt)
    inp = ki.build(wl)
    out, _ = solve(kda, inp, F32, "single")
    for _ in range(2):
        again, _ = solve(kda, inp, F32, "single")
        assert torch.equal(out, again)
    cu = inp.cu_seqlens.tolist()
    for s in range(len(lens)):
        sub = inp.A[:, cu[s]:cu[s + 1]].contiguous()
        d = ki.SolverInput(wl.with_(layout="dense", T=lens[s]), sub, None, [lens[s]])
        o, _ = solve(kda, d, F32, "single")
        assert torch.equal(o[0], out[0, cu[s]:cu[s + 1]]), s


def test_small_chunks_rejected_paths(kda):
    inp = ki.build(ki.Workload("p", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=1, B=1, T=40, bt=16))
    A, _ = to_dev(inp)
    with pytest.raises(ValueError):
        kda.solve_tril(A, path="split")
    with pytest.raises(ValueError):
        kda.solve_tril(A, workspace=torch.empty(4096, dtype=torch.uint8, device=DEV))
    with pytest.raises(ValueError):
        kda.solve_tril(A[..., :8].contiguous())


def test_chunk_length_entry_64_is_single_pass(kda):
    import ctypes
    inp = ki.build(ki.Workload("b64", "packed", H=4, in_dtype="bf16", out_dtype="f32", seed=4,
                               seqlens=(70, 64, 3)))
    A, cu = to_dev(inp)
    ref, _ = solve(kda, inp, F32, "single")
    out = torch.empty_like(ref)
    st = kda.lib().kda_solve_tril_bt(A.data_ptr(), out.data_ptr(), cu.data_ptr(), cu.numel() - 1, 1,
                                     inp.T, inp.H, 64, 1, 0,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0 and torch.equal(out, ref)


@pytest.mark.parametrize("bt", SMALL_BT)
@pytest.mark.parametrize("name", ["packed_16x512_h64_f32", "dense_8x16384_h64_f16"])
def test_small_chunks_specified_shapes(kda, orc, bt, name):
    """The specified workloads' shapes with bt-token chunks, every element."""
    wl = ki.WORKLOADS[name].with_(bt=bt)
    inp = ki.build(wl)
    out_dtype = ki.torch_dtype(wl.out_dtype)
    out, _ = solve(kda, inp, out_dtype, "single")
    check_large(orc, inp, out, out_dtype, f"{name} bt={bt}", slab_limit=200000)


# --------------------------------------- input guard bands and similarity

def _nan_padded(t: torch.Tensor, pad: int = 4096) -> torch.Tensor:
    """A device copy of t placed between NaN guard bands of `pad` elements."""
    flat = torch.full((pad + t.numel() + pad,), float("nan"), dtype=t.dtype, device=DEV)
    flat[pad:pad + t.numel()] = t.reshape(-1).to(DEV)
    return flat[pad:pad + t.numel()].view(t.shape)


@pytest.mark.parametrize("bt", [64, 32, 16])
@pytest.mark.parametrize("layout", ["dense", "packed"])
def test_inputs_between_nan_guard_bands(kda, bt, layout):
    """Inputs sized exactly, NaN before and after: any read past the first or last
    row would reach the output."""
    kw = dict(B=2, T=3 * bt - 5) if layout == "dense" else dict(seqlens=(bt + 3, 1, 2 * bt - 1))
    inp = ki.build(ki.Workload("guard", layout, H=3, in_dtype="bf16", out_dtype="f32", seed=bt, bt=bt,
                               kind="gauss", **kw))
    A, cu = to_dev(inp)
    ref = kda.solve_tril(A, cu)
    got = kda.solve_tril(_nan_padded(inp.A), cu)
    torch.cuda.synchronize()
    assert torch.equal(ref, got)
    if bt == 64:
        assert torch.equal(ref, kda.solve_tril(_nan_padded(inp.A), cu, path="split"))


def test_kgb_inputs_between_nan_guard_bands(kda):
    x = ki.build_kgb(ki.Workload("guard", "packed", H=3, in_dtype="bf16", out_dtype="f32", seed=6,
                                 seqlens=(67, 1, 127)))
    cu = x.cu_seqlens.to(DEV)
    ref = kda.solve_tril_kgb(x.k.to(DEV), x.g.to(DEV), x.beta.to(DEV), cu)
    got = kda.solve_tril_kgb(_nan_padded(x.k), _nan_padded(x.g), _nan_padded(x.beta), cu)
    torch.cuda.synchronize()
    assert torch.equal(ref, got)


@pytest.mark.parametrize("bt", [64, 32, 16])
def test_power_of_two_similarity_bitwise(kda, bt):
    """D A D^-1 -> D Ai D^-1 bit for bit (D = diag(2^e) per chunk row): the split-TF32
    products, the FP32 sums and the forward substitution all commute with scaling
    by powers of two."""
    inp = ki.build(ki.Workload("sim", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=bt, B=1, T=2 * bt,
                               kind="gauss", bt=bt))
    e = torch.from_numpy(np.random.default_rng(bt).integers(-2, 3, bt)).double()
    S = torch.pow(2.0, e[:, None] - e[None, :]).float()        # 2^(e_i - e_j), exact
    A = inp.A.view(1, 2, bt, 2, bt)                           # [B, chunk, i, H, j]
    As = (A * S[None, None, :, None, :]).reshape(inp.A.shape).contiguous()
    paths = ("single", "split") if bt == 64 else ("auto",)
    for path in paths:
        X = kda.solve_tril(inp.A.to(DEV), path=path).cpu().view(1, 2, bt, 2, bt)
        Xs = kda.solve_tril(As.to(DEV), path=path).cpu().view(1, 2, bt, 2, bt)
        assert torch.equal(Xs, X * S[None, None, :, None, :]), path
