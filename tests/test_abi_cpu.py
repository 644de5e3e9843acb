"""The C ABI on a machine without a GPU: loading, exports, sizing, selection and
argument checks (all of which return before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

import linear_attention_chunked_02_gb300 as kda
from linear_attention_chunked_02_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kda.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text, flags=re.M))
    return names


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"kda_solve_tril", "kda_solve_tril_ex", "kda_solve_tril_workspace_size",
            "kda_solve_tril_select", "kda_solve_tril_host", "kda_status_string",
            "kda_device_error", "kda_version"} <= names
    for n in names:
        assert hasattr(L, n), n
    bound = {s[0] for s in kda._lib.SIGNATURES}
    assert names == bound, names ^ bound


def test_workspace_size_and_selector(L):
    # 4 KiB per chunk-head; packed bound min(T, (T + 63 N) / 64)
    assert kda.workspace_size(1, 8192, 64, 16) == ((8192 + 63 * 16) // 64) * 64 * 4096
    assert kda.workspace_size(2, 100, 3, 0) == 2 * 2 * 3 * 4096
    assert kda.workspace_size(1, 5, 1, 5) == 5 * 4096          # capped by T
    assert kda.workspace_size(0, 0, 1, 0) == 0
    assert kda.workspace_size(2, 64, 1, 3) == 0                # packed needs B == 1
    # GB300 selector: the split path never paid at measured sizes, so AUTO is
    # single pass below the minimum length whatever the workspace
    need = kda.workspace_size(1, 8192, 64, 16)
    assert kda.select_path(1, 8192, 64, 16, need) == "single"
    assert kda.select_path(1, 64, 64, 0, 1 << 30) == "single"
    # the budget rule itself, above the minimum length (pure host arithmetic)
    T = 1 << 32
    need = kda.workspace_size(1, T, 8, 4096)
    assert kda.select_path(1, T, 8, 4096, need) == "split"
    assert kda.select_path(1, T, 8, 4096, need - 1) == "single"
    assert kda.select_path(1, T, 8, 4096, 0) == "single"
    # occupancy < 16 rows per chunk: the workspace would exceed the FP32 input
    N = (1 << 30) - 1                                          # requests of ~4 rows
    assert kda.workspace_size(1, T, 8, N) > T * 8 * 256
    assert kda.select_path(1, T, 8, N, 1 << 62) == "single"
    # the bound counts a possibly partial chunk per request, so 16-row
    # requests already exceed it while 32-row requests do not
    assert kda.select_path(1, T, 8, T // 16, 1 << 62) == "single"
    assert kda.select_path(1, T, 8, T // 32, 1 << 62) == "split"


def call(L, A=16, Ai=1 << 20, cu=None, nseq=0, B=1, T=64, H=1, ind=0, outd=0, ws=None, wsb=0, path=0):
    taken = ctypes.c_int32(-1)
    st = L.kda_solve_tril_ex(A, Ai, cu, nseq, B, T, H, ind, outd, ws, wsb, None, path, ctypes.byref(taken))
    return st, taken.value


def test_argument_errors_before_any_cuda_call(L):
    assert call(L, ind=7)[0] == UNSUPPORTED
    assert call(L, outd=-1)[0] == UNSUPPORTED
    assert call(L, H=0)[0] == INVALID
    assert call(L, T=-1)[0] == INVALID
    assert call(L, cu=4096, nseq=0)[0] == INVALID              # cu_seqlens without a count
    assert call(L, cu=None, nseq=2)[0] == INVALID
    assert call(L, cu=4096, nseq=1, B=2)[0] == INVALID         # packed needs B == 1
    assert call(L, A=None)[0] == INVALID
    assert call(L, A=8)[0] == INVALID                          # misaligned
    assert call(L, A=1 << 20, Ai=(1 << 20) + 4096)[0] == INVALID   # overlapping
    assert call(L, path=5)[0] == INVALID
    assert call(L, T=1 << 31)[0] == UNSUPPORTED
    assert call(L, H=1 << 19)[0] == UNSUPPORTED                # H * 64 * 64 >= 2^31
    assert call(L, A=1 << 40, Ai=1 << 44, H=(1 << 19) - 1)[0] != UNSUPPORTED
    assert call(L, path=1, ws=None)[0] == WORKSPACE            # forced split, no workspace
    assert call(L, path=1, ws=1 << 24, wsb=100)[0] == WORKSPACE
    assert call(L, path=1, ws=(1 << 24) + 8, wsb=1 << 20)[0] == INVALID  # misaligned workspace
    st, taken = call(L, T=0)
    assert st == OK                                            # empty input is a no-op
    st, taken = call(L, B=0)
    assert st == OK


def call_static(L, A=16, Ai=1 << 20, cu=None, nseq=0, B=1, T=64, H=1, ind=0, outd=0):
    return L.kda_solve_tril_split_static(A, Ai, cu, nseq, B, T, H, ind, outd, None)


def test_static_entry_argument_errors_before_any_cuda_call(L):
    """kda_solve_tril_split_static reports argument errors itself, before it looks
    up its built-in workspace: without a GPU, any CUDA call would give KDA_ERR_CUDA."""
    assert call_static(L, ind=7) == UNSUPPORTED
    assert call_static(L, outd=3) == UNSUPPORTED
    assert call_static(L, H=0) == INVALID
    assert call_static(L, A=None) == INVALID
    assert call_static(L, Ai=None) == INVALID
    assert call_static(L, A=8) == INVALID                      # misaligned
    assert call_static(L, A=1 << 20, Ai=(1 << 20) + 4096) == INVALID
    assert call_static(L, cu=4096, nseq=1, B=2) == INVALID     # packed needs B == 1
    assert call_static(L, cu=None, nseq=2) == INVALID
    assert call_static(L, T=1 << 31) == UNSUPPORTED
    assert call_static(L, A=1 << 40, Ai=1 << 44, T=1 << 20, H=64) == WORKSPACE   # beyond the built-in 64 MiB
    assert call_static(L, T=0) == OK
    assert call_static(L, B=0) == OK


def test_status_strings(L):
    for s in range(6):
        assert L.kda_status_string(s)
    assert L.kda_status_string(99) == b"unknown status"
    assert L.kda_version() >= 100


def test_no_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, taken = call(L, A=1 << 20, Ai=1 << 24)
    assert st == CUDA
    assert taken == 2


def test_host_entry_checks(L):
    st = L.kda_solve_tril_host(None, None, None, 0, 1, 64, 1, 0, 0, 16, 1 << 20, None, None, 0, None)
    assert st == INVALID
    st = L.kda_solve_tril_host(16, 32, 48, 1, 1, 64, 1, 0, 0, 16, 1 << 20, None, None, 0, None)
    assert st == INVALID                                       # host cu without device cu


def call_bt(L, A=16, Ai=1 << 20, cu=None, nseq=0, B=1, T=64, H=1, bt=16, ind=0, outd=0):
    return L.kda_solve_tril_bt(A, Ai, cu, nseq, B, T, H, bt, ind, outd, None)


def test_chunk_length_entry_checks(L):
    for bt in (0, 8, 48, 128, -16):
        assert call_bt(L, bt=bt) == UNSUPPORTED
    for bt in (16, 32):
        assert call_bt(L, bt=bt, ind=3) == UNSUPPORTED
        assert call_bt(L, bt=bt, outd=9) == UNSUPPORTED
        assert call_bt(L, bt=bt, H=0) == INVALID
        assert call_bt(L, bt=bt, cu=4096, nseq=0) == INVALID
        assert call_bt(L, bt=bt, cu=4096, nseq=1, B=2) == INVALID
        assert call_bt(L, bt=bt, A=None) == INVALID
        assert call_bt(L, bt=bt, Ai=(1 << 20) + 8) == INVALID      # misaligned
        # A [1, 64, 1, bt] fp32 spans 256 bt bytes: Ai inside it overlaps
        assert call_bt(L, bt=bt, A=1 << 20, Ai=(1 << 20) + 64 * bt * 4 - 16) == INVALID
        assert call_bt(L, bt=bt, A=1 << 20, Ai=(1 << 20) + 64 * bt * 4) != INVALID
        assert call_bt(L, bt=bt, T=1 << 31) == UNSUPPORTED
        assert call_bt(L, bt=bt, H=(1 << 31) // (bt * bt)) == UNSUPPORTED   # H * bt * bt >= 2^31
        # chunks * H counted with bt-row chunks: 2^30 rows hold 2^30 / bt
        # chunks, so bt heads reach the 2^30 chunk-head limit, bt / 2 do not
        assert call_bt(L, bt=bt, B=1, T=1 << 30, H=bt) == UNSUPPORTED
        assert call_bt(L, bt=bt, A=1 << 40, Ai=1 << 44, B=1, T=1 << 30, H=bt // 2) not in (UNSUPPORTED, INVALID)
        assert call_bt(L, bt=bt, T=0) == OK
        assert call_bt(L, bt=bt, B=0) == OK
    # 64 goes to the single-pass 64-token path with its checks
    assert call_bt(L, bt=64, ind=7) == UNSUPPORTED
    assert call_bt(L, bt=64, T=0) == OK


def test_chunk_length_entry_no_gpu(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for bt in (16, 32, 64):
        assert call_bt(L, bt=bt, A=1 << 20, Ai=1 << 24) == CUDA


def call_kgb(L, k=1 << 20, g=1 << 22, beta=1 << 24, Ai=1 << 26, cu=None, nseq=0, B=1, T=64, H=1, K=128,
             ind=0, outd=0):
    return L.kda_solve_tril_kgb(k, g, beta, Ai, cu, nseq, B, T, H, K, ind, outd, None)


def test_kgb_entry_checks(L):
    for K in (0, 16, 48, 160, 256):
        assert call_kgb(L, K=K) == UNSUPPORTED
    assert call_kgb(L, ind=5) == UNSUPPORTED
    assert call_kgb(L, outd=5) == UNSUPPORTED
    assert call_kgb(L, H=0) == INVALID
    assert call_kgb(L, cu=4096, nseq=1, B=2) == INVALID
    assert call_kgb(L, g=None) == INVALID
    assert call_kgb(L, beta=None) == INVALID
    assert call_kgb(L, k=None) == INVALID
    assert call_kgb(L, g=(1 << 22) + 4) == INVALID                # misaligned g
    assert call_kgb(L, beta=(1 << 24) + 2) == INVALID             # fp32 beta not 4-byte aligned
    assert call_kgb(L, beta=(1 << 24) + 2, ind=1) != INVALID      # bf16 beta: 2-byte alignment is enough
    assert call_kgb(L, Ai=(1 << 20) + 64 * 128 * 4 - 16) == INVALID   # Ai overlaps k
    assert call_kgb(L, T=0) == OK and call_kgb(L, B=0) == OK
    assert call_kgb(L, H=1 << 19) == UNSUPPORTED


def test_kgb_entry_no_gpu(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_kgb(L) == CUDA


def test_python_binding_rejects_host_tensors_and_bad_shapes(L):
    import torch
    with pytest.raises(ValueError):
        kda.solve_tril(torch.zeros(1, 64, 1, 64))                  # host tensor: no CPU path
    with pytest.raises(ValueError):
        kda.solve_tril_kgb(torch.zeros(1, 64, 1, 128), torch.zeros(1, 64, 1, 128), torch.zeros(1, 64, 1))
    meta = torch.zeros(1, 64, 1, 48, device="meta")
    with pytest.raises(ValueError):
        kda._shape(meta, None, kda.CHUNK_LENGTHS)                  # chunk length 48 is not a branch
    assert kda._shape(torch.zeros(2, 5, 3, 16, device="meta"), None, kda.CHUNK_LENGTHS) == (2, 5, 3, 0)
    with pytest.raises(ValueError):
        kda._shape(torch.zeros(2, 5, 3, 16, device="meta"), None)  # the 64-token entry points take 64 only


def call_prec(L, A=16, Ai=1 << 20, cu=None, nseq=0, B=1, T=64, H=1, ind=0, outd=0, prec=1):
    return L.kda_solve_tril_prec(A, Ai, cu, nseq, B, T, H, ind, outd, prec, None)


def test_precision_entry_argument_errors_before_any_cuda_call(L):
    """kda_solve_tril_prec checks the precision mode and every argument on the host
    (without a GPU, a CUDA call would give KDA_ERR_CUDA)."""
    assert call_prec(L, prec=2) == INVALID
    assert call_prec(L, prec=-1) == INVALID
    assert call_prec(L, ind=7) == UNSUPPORTED
    assert call_prec(L, H=0) == INVALID
    assert call_prec(L, A=8) == INVALID                        # misaligned
    assert call_prec(L, A=1 << 20, Ai=(1 << 20) + 4096) == INVALID   # overlapping
    assert call_prec(L, cu=4096, nseq=1, B=2) == INVALID
    assert call_prec(L, T=0) == OK and call_prec(L, B=0, prec=0) == OK


def test_python_precision_argument(monkeypatch):
    import torch
    A = torch.zeros(1, 64, 1, 64)
    with pytest.raises(ValueError, match="unknown precision"):
        kda.solve_tril(A, precision="fp8")


def test_selftest_entry_checks_its_limit(L):
    assert L.kda_selftest_wait(0, 0, None) == INVALID
    assert L.kda_selftest_wait(0, 1000001, None) == INVALID
