"""The allocation-free split solve, kda_solve_tril_split_static, through the C ABI.

Some callers cannot allocate device memory where they call the solver (a
plugin inside a framework that owns all device memory, or a serving loop that
must not call cudaMalloc / cudaFree after start-up because those calls can
synchronise the device).  For them the library carries the split path's FP32
workspace in a built-in device array.  Here two calls in a row, on different
inputs, must each agree with the regular entry point kda_solve_tril on the same
input, within the parity tolerance used by the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle.parity as parity

pytestmark = pytest.mark.gpu

DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_chunked_02_gb300 import build as kbuild
    kbuild.build()
    import linear_attention_chunked_02_gb300 as kda
    return kda.lib()


def _regular(L, A, cu, nseq, out_dtype):
    """kda_solve_tril with a workspace allocated by the caller (torch)."""
    B, T, H, _ = A.shape
    need = L.kda_solve_tril_workspace_size(B, T, H, nseq)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=A.device)
    out = torch.empty(A.shape, dtype=out_dtype, device=A.device)
    st = L.kda_solve_tril(A.data_ptr(), out.data_ptr(), cu.data_ptr() if cu is not None else None, nseq,
                          B, T, H, DTYPE_CODE[A.dtype], DTYPE_CODE[out_dtype], ws.data_ptr(), need,
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    return out


def _static(L, A, cu, nseq, out_dtype):
    """kda_solve_tril_split_static: inputs and outputs only."""
    B, T, H, _ = A.shape
    out = torch.empty(A.shape, dtype=out_dtype, device=A.device)
    st = L.kda_solve_tril_split_static(A.data_ptr(), out.data_ptr(), cu.data_ptr() if cu is not None else None,
                                       nseq, B, T, H, DTYPE_CODE[A.dtype], DTYPE_CODE[out_dtype],
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.kda_status_string(st)
    return out


def test_two_calls_match_regular_entry_point(lib):
    cases = [
        ki.WORKLOADS["packed_16x512_h64_f32"],
        ki.Workload("no_alloc_dense", "dense", H=8, in_dtype="bf16", out_dtype="bf16", seed=77, B=3, T=1000,
                    kind="nodecay"),
    ]
    for wl in cases:                                   # two calls in a row, different inputs
        inp = ki.build(wl)
        A = inp.A.cuda()
        cu = inp.cu_seqlens.cuda() if inp.cu_seqlens is not None else None
        nseq = 0 if cu is None else cu.numel() - 1
        out_dtype = ki.torch_dtype(wl.out_dtype)
        got = _static(lib, A, cu, nseq, out_dtype)
        ref = _regular(lib, A, cu, nseq, out_dtype)
        torch.cuda.synchronize()
        g = got.double().cpu().numpy()
        r = ref.double().cpu().numpy()
        want, tol = parity.bound(r, inp.A.dtype, out_dtype)
        assert np.all(np.abs(g - want) <= tol), wl.name
        assert torch.equal(got, ref), wl.name           # same kernels, same order: same bits


def test_rejects_shapes_beyond_the_builtin_workspace(lib):
    # dense [1, 65536, 64, 64] needs 1024 * 64 * 4 KiB = 256 MiB of workspace
    st = lib.kda_solve_tril_split_static(1 << 40, 1 << 44, None, 0, 1, 65536, 64, 0, 0, None)
    assert st == 3                                     # KDA_ERR_WORKSPACE, before any CUDA call
    assert lib.kda_solve_tril_workspace_size(1, 65536, 64, 0) > (64 << 20)
