"""KDA prefill chunk solver for GB300 (sm_103a): Python binding of the C ABI.

``solve_tril`` computes, for every 64-token chunk and head, ``(I + A)^-1`` of
the chunk's strictly lower-triangular matrix ``A`` (LightLLM PR #1703,
"perf(kda): parallelize diagonal solves in Prefill"); chunks of 16 and 32
tokens (the solver's shorter branches) are taken from A's last dimension.
Every step runs in the
CUDA kernels of ``libkda_solve_tril.so``; this module only checks and
marshals arguments (torch provides device memory and streams).
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from ._lib import lib, LIB_PATH  # noqa: F401

BT = 64
CHUNK_LENGTHS = (16, 32, 64)
WS_TILE_BYTES = 4096
DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
PATH_CODE = {"auto": 0, "split": 1, "single": 2}
PATH_NAME = {v: k for k, v in PATH_CODE.items()}
PRECISION_CODE = {"ieee": 0, "tf32": 1}


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib().kda_status_string(status).decode()} (status {status})")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise KdaError(status, where)


def _shape(A: torch.Tensor, cu_seqlens: Optional[torch.Tensor], lengths=(BT,)):
    if A.dim() != 4 or A.shape[3] not in lengths:
        raise ValueError(f"A must be [B, T, H, bt] with bt in {lengths}, got {tuple(A.shape)}")
    B, T, H, _ = A.shape
    nseq = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    return B, T, H, nseq


def workspace_size(B: int, T: int, H: int, num_seqs: int = 0) -> int:
    """Bytes of FP32 workspace the split path needs (upper bound on the chunk count)."""
    return int(lib().kda_solve_tril_workspace_size(B, T, H, num_seqs))


def select_path(B: int, T: int, H: int, num_seqs: int = 0, workspace_bytes: int = 0) -> str:
    """The path the automatic selector takes: "split" or "single"."""
    return PATH_NAME[int(lib().kda_solve_tril_select(B, T, H, num_seqs, workspace_bytes))]


def _stream_ptr(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def solve_tril(A: torch.Tensor, cu_seqlens: Optional[torch.Tensor] = None,
               out_dtype: torch.dtype = torch.float32, path: str = "auto",
               out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               stream: Optional[torch.cuda.Stream] = None, return_path: bool = False,
               precision: str = "ieee"):
    """Per chunk-head inverse of (I + strict_lower(A)).

    A: CUDA tensor [B, T, H, bt] (float32 / bfloat16 / float16), contiguous;
    bt = 64, or 16 / 32 for the shorter chunk lengths.
    cu_seqlens: int32 CUDA tensor [N+1] for the packed layout (then B == 1).
    path: "auto" (selector), "split" or "single"; chunks of 16 or 32 tokens have
    one path only ("auto" or "single").
    workspace: optional CUDA buffer for the split path; allocated here when the
    selector would split and none is given.
    precision: "ieee" (FP32-accurate, every path) or "tf32" (64-token chunks, the
    single pass with plain TF32 merge products; kda_solve_tril_prec).
    """
    if precision not in PRECISION_CODE:
        raise ValueError(f"unknown precision {precision!r}")
    if not A.is_cuda:
        raise ValueError("A must be a CUDA tensor")
    if A.dtype not in DTYPE_CODE or out_dtype not in DTYPE_CODE:
        raise ValueError(f"unsupported dtype {A.dtype} -> {out_dtype}")
    A = A.contiguous()
    B, T, H, nseq = _shape(A, cu_seqlens, CHUNK_LENGTHS)
    bt = A.shape[3]
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        cu_seqlens = cu_seqlens.contiguous()
    if out is None:
        out = torch.empty(A.shape, dtype=out_dtype, device=A.device)
    elif out.shape != A.shape or out.dtype != out_dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of A's shape and out_dtype")
    if precision == "tf32":
        if bt != BT or path not in ("auto", "single") or workspace is not None:
            raise ValueError("the tf32 precision mode is the 64-token single pass (no workspace)")
        with torch.cuda.device(A.device):
            st = lib().kda_solve_tril_prec(
                A.data_ptr(), out.data_ptr(), cu_seqlens.data_ptr() if cu_seqlens is not None else None,
                nseq, B, T, H, DTYPE_CODE[A.dtype], DTYPE_CODE[out_dtype], PRECISION_CODE[precision],
                _stream_ptr(stream, A.device))
        _check(st, "kda_solve_tril_prec")
        return (out, "single") if return_path else out
    if bt != BT:
        if path not in ("auto", "single") or workspace is not None:
            raise ValueError(f"{bt}-token chunks have a single path and take no workspace")
        with torch.cuda.device(A.device):
            st = lib().kda_solve_tril_bt(
                A.data_ptr(), out.data_ptr(), cu_seqlens.data_ptr() if cu_seqlens is not None else None,
                nseq, B, T, H, bt, DTYPE_CODE[A.dtype], DTYPE_CODE[out_dtype], _stream_ptr(stream, A.device))
        _check(st, "kda_solve_tril_bt")
        return (out, "single") if return_path else out
    if workspace is None and path in ("auto", "split"):
        need = workspace_size(B, T, H, nseq)
        if need > 0 and (path == "split" or select_path(B, T, H, nseq, need) == "split"):
            workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    taken = ctypes.c_int32(-1)
    with torch.cuda.device(A.device):
        st = lib().kda_solve_tril_ex(
            A.data_ptr(), out.data_ptr(), cu_seqlens.data_ptr() if cu_seqlens is not None else None,
            nseq, B, T, H, DTYPE_CODE[A.dtype], DTYPE_CODE[out_dtype], ws_ptr, ws_bytes,
            _stream_ptr(stream, A.device), PATH_CODE[path], ctypes.byref(taken))
    _check(st, "kda_solve_tril_ex")
    if return_path:
        return out, PATH_NAME.get(taken.value, "none")
    return out


def solve_tril_kgb(k: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                   cu_seqlens: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
                   out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Per 64-token chunk-head, (I + A)^-1 for the chunk matrix built on chip from
    keys k [B, T, H, K], cumulative log decays g [B, T, H, K] (float32) and betas
    [B, T, H]: A[i][j] = beta_i sum_d k_id k_jd exp(g_id - g_jd), j < i.  k and beta
    share a dtype (float32 / bfloat16 / float16); K is 32, 64, 96 or 128."""
    for name, t in (("k", k), ("g", g), ("beta", beta)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    if k.dim() != 4 or g.shape != k.shape or beta.shape != k.shape[:3]:
        raise ValueError(f"shapes k {tuple(k.shape)}, g {tuple(g.shape)}, beta {tuple(beta.shape)} do not match")
    if k.dtype not in DTYPE_CODE or beta.dtype != k.dtype or g.dtype != torch.float32 or out_dtype not in DTYPE_CODE:
        raise ValueError(f"unsupported dtypes k {k.dtype}, g {g.dtype}, beta {beta.dtype} -> {out_dtype}")
    k, g, beta = k.contiguous(), g.contiguous(), beta.contiguous()
    B, T, H, K = k.shape
    nseq = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        cu_seqlens = cu_seqlens.contiguous()
    shape = (B, T, H, BT)
    if out is None:
        out = torch.empty(shape, dtype=out_dtype, device=k.device)
    elif tuple(out.shape) != shape or out.dtype != out_dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, T, H, 64] tensor of out_dtype")
    with torch.cuda.device(k.device):
        st = lib().kda_solve_tril_kgb(
            k.data_ptr(), g.data_ptr(), beta.data_ptr(), out.data_ptr(),
            cu_seqlens.data_ptr() if cu_seqlens is not None else None, nseq, B, T, H, K,
            DTYPE_CODE[k.dtype], DTYPE_CODE[out_dtype], _stream_ptr(stream, k.device))
    _check(st, "kda_solve_tril_kgb")
    return out


def solve_tril_host(A_host: torch.Tensor, Ai_host: torch.Tensor, A_dev: torch.Tensor, Ai_dev: torch.Tensor,
                    cu_seqlens_host: Optional[torch.Tensor] = None, cu_dev: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> None:
    """End-to-end call: host A -> device, solve, device Ai -> host Ai_host (enqueued, not synchronised)."""
    B, T, H, nseq = _shape(A_host, cu_seqlens_host)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(A_dev.device):
        st = lib().kda_solve_tril_host(
            A_host.data_ptr(), Ai_host.data_ptr(),
            cu_seqlens_host.data_ptr() if cu_seqlens_host is not None else None, nseq, B, T, H,
            DTYPE_CODE[A_host.dtype], DTYPE_CODE[Ai_host.dtype], A_dev.data_ptr(), Ai_dev.data_ptr(),
            cu_dev.data_ptr() if cu_dev is not None else None, ws_ptr, ws_bytes,
            _stream_ptr(stream, A_dev.device))
    _check(st, "kda_solve_tril_host")


def device_error(device: int = 0) -> int:
    """Read and clear the library's device-side error word (synchronises the device)."""
    code = ctypes.c_uint32(0)
    _check(lib().kda_device_error(device, ctypes.byref(code)), "kda_device_error")
    return int(code.value)
