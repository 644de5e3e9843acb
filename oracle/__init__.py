"""fp64 CPU oracle for the KDA prefill chunk solver -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline import this package.  The product path (the CUDA library and its
Python binding) never does, and this package imports nothing from it.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, forward substitution
per chunk-head; see that file's header for the passage it follows).  This
module compiles it with gcc and wraps it with ctypes and numpy.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "kda_oracle.c")
LIB = os.path.join(_HERE, "libkda_oracle.so")
BT = 64


def compile_oracle(out_path: str = LIB, plant: int = 0, openmp: bool = True) -> str:
    """Compile ``kda_oracle.c`` into a shared library at ``out_path``.

    ``plant`` != 0 builds a copy with a deliberate mistake (negative controls).
    Falls back to a single-threaded build when the compiler has no OpenMP.
    """
    cc = os.environ.get("CC", shutil.which("gcc") or "cc")
    base = [cc, "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
            f"-DKDA_ORACLE_PLANT={int(plant)}", SRC, "-lm", "-o", out_path]
    tmp = out_path + ".tmp"
    cmds = ([base[:-1] + [tmp, "-fopenmp"]] if openmp else []) + [base[:-1] + [tmp]]
    assert base[-2] == "-o"
    err = ""
    for cmd in cmds:
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, out_path)
            return out_path
        err = r.stderr
    raise RuntimeError(f"oracle build failed:\n{err}")


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        lib.kda_oracle_invert_chunk.argtypes = [dp, ctypes.c_int64, ctypes.c_int, dp]
        lib.kda_oracle_invert_chunk.restype = None
        lib.kda_oracle_solve_tril.argtypes = [dp, dp, ip, ctypes.c_int32, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_int32]
        lib.kda_oracle_solve_tril.restype = ctypes.c_int
        lib.kda_oracle_invert_chunk_bt.argtypes = [dp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, dp]
        lib.kda_oracle_invert_chunk_bt.restype = None
        lib.kda_oracle_solve_tril_bt.argtypes = [dp, dp, ip, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_int32, ctypes.c_int32]
        lib.kda_oracle_solve_tril_bt.restype = ctypes.c_int
        lib.kda_oracle_solve_kgb.argtypes = [dp, dp, dp, dp, dp, ip, ctypes.c_int32, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
        lib.kda_oracle_solve_kgb.restype = ctypes.c_int
        lib.kda_oracle_num_chunks.argtypes = [ip, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]
        lib.kda_oracle_num_chunks.restype = ctypes.c_int64
        lib.kda_oracle_num_threads.restype = ctypes.c_int
        lib.kda_oracle_planted.restype = ctypes.c_int
        self.lib = lib

    @staticmethod
    def _dptr(a: np.ndarray):
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))

    def invert_chunk(self, M: np.ndarray, n: Optional[int] = None, bt: int = BT) -> np.ndarray:
        """(I + strict_lower(M[:n, :n]))^-1 embedded in a bt x bt identity, fp64."""
        M = np.ascontiguousarray(M, dtype=np.float64)
        if n is None:
            n = M.shape[0]
        if M.ndim != 2 or not (0 <= n <= min(M.shape[0], M.shape[1], bt)) or not 1 <= bt <= BT:
            raise ValueError(f"bad chunk shape {M.shape} for n={n}, bt={bt}")
        X = np.empty((bt, bt), dtype=np.float64)
        self.lib.kda_oracle_invert_chunk_bt(self._dptr(M), M.shape[1], int(n), int(bt), self._dptr(X))
        return X

    def solve_tril(self, A: np.ndarray, cu_seqlens: Optional[np.ndarray] = None) -> np.ndarray:
        """Solve every chunk-head of A ([B, T, H, bt], any float dtype, upcast exactly);
        the chunk length bt is A's last dimension.

        Returns fp64 Ai of the same shape; rows that belong to no chunk are zero.
        """
        A64 = np.ascontiguousarray(A, dtype=np.float64)
        assert A64.ndim == 4 and 1 <= A64.shape[3] <= BT
        B, T, H, bt = A64.shape
        Ai = np.zeros_like(A64)
        if cu_seqlens is not None:
            cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
            cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
            nseq = cu.shape[0] - 1
        else:
            cup, nseq = None, 0
        rc = self.lib.kda_oracle_solve_tril_bt(self._dptr(A64), self._dptr(Ai), cup, nseq, B, T, H, bt)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return Ai

    def solve_kgb(self, k: np.ndarray, g: np.ndarray, beta: np.ndarray,
                  cu_seqlens: Optional[np.ndarray] = None, return_A: bool = False):
        """Build every 64-token chunk's A from keys k [B, T, H, K], cumulative log
        decays g [B, T, H, K] and betas [B, T, H] (any float dtype, upcast exactly)
        and solve it.  Returns fp64 Ai [B, T, H, 64] (and A if return_A); rows that
        belong to no chunk are zero."""
        k64 = np.ascontiguousarray(k, dtype=np.float64)
        g64 = np.ascontiguousarray(g, dtype=np.float64)
        b64 = np.ascontiguousarray(beta, dtype=np.float64)
        assert k64.ndim == 4 and g64.shape == k64.shape and b64.shape == k64.shape[:3]
        B, T, H, K = k64.shape
        Ai = np.zeros((B, T, H, BT))
        A = np.zeros((B, T, H, BT)) if return_A else None
        if cu_seqlens is not None:
            cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
            cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
            nseq = cu.shape[0] - 1
        else:
            cup, nseq = None, 0
        rc = self.lib.kda_oracle_solve_kgb(self._dptr(k64), self._dptr(g64), self._dptr(b64), self._dptr(Ai),
                                           self._dptr(A) if A is not None else None, cup, nseq, B, T, H, K)
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return (Ai, A) if return_A else Ai

    def num_threads(self) -> int:
        return int(self.lib.kda_oracle_num_threads())

    def planted(self) -> int:
        return int(self.lib.kda_oracle_planted())


_ORACLE: Optional[Oracle] = None


def get() -> Oracle:
    """The real oracle, compiled on first use if its library is missing or stale."""
    global _ORACLE
    if _ORACLE is None:
        if (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            compile_oracle(LIB)
        _ORACLE = Oracle(LIB)
    return _ORACLE


def to_f64(t) -> np.ndarray:
    """Exact fp64 copy of a (CPU or CUDA) torch tensor or numpy array."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)
