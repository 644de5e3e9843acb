"""Seeded synthetic inputs for the KDA chunk solver.

This module only *builds* the strictly-lower-triangular chunk matrices ``A``
that the solver consumes; it contains none of the solver's arithmetic, so the
fp64 oracle (``oracle/``) and the CUDA path can both consume its output
without sharing any code with one another.

Where the numbers come from
---------------------------
LightLLM PR #1703 ("perf(kda): parallelize diagonal solves in Prefill", PR
description) solves ``(I + A)^-1`` for each 64-token chunk of a KDA (Kimi
Delta Attention) prefill.  The page gives no input values, so ``A`` follows
the KDA intra-chunk construction, per token ``t`` and head ``h``::

    k_t   ~ N(0, 1)^128, L2-normalised over the 128 key channels
    beta_t = sigmoid(N(0, 1))
    g_t    = within-chunk cumulative sum of -softplus(N(0, 1)), per channel,
             restarting at every chunk start
    A[t, h, j] = beta_t * sum_d k_{t,d} k_{s,d} exp(g_{t,d} - g_{s,d})
                 for the chunk's column-j token s with j < i (i = row in chunk)
    A[t, h, j] = 0 otherwise

Because ``g_t - g_s <= 0`` for s before t and the keys are unit vectors,
``|A| <= beta <= 1``.  Everything is computed in fp64 and then rounded to the
input dtype (fp64 -> fp32 round-to-nearest-even, then fp32 -> bf16/fp16
round-to-nearest-even).

Draw order (all from ``numpy.random.default_rng(seed)``): the request lengths
of a ragged packed workload first, then, slab by slab (a slab is one batch row
of a dense layout or one request of a packed layout), ``k``, the ``beta``
pre-activations and the ``g`` pre-activations.

Two stress kinds exist because the decay makes far-off-diagonal blocks of the
inverse tiny (about 1e-10 for the block three below the diagonal), so a solver
that dropped them would still pass a tolerance test on KDA-style inputs:

* ``"nodecay"``: the same construction with ``g == 0``;
* ``"gauss"``: ``A[t, h, j] ~ N(0, 0.2^2)`` for ``j < i``, 0 otherwise.

A third kind, ``"steep"``, exists only for the keys/decays/betas inputs
(``build_kgb``): KDA's decay may fall steeply, and a construction that factors
``exp(g_i - g_j)`` through a reference row can overflow or lose the large terms
there.  Per channel ``d`` the per-token drop of ``g`` is, by ``d mod 4``:
0: uniform in [8, 20] nats; 1: the KDA drop plus, with probability 1/16 per
token, a cliff of 100 nats; 2: uniform in [3, 8] nats; 3: the KDA drop.  The
extra uniforms are drawn after the ``g`` pre-activations of each slab.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

BT = 64          # chunk length (tokens per chunk); the solver's only supported size
KEY_DIM = 128    # key channels of the KDA construction

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Workload:
    """One synthetic solver input: layout, sizes, dtypes and seed."""

    name: str
    layout: str                      # "dense" ([B, T, H, 64]) or "packed" ([1, T_total, H, 64])
    H: int
    in_dtype: str                    # "f32" | "bf16" | "f16"
    out_dtype: str
    seed: int
    B: int = 1                       # dense only
    T: int = 0                       # dense: tokens per batch row
    seqlens: Optional[Sequence[int]] = None   # packed: fixed request lengths
    ragged: Optional[tuple] = None   # packed: (num_requests, min_len, max_len) drawn from the seed
    kind: str = "kda"                # "kda" | "nodecay" | "gauss" | "steep" (build_kgb only)
    bt: int = BT                     # chunk length (64, or the 32 / 16 branches)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five workloads the solver is specified and measured on.
WORKLOADS = {
    "dense_1x64_h4_f32": Workload("dense_1x64_h4_f32", "dense", H=4, in_dtype="f32",
                                  out_dtype="f32", seed=0, B=1, T=64),
    "dense_1x64_h64_bf16": Workload("dense_1x64_h64_bf16", "dense", H=64, in_dtype="bf16",
                                    out_dtype="f32", seed=1, B=1, T=64),
    "packed_16x512_h64_f32": Workload("packed_16x512_h64_f32", "packed", H=64, in_dtype="f32",
                                      out_dtype="f32", seed=2, seqlens=(512,) * 16),
    "packed_ragged37_h32_bf16": Workload("packed_ragged37_h32_bf16", "packed", H=32,
                                         in_dtype="bf16", out_dtype="f32", seed=3,
                                         ragged=(37, 1, 2048)),
    "dense_8x16384_h64_f16": Workload("dense_8x16384_h64_f16", "dense", H=64, in_dtype="f16",
                                      out_dtype="bf16", seed=4, B=8, T=16384),
}


@dataclass
class SolverInput:
    """A built input: ``A`` on the host (in its input dtype) plus layout metadata."""

    workload: Workload
    A: torch.Tensor                          # [B, T, H, 64], CPU, input dtype
    cu_seqlens: Optional[torch.Tensor]       # int32 [N+1] (packed) or None (dense)
    seqlens: list = field(default_factory=list)

    @property
    def B(self) -> int:
        return self.A.shape[0]

    @property
    def T(self) -> int:
        return self.A.shape[1]

    @property
    def H(self) -> int:
        return self.A.shape[2]

    @property
    def bt(self) -> int:
        return self.A.shape[3]

    def chunks(self):
        """(row0, n_valid) of every chunk, in order; rows index the flattened B*T axis."""
        bt = self.bt
        out = []
        if self.cu_seqlens is None:
            for b in range(self.B):
                for t0 in range(0, self.T, bt):
                    out.append((b * self.T + t0, min(bt, self.T - t0)))
        else:
            cu = self.cu_seqlens.tolist()
            for s in range(len(cu) - 1):
                for t0 in range(cu[s], cu[s + 1], bt):
                    out.append((t0, min(bt, cu[s + 1] - t0)))
        return out


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def _draw_kgb(rng: np.random.Generator, L: int, H: int, kind: str, bt: int = BT, K: int = KEY_DIM):
    """fp64 (k [L, H, K], beta [L, H], g [L, H, K]) of one slab of L tokens, drawn in
    the order k, beta pre-activations, g pre-activations; g restarts at every chunk
    of bt tokens (zero for the "nodecay" kind)."""
    C = (L + bt - 1) // bt
    Lp = C * bt
    k = rng.standard_normal((L, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((L, H))))
    gpre = rng.standard_normal((L, H, K))
    pad = ((0, Lp - L), (0, 0), (0, 0))
    if kind == "nodecay":
        g = np.zeros_like(k)
    elif kind in ("kda", "steep"):
        drop = _softplus(gpre)
        if kind == "steep":
            u = rng.random((L, H, K))
            cls = np.arange(K) % 4
            drop = np.where(cls == 0, 8.0 + 12.0 * u,
                            np.where(cls == 1, drop + 100.0 * (u < 1.0 / 16.0),
                                     np.where(cls == 2, 3.0 + 5.0 * u, drop)))
        g = np.cumsum(-np.pad(drop, pad).reshape(C, bt, H, K), axis=1).reshape(Lp, H, K)[:L]
    else:
        raise ValueError(f"unknown input kind {kind!r}")
    return k, beta, g


def _slab(rng: np.random.Generator, L: int, H: int, kind: str, bt: int = BT) -> np.ndarray:
    """fp64 A for one slab of L tokens: [L, H, bt], strictly lower within each chunk of bt."""
    C = (L + bt - 1) // bt
    Lp = C * bt
    row = np.arange(bt)[:, None]
    col = np.arange(bt)[None, :]
    if kind == "gauss":
        vals = rng.standard_normal((L, H, bt)) * 0.2
        vals = np.concatenate([vals, np.zeros((Lp - L, H, bt))], axis=0)
        S = vals.reshape(C, bt, H, bt)                       # [C, i, H, j]
        keep = (col < row)[None, :, None, :]
    elif kind == "steep":
        raise ValueError("the steep kind is defined for build_kgb only")
    else:
        k, beta, g = _draw_kgb(rng, L, H, kind, bt)
        pad = ((0, Lp - L), (0, 0), (0, 0))
        k = np.pad(k, pad).reshape(C, bt, H, KEY_DIM)
        g = np.pad(g, pad).reshape(C, bt, H, KEY_DIM)
        beta = np.pad(beta, ((0, Lp - L), (0, 0))).reshape(C, bt, H)
        # sum_d (k_i e^{g_i})_d (k_j e^{-g_j})_d, batched over chunks and heads.
        q = torch.from_numpy(np.ascontiguousarray((k * np.exp(g)).transpose(0, 2, 1, 3)))
        kk = torch.from_numpy(np.ascontiguousarray((k * np.exp(-g)).transpose(0, 2, 3, 1)))
        Sc = torch.matmul(q, kk).numpy()                     # [C, H, i, j]
        S = Sc.transpose(0, 2, 1, 3) * beta[..., None]       # [C, i, H, j]
        keep = (col < row)[None, :, None, :]
    # positions past the slab end (only in the padded last chunk) are dropped below
    A = np.where(keep, S, 0.0).reshape(Lp, H, bt)[:L]
    # a partial last chunk: columns >= n_valid are zero by construction (j < i < n_valid)
    return A


def _round(a64: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(a64.astype(np.float32))   # fp64 -> fp32, round to nearest even
    return t.to(_DTYPES[dtype])                     # fp32 -> target, round to nearest even


def build(wl: Workload, poison: bool = False) -> SolverInput:
    """Build the seeded input for ``wl`` on the host.

    ``poison=True`` overwrites every element the solver must ignore (the
    diagonal and upper triangle of each chunk, which includes the columns at
    or past a partial chunk's length) with NaN.
    """
    rng = np.random.default_rng(wl.seed)
    if wl.layout == "dense":
        lens = [wl.T] * wl.B
    elif wl.layout == "packed":
        if wl.ragged is not None:
            n, lo, hi = wl.ragged
            lens = [int(x) for x in rng.integers(lo, hi + 1, size=n)]
        else:
            lens = [int(x) for x in wl.seqlens]
    else:
        raise ValueError(wl.layout)
    bt = wl.bt
    slabs = [_slab(rng, L, wl.H, wl.kind, bt) if L > 0 else np.zeros((0, wl.H, bt)) for L in lens]
    if wl.layout == "dense":
        a = np.stack(slabs, 0) if lens else np.zeros((0, wl.T, wl.H, bt))
        A = _round(a, wl.in_dtype)
        cu = None
    else:
        a = np.concatenate(slabs, 0)[None] if slabs else np.zeros((1, 0, wl.H, bt))
        A = _round(a, wl.in_dtype)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    out = SolverInput(wl, A.contiguous(), cu, lens)
    if poison:
        poison_ignored(out)
    return out


@dataclass
class KgbInput:
    """The inputs the chunk matrices are built from: keys ``k`` [B, T, H, K] and
    ``beta`` [B, T, H] in the input dtype, and the per-channel cumulative log
    decay ``g`` [B, T, H, K] in float32 (restarting at every chunk)."""

    workload: Workload
    k: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: Optional[torch.Tensor]
    seqlens: list = field(default_factory=list)

    @property
    def B(self) -> int:
        return self.k.shape[0]

    @property
    def T(self) -> int:
        return self.k.shape[1]

    @property
    def H(self) -> int:
        return self.k.shape[2]

    @property
    def K(self) -> int:
        return self.k.shape[3]

    @property
    def bt(self) -> int:
        return BT

    def chunks(self):
        """(row0, n_valid) of every 64-token chunk, in order (flattened B*T rows)."""
        return SolverInput.chunks(self)


def build_kgb(wl: Workload, K: int = KEY_DIM) -> KgbInput:
    """Seeded (k, g, beta) for ``wl`` (kinds "kda", "nodecay" and "steep"), drawn exactly as
    for ``build``: with K = 128 and the same workload, the chunk matrices built from
    them by the KDA construction are the ``A`` that ``build`` returns (before rounding)."""
    if wl.kind == "gauss":
        raise ValueError("the gauss kind has no keys and decays")
    rng = np.random.default_rng(wl.seed)
    if wl.layout == "dense":
        lens = [wl.T] * wl.B
    elif wl.layout == "packed":
        if wl.ragged is not None:
            n, lo, hi = wl.ragged
            lens = [int(x) for x in rng.integers(lo, hi + 1, size=n)]
        else:
            lens = [int(x) for x in wl.seqlens]
    else:
        raise ValueError(wl.layout)
    draws = [_draw_kgb(rng, L, wl.H, wl.kind, BT, K) if L > 0 else
             (np.zeros((0, wl.H, K)), np.zeros((0, wl.H)), np.zeros((0, wl.H, K))) for L in lens]
    if wl.layout == "dense":
        k = np.stack([d[0] for d in draws], 0) if lens else np.zeros((0, wl.T, wl.H, K))
        beta = np.stack([d[1] for d in draws], 0) if lens else np.zeros((0, wl.T, wl.H))
        g = np.stack([d[2] for d in draws], 0) if lens else np.zeros((0, wl.T, wl.H, K))
        cu = None
    else:
        k = np.concatenate([d[0] for d in draws], 0)[None]
        beta = np.concatenate([d[1] for d in draws], 0)[None]
        g = np.concatenate([d[2] for d in draws], 0)[None]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    return KgbInput(wl, _round(k, wl.in_dtype).contiguous(), torch.from_numpy(g.astype(np.float32)).contiguous(),
                    _round(beta, wl.in_dtype).contiguous(), cu, lens)


def poison_ignored(inp: SolverInput) -> None:
    """Write NaN into every element of ``inp.A`` the solver is specified to ignore."""
    bt = inp.bt
    flat = inp.A.view(-1, inp.H, bt)
    col = torch.arange(bt)
    for row0, n in inp.chunks():
        i = torch.arange(n)[:, None]
        mask = (col[None, :] >= i)                       # diagonal + upper triangle
        blk = flat[row0:row0 + n]
        blk[mask[:, None, :].expand(n, inp.H, bt)] = float("nan")
