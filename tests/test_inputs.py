"""The seeded input generator: determinism, structure and workload shapes."""
import numpy as np
import torch

import kda_inputs as ki


def test_deterministic_and_strictly_lower():
    wl = ki.Workload("t", "packed", H=3, in_dtype="f32", out_dtype="f32", seed=5,
                     seqlens=(70, 1, 64))
    a = ki.build(wl)
    b = ki.build(wl)
    assert torch.equal(a.A, b.A)
    A = a.A.view(-1, 3, 64).double()
    for row0, n in a.chunks():
        blk = A[row0:row0 + n]                       # [n, H, 64]
        i = torch.arange(n)[:, None, None]
        j = torch.arange(64)[None, None, :]
        assert torch.all(blk[(j >= i).expand_as(blk)] == 0)
        assert blk.abs().max() <= 1.0                # |A| <= beta <= 1


def test_kda_decay_shrinks_far_blocks():
    wl = ki.Workload("t", "dense", H=2, in_dtype="f32", out_dtype="f32", seed=6, B=1, T=64)
    A = ki.build(wl).A[0].double()
    near = A[16:32, :, 0:16].abs().max()
    far = A[48:64, :, 0:16].abs().max()
    assert far < 1e-3 * near


def test_workload_shapes():
    wl = ki.WORKLOADS["packed_ragged37_h32_bf16"]
    rng = np.random.default_rng(wl.seed)
    lens = rng.integers(1, 2049, size=37)
    assert lens.min() >= 1 and lens.max() <= 2048
    small = ki.build(ki.WORKLOADS["dense_1x64_h4_f32"])
    assert small.A.shape == (1, 64, 4, 64) and small.A.dtype == torch.float32
    small = ki.build(ki.WORKLOADS["dense_1x64_h64_bf16"])
    assert small.A.shape == (1, 64, 64, 64) and small.A.dtype == torch.bfloat16


def test_poison_marks_only_ignored():
    wl = ki.Workload("t", "packed", H=2, in_dtype="bf16", out_dtype="f32", seed=7,
                     seqlens=(10, 64))
    clean = ki.build(wl)
    dirty = ki.build(wl, poison=True)
    nan = torch.isnan(dirty.A.float())
    assert nan.any()
    assert torch.equal(clean.A[~nan], dirty.A[~nan])
    assert torch.all(clean.A.float()[nan] == 0)
