"""Device-side failure detection without a GPU fault (GPU).

Every wait of the library's kernels on an mbarrier (a TMA copy's arrival, a
hand-off between warps) is bounded: after its limit the kernel records bit 1 in
the device error word and returns, so a copy that never lands stops the kernel
instead of hanging the GPU.  kda_selftest_wait runs that wait on an mbarrier that
nothing completes (a short limit), which is how the tests make it run out; the
context must stay usable and the word must read back and clear.
"""
from __future__ import annotations

import ctypes
import time

import pytest
import torch

import kda_inputs as ki

pytestmark = pytest.mark.gpu

ERR_WAIT_TIMEOUT = 1


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_chunked_02_gb300 import build as kbuild
    kbuild.build()
    import linear_attention_chunked_02_gb300 as k
    return k


def selftest(kda, complete, limit_us):
    s = torch.cuda.current_stream()
    st = kda.lib().kda_selftest_wait(complete, limit_us, ctypes.c_void_p(s.cuda_stream))
    assert st == 0
    t0 = time.time()
    torch.cuda.synchronize()
    return time.time() - t0


def test_completed_wait_records_nothing(kda):
    assert kda.device_error() == 0                   # clear anything earlier
    selftest(kda, 1, 2000)
    assert kda.device_error() == 0


def test_wait_that_never_completes_is_reported_and_returns(kda):
    assert kda.device_error() == 0
    took = selftest(kda, 0, 2000)
    assert took < 5.0, took                          # 2 ms limit, checked every 64 suspended tries
    assert kda.device_error() == ERR_WAIT_TIMEOUT
    assert kda.device_error() == 0                   # reading clears the word


def test_context_stays_usable_after_a_timeout(kda):
    selftest(kda, 0, 1000)
    assert kda.device_error() == ERR_WAIT_TIMEOUT
    inp = ki.build(ki.WORKLOADS["dense_1x64_h4_f32"])
    A = inp.A.to("cuda:0")
    out = kda.solve_tril(A, out_dtype=torch.float32, path="single")
    ref = kda.solve_tril(A, out_dtype=torch.float32, path="split")
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and bool(torch.isfinite(out).all())
    assert kda.device_error() == 0
