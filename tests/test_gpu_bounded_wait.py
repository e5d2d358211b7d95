"""Failure handling without a GPU fault: a kernel wait that runs out of time.

Every mbarrier wait in the tensor-core kernels is bounded; when one expires the
CTA raises the device error word, winds down and returns, so the CUDA context
stays usable and the host learns of it through rlk_get_device_error.  Here a
diagnostic kernel waits on an mbarrier that nothing completes, with a 50 ms
limit, through that same wait routine.
"""
import ctypes

import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    dev = cuda_or_skip()
    lib = rlk.lib()
    assert rlk.device_error() == 0                       # clean start
    assert lib.rlk_selftest_bounded_wait(0, None) == 2   # limit out of range
    st = lib.rlk_selftest_bounded_wait(50_000, rlk._stream_ptr(None))
    assert st == 0
    flags = ctypes.c_uint32(0)
    assert lib.rlk_get_device_error(rlk._stream_ptr(None), ctypes.byref(flags)) == 8
    assert flags.value == 1                              # RLK_DEVERR_TIMEOUT
    assert rlk.device_error() == 0                       # read-and-clear
    # the context still works: a regular call runs and raises nothing
    hidden, weight, bias, target = si.linear_logp_inputs(40, 256, 600, bias=True, seed=3,
                                                         device=dev)
    logp, lse = rlk.linear_logp(hidden, weight, target, bias)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(lse).all()) and bool((logp <= 0).all())
    assert rlk.device_error() == 0
