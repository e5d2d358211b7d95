"""The allocation-free linear-logp entry point, rlk_linear_logp_noalloc.

It serves callers that cannot allocate device memory where they call the
operator: a plugin inside a host framework that owns the device allocator, code
held to a device-memory budget fixed in advance, or a latency-critical loop that
must not call cudaMalloc / cudaFree.  Its scratch is a fixed 32 MiB array in the
library's device image instead of a caller workspace.

These tests call it through the C ABI and compare its outputs with those of the
regular entry point, rlk_linear_logp (workspace allocated by the caller), on two
calls in a row; the results must agree within the parity tolerance used
everywhere (|delta| <= 1e-3), and in fact bit for bit, since both run the same
kernels.  This file is collected last so that, if it fails, a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import LOGP_ATOL, cuda_or_skip

pytestmark = pytest.mark.gpu


def _noalloc(hidden, weight, target, bias, logp, lse, zt):
    f = rlk.lib().rlk_linear_logp_noalloc
    N, H = hidden.shape
    V = weight.size(0)
    return f(rlk._ptr(hidden), N, H, hidden.stride(0), rlk._ptr(weight), V, weight.stride(0),
             rlk._ptr(bias), rlk._ptr(target), target.stride(0), rlk._ptr(logp), rlk._ptr(lse),
             rlk._ptr(zt), rlk._stream_ptr(None))


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    dev = cuda_or_skip()
    for seed, (N, H, V, bias) in ((31, (300, 1024, 40000, True)), (32, (1000, 2048, 32003, False))):
        hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=bias, seed=seed, device=dev)
        ref_logp, ref_lse, ref_zt = rlk.linear_logp(hidden, weight, target, b,
                                                    return_target_logit=True)
        logp = torch.full((N,), float("nan"), device=dev)
        lse = torch.full((N,), float("nan"), device=dev)
        zt = torch.full((N,), float("nan"), device=dev)
        assert _noalloc(hidden, weight, target, b, logp, lse, zt) == 0
        torch.cuda.synchronize()
        for got, ref in ((logp, ref_logp), (lse, ref_lse), (zt, ref_zt)):
            assert float((got - ref).abs().max()) <= LOGP_ATOL
            assert torch.equal(got, ref)
    assert rlk.device_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    dev = cuda_or_skip()
    # 7200 rows x 594 splits x 8 bytes > 32 MiB: refused before anything launches
    N, H, V = 7200, 64, 151936
    hidden = torch.zeros(N, H, dtype=torch.bfloat16, device=dev)
    weight = torch.zeros(V, H, dtype=torch.bfloat16, device=dev)
    target = torch.zeros(N, dtype=torch.int64, device=dev)
    logp = torch.full((N,), -5.0, device=dev)
    lse = torch.full((N,), -5.0, device=dev)
    assert _noalloc(hidden, weight, target, None, logp, lse, None) == 5   # RLK_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((logp == -5.0).all()) and bool((lse == -5.0).all())
