"""Performance regression guards: ratios of times measured in one process, so the
checks hold on any GB300 whatever its clock, and fail only on a cliff (a path that
falls off its vector or tensor-core route), not on ordinary variance.

  * a det_gemm output whose row pitch is not a 16-byte multiple costs at most 1.5x
    (per FLOP) an aligned one (the epilogue keeps 8- / 4-byte vector stores);
  * the two-product backward with an FP32 dC costs at most 1.4x the BF16 one (the
    FP32 -> BF16 cast streams at memory speed);
  * a linear-logp call whose weight must be staged (odd pitch) costs at most 1.8x an
    aligned call at the mid shape (the staging copy streams, the kernels are the same);
  * the mid partials kernel runs at no less than half the fallback BF16 peak.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _median_us(fn, dev, reps=11, flush=True):
    buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    for _ in range(3):
        fn()
    ts = []
    for _ in range(reps):
        if buf is not None:
            buf.zero_()
            buf.view(torch.int64).sum()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e) * 1e3)
    return float(np.median(ts))


def _padded(t, extra, dev):
    r, c = t.shape
    buf = torch.zeros(r, c + extra, dtype=t.dtype, device=dev)
    buf[:, :c] = t
    return buf[:, :c]


def test_odd_output_pitch_keeps_vector_stores(dev):
    M, K = 3000, 2500
    A, B, _ = si.det_gemm_inputs(M, K, 3072, seed=1, device=dev)
    Bn = B[:, :2900]             # a TMA-ready view (pitch 3072): only the output pitch is odd
    odd = _median_us(lambda: rlk.det_gemm_fwd(A, Bn), dev)      # C pitch 5800 B
    even = _median_us(lambda: rlk.det_gemm_fwd(A, B), dev)      # C pitch 6144 B
    assert odd / 2900 <= 1.5 * even / 3072, (odd, even)
    assert rlk.device_error() == 0


def test_fp32_gradient_cast_streams(dev):
    A, B, dC = si.det_gemm_inputs(4096, 4096, 4096, seed=2, device=dev)
    dC32 = dC.float()
    t16 = _median_us(lambda: rlk.det_gemm_backward(dC, A, B), dev)
    t32 = _median_us(lambda: rlk.det_gemm_backward(dC32, A, B), dev)
    assert t32 <= 1.4 * t16, (t32, t16)
    assert rlk.device_error() == 0


def test_staged_weight_streams_and_partials_use_the_tensor_cores(dev):
    w = si.MID
    hidden, weight, _, target = si.workload_inputs(w, seed=3, device=dev)
    staged = _padded(weight, 3, dev)                  # pitch H + 3: copied into the workspace
    call = rlk.LinearLogpCall(hidden, weight, target)
    aligned = _median_us(lambda: rlk.linear_logp(hidden, weight, target), dev, reps=5, flush=False)
    odd = _median_us(lambda: rlk.linear_logp(hidden, staged, target), dev, reps=5, flush=False)
    assert odd <= 1.8 * aligned, (odd, aligned)
    part = _median_us(call.partials, dev, reps=7, flush=False)
    tflops = 2.0 * w.N * w.H * w.V / (part * 1e-6) / 1e12
    assert tflops >= 0.5 * 1900.0, tflops             # half the fallback BF16 peak
    assert rlk.device_error() == 0
