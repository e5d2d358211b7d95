"""GPU parity of the linear-layout GEMMs and the FP32 accumulate forward.

"feat(musa): add native deterministic gemm kernel", Implementation: the
transposed-RHS forward / linear(A, weight[N, K]) layout, the canonical transposed
dB for [N, K] weight gradients, and forward_accum_fp32 (read as C += A.B with C
added once after the full K sum).  The oracle's definitions cover them directly:
X.W^T = gemm_da(X, W), dY.W = gemm_fwd(dY, W), dY^T.X = gemm_db(dY, X).
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import (GEMM_FP32_REL_FRO, bf16_within_one_ulp, cuda_or_skip, dec_bf16, rel_fro,
                     sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _inputs(M, K, N, seed, device):
    g = torch.Generator(device=device).manual_seed(seed)
    X = (torch.randn(M, K, generator=g, device=device) / K ** 0.5).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device=device) / K ** 0.5).to(torch.bfloat16)
    dY = torch.randn(M, N, generator=g, device=device)
    return X, W, dY


@pytest.mark.parametrize("shape", [(1, 1, 1), (33, 33, 33), (300, 200, 520), (257, 1000, 129)])
def test_integer_inputs_bit_exact(dev, shape):
    M, K, N = shape
    X = si.integer_bf16((M, K), -16, 16, seed=4)
    W = si.integer_bf16((N, K), -16, 16, seed=5)
    dY = si.integer_bf16((M, N), -16, 16, seed=6)
    x, w, d = (t.float().numpy().astype(np.int64) for t in (X, W, dY))
    f32 = torch.float32
    assert np.array_equal(rlk.det_linear(X.to(dev), W.to(dev), f32).cpu().numpy(), (x @ w.T).astype(np.float32))
    assert np.array_equal(rlk.det_linear_dx(dY.to(dev), W.to(dev), f32).cpu().numpy(), (d @ w).astype(np.float32))
    assert np.array_equal(rlk.det_linear_dw(dY.to(dev), X.to(dev), f32).cpu().numpy(), (d.T @ x).astype(np.float32))
    C = torch.full((M, N), 3.0, device=dev)
    B = W.T.contiguous().to(dev)
    rlk.det_gemm_fwd_accum_fp32_(C, X.to(dev), B)
    assert np.array_equal(C.cpu().numpy(), (x @ w.T + 3).astype(np.float32))


def test_linear_parity_sampled(dev, orc):
    M, K, N = 2048, 4096, 3000
    X, W, dY32 = _inputs(M, K, N, 7, dev)
    rows = sample_rows(M, 32, seed=4)
    Xb, Wb, dYb = si.bf16_bits(X), si.bf16_bits(W), orc.f32_to_bf16_rne(dY32.cpu().numpy())
    cases = [
        ("fwd", lambda o: rlk.det_linear(X, W, o), lambda: orc.gemm_da(Xb, Wb, rows=rows), rows, K),
        ("dx", lambda o: rlk.det_linear_dx(dY32, W, o), lambda: orc.gemm_fwd(dYb, Wb, rows=rows), rows, N),
        ("dw", lambda o: rlk.det_linear_dw(dY32, X, o), lambda: orc.gemm_db(dYb, Xb, rows=sample_rows(N, 32)),
         sample_rows(N, 32), M),
    ]
    for name, run, ref_fn, r, red in cases:
        out32 = run(torch.float32)
        out16 = run(torch.bfloat16)
        torch.cuda.synchronize()
        ref = ref_fn()
        assert rel_fro(out32.cpu().numpy()[r].astype(np.float64), ref) <= GEMM_FP32_REL_FRO, name
        assert torch.equal(out16, out32.to(torch.bfloat16)), name
        # one-ulp check against the exact result's BF16 rounding
        if name == "fwd":
            terms = np.abs(X.cpu().double().numpy()[r]) @ np.abs(W.cpu().double().numpy()).T
        elif name == "dx":
            terms = np.abs(dec_bf16(dYb)[r]) @ np.abs(W.cpu().double().numpy())
        else:
            terms = np.abs(dec_bf16(dYb)).T[r] @ np.abs(X.cpu().double().numpy())
        n, strict, cancelled, beyond, worst = bf16_within_one_ulp(
            dec_bf16(si.bf16_bits(out16)[r]), ref, orc.f64_to_bf16_rne(ref), terms, red)
        print(f"BF16 classes det_linear {name}: entries={n} strict={strict} "
              f"cancellation-bound={cancelled} beyond one ulp={beyond} worst strict={worst:.3f} ulp")
    assert rlk.device_error() == 0


def test_fp32_grad_is_rounded_first(dev):
    X, W, dY32 = _inputs(500, 384, 264, 8, dev)
    dYb = dY32.to(torch.bfloat16)
    for out in (torch.float32, torch.bfloat16):
        assert torch.equal(rlk.det_linear_dx(dY32, W, out), rlk.det_linear_dx(dYb, W, out))
        assert torch.equal(rlk.det_linear_dw(dY32, X, out), rlk.det_linear_dw(dYb, X, out))


def test_accumulate_equals_fp32_sum(dev):
    A, B, _ = si.det_gemm_inputs(700, 1000, 520, seed=9, device=dev)
    C0 = torch.randn(700, 520, device=dev)
    C = C0.clone()
    rlk.det_gemm_fwd_accum_fp32_(C, A, B)
    assert torch.equal(C, C0 + rlk.det_gemm_fwd(A, B, out_dtype=torch.float32))
    # a strided (wider-pitch) C is updated in place, the pad untouched
    big = torch.full((700, 640), 7.0, device=dev)
    big[:, :520] = C0
    rlk.det_gemm_fwd_accum_fp32_(big[:, :520], A, B)
    assert torch.equal(big[:, :520], C)
    assert bool((big[:, 520:] == 7.0).all())


def test_rows_independent_and_run_to_run(dev):
    X, W, dY32 = _inputs(1000, 768, 640, 10, dev)
    full = rlk.det_linear(X, W, torch.float32)
    parts = [rlk.det_linear(X[s:s + 7], W, torch.float32) for s in range(0, 1000, 7)]
    assert torch.equal(torch.cat(parts), full)
    full_dx = rlk.det_linear_dx(dY32, W)
    parts = [rlk.det_linear_dx(dY32[s:s + 129], W) for s in range(0, 1000, 129)]
    assert torch.equal(torch.cat(parts), full_dx)
    first = rlk.det_linear_dw(dY32, X)
    for _ in range(3):
        assert torch.equal(rlk.det_linear_dw(dY32, X), first)
    # 3-D activations are rows
    Y3 = rlk.det_linear(X.view(10, 100, 768), W, torch.float32)
    assert Y3.shape == (10, 100, 640) and torch.equal(Y3.reshape(1000, 640), full)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_trainable_autograd_matches_the_backward_entries(dev, out_dtype):
    """det_gemm_trainable / det_linear_trainable under autograd: forwards bitwise
    equal to det_gemm_fwd / det_linear, gradients bitwise equal to the two-product
    backward entries with the same upstream gradient (an FP32 one rounded to BF16
    once), for a 3-D left operand."""
    g = torch.Generator(device=dev).manual_seed(5)
    A = (torch.randn(3, 100, 384, generator=g, device=dev) / 20).to(torch.bfloat16)
    B = (torch.randn(384, 200, generator=g, device=dev) / 20).to(torch.bfloat16)
    W = (torch.randn(200, 384, generator=g, device=dev) / 20).to(torch.bfloat16)
    up = torch.randn(3, 100, 200, generator=g, device=dev)
    a, b, w = (t.clone().requires_grad_() for t in (A, B, W))
    C = rlk.det_gemm_trainable(a, b, out_dtype)
    assert torch.equal(C.detach(), rlk.det_gemm_fwd(A, B, out_dtype))
    (C.float() * up).sum().backward()
    dC = up.to(out_dtype)
    dA, dB = rlk.det_gemm_backward(dC, A, B)
    assert torch.equal(a.grad, dA.reshape(A.shape)) and torch.equal(b.grad, dB)
    a2 = A.clone().requires_grad_()
    Y = rlk.det_linear_trainable(a2, w, out_dtype)
    assert torch.equal(Y.detach(), rlk.det_linear(A, W, out_dtype))
    (Y.float() * up).sum().backward()
    dX, dW = rlk.det_linear_backward(up.to(out_dtype), A, W)
    assert torch.equal(a2.grad, dX.reshape(A.shape)) and torch.equal(w.grad, dW)
    # only the requested gradient is formed
    b3 = B.clone().requires_grad_()
    rlk.det_gemm_trainable(A, b3, out_dtype).float().sum().backward()
    assert b3.grad is not None and b3.grad.dtype == torch.bfloat16
