"""Shared helpers for the GPU parity tests: device guard, tolerance checks."""
import math

import numpy as np
import pytest
import torch

# Tolerances (stated once, used everywhere):
LOGP_ATOL = 1e-3          # |delta logp|, |delta lse| against the FP64 oracle
GEMM_FP32_REL_FRO = 1e-5  # relative Frobenius error of an FP32-output GEMM
# BF16-output GEMM: within one BF16 ulp of the oracle's exact result rounded to
# BF16, except where cancellation makes the exact result small against the FP32
# accumulation error bound (see bf16_within_one_ulp).


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch.device("cuda:0")


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bit-pattern equality (torch.equal calls -0.0 and +0.0 equal and NaN unequal)."""
    if a.dtype != b.dtype or a.shape != b.shape:
        return False
    if a.dtype in (torch.float32, torch.float16, torch.bfloat16):
        view = torch.int32 if a.dtype == torch.float32 else torch.int16
        return torch.equal(a.contiguous().view(view), b.contiguous().view(view))
    return torch.equal(a, b)


def dec_bf16(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |x| (8 significant bits; subnormal spacing 2^-133)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def bf16_within_one_ulp(gpu_bf16: np.ndarray, ref: np.ndarray, ref_rne_bits: np.ndarray,
                        abs_terms: np.ndarray, K: int):
    """Elementwise BF16 check: one BF16 ulp of the exact result's rounding (RNE).

    gpu_bf16      decoded GPU BF16 outputs
    ref           exact (FP64) results
    ref_rne_bits  the oracle's single rounding of ref to BF16
    abs_terms     sum_k |a_ik b_kj| per element
    Reading of the one-ulp bar for an FP32-accumulating product: an entry whose
    exact value is not cancelled, |ref| >= 2^-8 sum|ab|, must lie within one ulp
    of RNE(ref) with no exception.  Below that ratio the FP32 accumulation error
    (at most K 2^-24 sum|ab|, the textbook bound) can exceed an ulp of the small
    result, and the entry is held to |gpu - ref| <= 1 ulp + K 2^-24 sum|ab|.
    Returns (entries, strict_entries, cancelled_entries, beyond_one_ulp,
    worst |gpu - RNE(ref)| / ulp over the strict entries); raises on failure.
    """
    rne = dec_bf16(ref_rne_bits)
    ulp = np.maximum(bf16_ulp(rne), bf16_ulp(ref))
    strict = np.abs(ref) >= 2.0 ** -8 * abs_terms
    d = np.abs(gpu_bf16 - rne)
    within = d <= ulp
    loose_ok = np.abs(gpu_bf16 - ref) <= ulp + K * 2.0 ** -24 * abs_terms
    bad = np.where(strict, ~within, ~loose_ok)
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{bad.sum()} BF16 outputs off: gpu={gpu_bf16.flat[i]} ref={ref.flat[i]} "
                             f"rne={rne.flat[i]} ulp={ulp.flat[i]} strict={strict.flat[i]}")
    worst = float(np.max(np.where(strict, d / ulp, 0.0))) if d.size else 0.0
    return int(d.size), int(strict.sum()), int((~strict).sum()), int((~within).sum()), worst


def rel_fro(gpu: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(gpu - ref) / (den if den > 0 else 1.0))


def sample_rows(N: int, k: int, seed: int = 0, must=()) -> np.ndarray:
    """Sorted unique rows: the edge rows, the given ones, and k seeded random rows."""
    rng = np.random.default_rng(seed)
    base = {0, N - 1, min(127, N - 1), min(128, N - 1), *[m for m in must if 0 <= m < N]}
    extra = rng.choice(N, size=min(k, N), replace=False) if N > 0 else []
    return np.array(sorted(base.union(int(x) for x in extra)), dtype=np.int64)


def assert_logp_close(logp, lse, ref_logp, ref_lse, what=""):
    lp = np.asarray(logp, np.float64)
    ls = np.asarray(lse, np.float64)
    dl = np.abs(lp - ref_logp)
    ds = np.abs(ls - ref_lse)
    assert np.all(np.isfinite(lp)) and np.all(np.isfinite(ls)), what
    assert dl.max() <= LOGP_ATOL, f"{what}: max |dlogp| = {dl.max()}"
    assert ds.max() <= LOGP_ATOL, f"{what}: max |dlse| = {ds.max()}"
    return float(dl.max()), float(ds.max())


def ln(x):
    return math.log(x)
