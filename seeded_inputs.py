"""Seeded synthetic inputs for the linear-logp and det_gemm workloads.

This module is the one piece shared by the CUDA path's tests/bench and the
FP64 oracle: it draws random numbers and rounds them to the storage dtypes
(BF16 operands, FP32 bias/dC, int64 targets).  It holds none of the method's
arithmetic — no dot product, no log-sum-exp, no GEMM.

Value distributions follow the workloads named for the operators:
  * hidden  ~ N(0, 1)            (std 1)
  * weight  ~ N(0, 1/sqrt(H))    (std 1/sqrt(H), so logits are ~ N(0, 1))
  * bias    ~ N(0, 0.01)         (std 0.01, fp32)
  * targets uniform int64 in [0, V); the "large" workload additionally sets
    exactly floor(0.1 * N) seeded positions to id 0.
  * det_gemm A, B ~ N(0, 1/sqrt(K)), dC ~ N(0, 1).
The "sigma" in N(0, sigma) is read as the standard deviation.

Draw order inside one generator is fixed: hidden -> weight -> bias -> targets
(and A -> B -> dC for det_gemm), so a (seed, shape) pair fixes every bit.
Small cases draw on the CPU; the full-size workloads may draw on a CUDA
device with a seeded CUDA generator (same bits every run on that device), and
whoever checks them copies the very same tensors to the host.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class LinearLogpWorkload:
    name: str
    N: int
    H: int
    V: int
    bias: bool
    target_mode: str = "uniform"      # "uniform" | "uniform+10pct_id0"
    lead_shape: tuple = field(default=())  # e.g. (8, 2048) for packed sequences


@dataclass(frozen=True)
class DetGemmWorkload:
    name: str
    M: int
    K: int
    N: int
    batch: int = 1                     # A is [batch, M/batch, K] when batch > 1


# Named workloads (sizes of the linear-logp and det_gemm configurations).
TINY = LinearLogpWorkload("linear-logp tiny", N=64, H=256, V=1024, bias=True)
MID = LinearLogpWorkload("linear-logp mid", N=4096, H=4096, V=151936, bias=False)
LARGE = LinearLogpWorkload("linear-logp large", N=16384, H=5120, V=152064, bias=True,
                           target_mode="uniform+10pct_id0", lead_shape=(8, 2048))
RAGGED_N = (1, 3, 17, 255, 1024, 8191)


def ragged(N: int) -> LinearLogpWorkload:
    return LinearLogpWorkload(f"linear-logp ragged N={N}", N=N, H=2048, V=32003, bias=False)


DET_GEMM = DetGemmWorkload("det_gemm 4096^3", M=4096, K=4096, N=4096)
DET_GEMM_3D = DetGemmWorkload("det_gemm batched [8,512,4096]", M=4096, K=4096, N=4096, batch=8)
DET_GEMM_RAGGED = (1, 33, 1000)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def linear_logp_inputs(N: int, H: int, V: int, *, bias: bool = False, seed: int = 0,
                       target_mode: str = "uniform", device="cpu"):
    """Draw (hidden bf16 [N,H], weight bf16 [V,H], bias fp32 [V] | None, target int64 [N])."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    hidden = torch.randn(N, H, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    weight = (torch.randn(V, H, generator=g, device=dev, dtype=torch.float32)
              * (1.0 / math.sqrt(H))).to(torch.bfloat16)
    b = None
    if bias:
        b = torch.randn(V, generator=g, device=dev, dtype=torch.float32) * 0.01
    target = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int64)
    if target_mode == "uniform+10pct_id0":
        n0 = (N * 10) // 100
        pos = torch.randperm(N, generator=g, device=dev)[:n0]
        target[pos] = 0
    elif target_mode != "uniform":
        raise ValueError(f"unknown target_mode {target_mode!r}")
    return hidden, weight, b, target


def workload_inputs(w: LinearLogpWorkload, *, seed: int = 0, device="cpu"):
    return linear_logp_inputs(w.N, w.H, w.V, bias=w.bias, seed=seed,
                              target_mode=w.target_mode, device=device)


def det_gemm_inputs(M: int, K: int, N: int, *, seed: int = 0, device="cpu",
                    dc_dtype=torch.bfloat16):
    """Draw (A bf16 [M,K], B bf16 [K,N], dC [M,N] in dc_dtype)."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    s = 1.0 / math.sqrt(K)
    A = (torch.randn(M, K, generator=g, device=dev) * s).to(torch.bfloat16)
    B = (torch.randn(K, N, generator=g, device=dev) * s).to(torch.bfloat16)
    dC = torch.randn(M, N, generator=g, device=dev).to(dc_dtype)
    return A, B, dC


def integer_bf16(shape, lo: int, hi: int, *, seed: int = 0, device="cpu"):
    """Integer-valued BF16 tensor with entries uniform in [lo, hi] (exact in BF16 for |x| <= 256)."""
    g = _gen(seed, torch.device(device))
    return torch.randint(lo, hi + 1, shape, generator=g, device=device).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a BF16 tensor's bit patterns (contiguous copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
