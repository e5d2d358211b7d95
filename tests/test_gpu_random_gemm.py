"""A seeded sweep of det_gemm shapes off the tile grid, against the FP64 oracle.

16 (M, K, N) drawn from a fixed generator (extents 1 - 1500, mostly not
multiples of 64 / 256) and four larger ragged ones spanning several waves of
output tiles, each through fwd, dA and dB ("feat(musa): add native
deterministic gemm kernel", Summary), with a BF16 dC or, on every third shape,
an FP32 dC that the library rounds to BF16 first (that page's review comment).
FP32 outputs within relative Frobenius error 1e-5 of the oracle; BF16 outputs
within one BF16 ulp of the exact result's rounding (helpers.bf16_within_one_ulp);
every output bitwise equal on a second call.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import GEMM_FP32_REL_FRO, bf16_within_one_ulp, cuda_or_skip, dec_bf16, rel_fro

pytestmark = pytest.mark.gpu


def _shapes():
    g = np.random.default_rng(31337)
    dims = [1, 2, 7, 33, 64, 65, 127, 129, 255, 257, 300, 511, 640, 1000, 1500]
    drawn = [(i, int(g.choice(dims)), int(g.choice(dims)), int(g.choice(dims))) for i in range(16)]
    # and four that span several waves of output tiles with ragged edges
    return drawn + [(16, 1500, 1000, 1300), (17, 1000, 1500, 257), (18, 777, 2048, 1500),
                    (19, 2049, 640, 1025)]


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _np(t):
    return t.detach().cpu().double().numpy()


@pytest.mark.parametrize("i,M,K,N", _shapes())
def test_random_gemm_shape(dev, orc, i, M, K, N):
    fp32_dc = i % 3 == 2
    A, B, dC = si.det_gemm_inputs(M, K, N, seed=500 + i,
                                  dc_dtype=torch.float32 if fp32_dc else torch.bfloat16)
    Ad, Bd, dCd = A.to(dev), B.to(dev), dC.to(dev)
    a16, b16 = si.bf16_bits(A), si.bf16_bits(B)
    d16 = orc.f32_to_bf16_rne(dC.numpy()) if fp32_dc else si.bf16_bits(dC)
    refs = {"fwd": orc.gemm_fwd(a16, b16), "da": orc.gemm_da(d16, b16), "db": orc.gemm_db(a16, d16)}
    Aab, Bab, Dab = (np.abs(orc.bf16_to_f64(x)) for x in (a16, b16, d16))
    terms = {"fwd": Aab @ Bab, "da": Dab @ Bab.T, "db": Aab.T @ Dab}
    reduced = {"fwd": K, "da": N, "db": M}
    calls = {"fwd": lambda dt: rlk.det_gemm_fwd(Ad, Bd, out_dtype=dt),
             "da": lambda dt: rlk.det_gemm_da(dCd, Bd, out_dtype=dt),
             "db": lambda dt: rlk.det_gemm_db(Ad, dCd, out_dtype=dt)}
    for op, fn in calls.items():
        ref = refs[op]
        out32 = fn(torch.float32)
        out16 = fn(torch.bfloat16)
        again32, again16 = fn(torch.float32), fn(torch.bfloat16)
        torch.cuda.synchronize()
        assert out32.shape == ref.shape and out16.shape == ref.shape, op
        assert torch.equal(out32.view(torch.int32), again32.view(torch.int32)), op
        assert torch.equal(out16.view(torch.int16), again16.view(torch.int16)), op
        if np.abs(ref).max() > 0:
            assert rel_fro(_np(out32), ref) <= GEMM_FP32_REL_FRO, op
        else:
            assert np.abs(_np(out32)).max() == 0.0, op
        bf16_within_one_ulp(dec_bf16(si.bf16_bits(out16)), ref, orc.f64_to_bf16_rne(ref),
                            terms[op], reduced[op])
    assert rlk.device_error() == 0
