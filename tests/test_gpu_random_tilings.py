"""The det_gemm tiling never changes a bit: seeded random shapes whose products are
computed whole and as row chunks of random sizes, so that the same output rows run
under different tile plans (128-wide tiles throughout, 256-wide tiles, 224-wide tiles
for dA, a last wave split into 128-wide halves), compared bit for bit; random BF16
inputs (not integers), FP32 and BF16 outputs.  The plans are read back through
rlk_det_gemm_tile_plan and the module checks that every kind occurred.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import bits_equal, cuda_or_skip

pytestmark = pytest.mark.gpu

SEEN = set()


def _cases():
    g = np.random.default_rng(20261204)
    out = []
    for i in range(10):
        out.append((i, int(g.choice([1792, 2304, 3000, 4096])), int(g.choice([640, 2048, 4096])),
                    int(g.choice([1500, 3900, 4096]))))
    out.append((10, 4096, 16384, 3900))          # a long reduction: split last waves
    return out


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _note(op, rows, cols, red, sms):
    p = rlk.det_gemm_tile_plan(op, rows, cols, red, sms)
    SEEN.add("split" if p["split_blocks"] else p["tile_cols"])


@pytest.mark.parametrize("i,M,K,N", _cases())
def test_row_chunks_across_tilings(dev, i, M, K, N):
    out_dtype = torch.float32 if i % 2 == 0 else torch.bfloat16
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    A, B, dC = si.det_gemm_inputs(M, K, N, seed=900 + i, device=dev)
    rng = np.random.default_rng(i)

    def bounds(n):
        cuts = sorted(set(int(c) for c in rng.integers(1, n, 3)))
        return list(zip([0] + cuts, cuts + [n]))

    # fwd [M, N] over K and dA [M, K] over N: chunks of A's / dC's rows
    for op, code, whole, part, cols, red in (
            ("fwd", rlk.RLK_GEMM_FWD, lambda: rlk.det_gemm_fwd(A, B, out_dtype),
             lambda a, b: rlk.det_gemm_fwd(A[a:b], B, out_dtype), N, K),
            ("da", rlk.RLK_GEMM_DA, lambda: rlk.det_gemm_da(dC, B, out_dtype),
             lambda a, b: rlk.det_gemm_da(dC[a:b], B, out_dtype), K, N)):
        full = whole()
        chunks = bounds(M)
        got = torch.cat([part(a, b) for a, b in chunks])
        assert bits_equal(got, full), (op, chunks)
        for a, b in [(0, M)] + chunks:
            _note(code, b - a, cols, red, sms)
    # dB [K, N] over M: chunks of A's columns (odd offsets are staged, bit for bit)
    full = rlk.det_gemm_db(A, dC, out_dtype)
    chunks = bounds(K)
    got = torch.cat([rlk.det_gemm_db(A[:, a:b], dC, out_dtype) for a, b in chunks])
    assert bits_equal(got, full), ("db", chunks)
    for a, b in [(0, K)] + chunks:
        _note(rlk.RLK_GEMM_DB, b - a, N, M, sms)
    assert rlk.device_error() == 0


def test_every_tiling_occurred(dev):
    if torch.cuda.get_device_properties(dev).multi_processor_count != 152:
        pytest.skip("the shapes are chosen for 76 SM pairs")
    assert {128, 224, 256, "split"} <= SEEN, SEEN
