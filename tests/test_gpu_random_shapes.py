"""A seeded sweep of linear-logp shapes off the tile grid, against the FP64 oracle.

24 (N, H, V) drawn from a fixed generator (H and V mostly not multiples of 64 /
256; N across the one-CTA and 2-SM loops), half with a bias, a few targets out of
range.  For each: lse within 1e-3 absolute of the oracle on every row, logp
within 1e-3 where the target is in [0, V) and NaN where it is not, and the full
call bit-equal to two row chunks split at a drawn row (the operator's batch
invariance).  Every fourth shape also runs the backward and compares
grad_hidden / grad_weight / grad_bias with the oracle's exact gradients within
1e-2 relative Frobenius error (the BF16 rounding of G dominates).
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import LOGP_ATOL, cuda_or_skip, rel_fro

pytestmark = pytest.mark.gpu


def _shapes():
    g = np.random.default_rng(20261203)
    out = []
    for i in range(24):
        N = int(g.choice([1, 2, 5, 31, 64, 127, 128, 129, 200, 255, 256, 257, 400, 700]))
        H = int(g.choice([1, 3, 8, 63, 64, 65, 100, 255, 320, 777, 1024, 1500]))
        V = int(g.choice([1, 2, 255, 256, 257, 1000, 3001, 4099, 9000]))
        out.append((i, N, H, V, bool(i % 2)))
    return out


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


@pytest.mark.parametrize("i,N,H,V,bias", _shapes())
def test_random_shape(dev, orc, i, N, H, V, bias):
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=bias, seed=1000 + i)
    if N >= 3:                                   # out-of-range targets on both sides
        target[0] = -1
        target[N // 2] = V
    hd, wd, td = hidden.to(dev), weight.to(dev), target.to(dev)
    bd = None if b is None else b.to(dev)
    logp, lse = rlk.linear_logp(hd, wd, td, bd)
    torch.cuda.synchronize()
    rlp, rls, _ = orc.linear_logp(si.bf16_bits(hidden), si.bf16_bits(weight), target.numpy(),
                                  None if b is None else b.numpy())
    lp, ls = logp.cpu().double().numpy(), lse.cpu().double().numpy()
    ok = (target.numpy() >= 0) & (target.numpy() < V)
    assert np.all(np.isfinite(ls)) and np.abs(ls - rls).max() <= LOGP_ATOL
    assert np.all(np.isnan(lp[~ok]))
    if ok.any():
        assert np.abs(lp[ok] - rlp[ok]).max() <= LOGP_ATOL
        assert np.all(lp[ok] <= 0.0)
    # batch invariance: two chunks split at a drawn row give the full call's bits
    if N >= 2:
        cut = int(np.random.default_rng(i).integers(1, N))
        parts = [rlk.linear_logp(hd[a:c], wd, td[a:c], bd) for a, c in ((0, cut), (cut, N))]
        cat_lp = torch.cat([p[0] for p in parts])
        cat_ls = torch.cat([p[1] for p in parts])
        assert torch.equal(cat_ls.view(torch.int32), lse.view(torch.int32))
        assert torch.equal(cat_lp.view(torch.int32), logp.view(torch.int32))
    if i % 4 == 0 and N * H * V <= 700 * 1500 * 9000:
        g = torch.randn(N, generator=torch.Generator().manual_seed(i))
        gh, gw, gb = rlk.linear_logp_backward(hd, wd, td, lse, g.to(dev), bd,
                                              out_dtype=torch.float32)
        torch.cuda.synchronize()
        ref_gh, ref_gw, ref_gb, _ = orc.linear_logp_backward(
            si.bf16_bits(hidden), si.bf16_bits(weight), target.numpy(), g.double().numpy(),
            None if b is None else b.numpy())
        for got, ref in ((gh, ref_gh), (gw, ref_gw)):
            if np.abs(ref).max() > 0:
                assert rel_fro(got.cpu().double().numpy(), ref) <= 1e-2
            else:
                assert np.abs(got.cpu().numpy()).max() == 0.0
        if gb is not None and np.abs(ref_gb).max() > 0:
            assert rel_fro(gb.cpu().double().numpy(), ref_gb) <= 1e-2
    assert rlk.device_error() == 0
