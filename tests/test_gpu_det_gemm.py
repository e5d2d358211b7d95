"""GPU parity of the deterministic GEMM family against the FP64 oracle.

"feat(musa): add native deterministic gemm kernel", Summary: C = A B,
dA = dC B^T, dB = A^T dC, FP32 accumulation in ascending K order, BF16 or FP32
output; review comment: an FP32 dC (gradient of an FP32-output forward) is
rounded to BF16 before dA / dB.  Tolerances: FP32 output within relative
Frobenius error 1e-5; BF16 output within one BF16 ulp of the exact result's
rounding (see helpers.bf16_within_one_ulp); integer-valued inputs bit-exact.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import (GEMM_FP32_REL_FRO, bits_equal, bf16_within_one_ulp, cuda_or_skip, dec_bf16, rel_fro,
                     sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def np64(t):
    return t.detach().cpu().double().numpy()


def call(op, x, y, out_dtype):
    f = {"fwd": rlk.det_gemm_fwd, "da": rlk.det_gemm_da, "db": rlk.det_gemm_db}[op]
    out = f(x, y, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out


def oracle(orc, op, x, y, rows=None):
    xb = si.bf16_bits(x) if x.dtype == torch.bfloat16 else orc.f32_to_bf16_rne(x.cpu().numpy())
    yb = si.bf16_bits(y) if y.dtype == torch.bfloat16 else orc.f32_to_bf16_rne(y.cpu().numpy())
    return {"fwd": orc.gemm_fwd, "da": orc.gemm_da, "db": orc.gemm_db}[op](xb, yb, rows=rows)


def abs_terms(op, x, y, rows):
    """sum_k |a_ik b_kj| for the sampled output rows (numpy float64)."""
    X = np.abs(np64(x.float().to(torch.bfloat16)))
    Y = np.abs(np64(y.float().to(torch.bfloat16)))
    if op == "fwd":
        return X[rows] @ Y
    if op == "da":
        return X[rows] @ Y.T
    return X.T[rows] @ Y


OPS = ["fwd", "da", "db"]


def operands(op, A, B, dC):
    return {"fwd": (A, B), "da": (dC, B), "db": (A, dC)}[op]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (33, 33, 33), (128, 64, 256), (300, 200, 520),
                                   (257, 1000, 129)])
def test_integer_inputs_bit_exact(dev, op, shape):
    """|a|, |b| <= 16 with K <= 4096: every partial sum is an integer below 2^24,
    so the FP32 result is exact in any order and must equal int64 matmul."""
    M, K, N = shape
    A = si.integer_bf16((M, K), -16, 16, seed=1)
    B = si.integer_bf16((K, N), -16, 16, seed=2)
    dC = si.integer_bf16((M, N), -16, 16, seed=3)
    x, y = operands(op, A, B, dC)
    out = call(op, x.to(dev), y.to(dev), torch.float32)
    a, b, d = (t.float().numpy().astype(np.int64) for t in (A, B, dC))
    want = {"fwd": a @ b, "da": d @ b.T, "db": a.T @ d}[op]
    assert np.array_equal(out.cpu().numpy().astype(np.int64), want)
    assert np.array_equal(out.cpu().numpy(), want.astype(np.float32))


@pytest.mark.parametrize("op", OPS)
def test_4096_parity_sampled(dev, orc, op):
    A, B, dC = si.det_gemm_inputs(4096, 4096, 4096, seed=0, device=dev)
    x, y = operands(op, A, B, dC)
    c32 = call(op, x, y, torch.float32)
    c16 = call(op, x, y, torch.bfloat16)
    rows = sample_rows(4096, 40, seed=3, must=(255, 256, 4000))
    ref = oracle(orc, op, x, y, rows)
    assert rel_fro(c32.cpu().numpy()[rows].astype(np.float64), ref) <= GEMM_FP32_REL_FRO
    # BF16 output: the epilogue's rounding of the very same accumulator ...
    assert torch.equal(c16, c32.to(torch.bfloat16))
    # ... and within one BF16 ulp of the exact result's rounding
    g = dec_bf16(si.bf16_bits(c16)[rows])
    n, strict, cancelled, beyond, worst = bf16_within_one_ulp(
        g, ref, orc.f64_to_bf16_rne(ref), abs_terms(op, x, y, rows), 4096)
    print(f"BF16 classes det_gemm {op} 4096^3, {len(rows)} rows: entries={n} strict={strict} "
          f"cancellation-bound={cancelled} beyond one ulp={beyond} (all cancellation-bound) "
          f"worst strict |gpu - RNE(exact)| = {worst:.3f} ulp")
    assert n == ref.size and strict + cancelled == n
    assert rlk.device_error() == 0


@pytest.mark.parametrize("n", si.DET_GEMM_RAGGED)
def test_ragged_fp32_output_backward(dev, orc, n):
    """FP32-output forward, then dA / dB from an FP32 grad rounded to BF16."""
    A, B, _ = si.det_gemm_inputs(n, n, n, seed=n, device="cpu")
    dC32 = torch.randn(n, n, generator=torch.Generator().manual_seed(n + 1))
    C = call("fwd", A.to(dev), B.to(dev), torch.float32)
    assert C.dtype == torch.float32
    ref = oracle(orc, "fwd", A, B)
    assert rel_fro(np64(C), ref) <= GEMM_FP32_REL_FRO
    for op, (x, y) in (("da", (dC32, B)), ("db", (A, dC32))):
        for out_dtype in (torch.float32, torch.bfloat16):
            out = call(op, x.to(dev), y.to(dev), out_dtype)
            ref = oracle(orc, op, x, y)                  # oracle rounds dC with its own RNE
            if out_dtype == torch.float32:
                assert rel_fro(np64(out), ref) <= GEMM_FP32_REL_FRO, (op, n)
            else:
                rows = np.arange(ref.shape[0])
                bf16_within_one_ulp(dec_bf16(si.bf16_bits(out)), ref, orc.f64_to_bf16_rne(ref),
                                    abs_terms(op, x, y, rows), n)
            # the FP32 grad path equals feeding the BF16-rounded grad directly
            xb = x.to(torch.bfloat16) if x.dtype == torch.float32 else x
            yb = y.to(torch.bfloat16) if y.dtype == torch.float32 else y
            assert torch.equal(out, call(op, xb.to(dev), yb.to(dev), out_dtype))


def test_batched_3d_is_flattened(dev):
    """A[8, 512, 4096]: forward and dA equal the flattened 2-D call and each
    batch slice on its own (row invariance); dB sums over all 4096 rows."""
    A, B, dC = si.det_gemm_inputs(4096, 4096, 4096, seed=5, device=dev)
    A3, dC3 = A.view(8, 512, 4096), dC.view(8, 512, 4096)
    C3 = rlk.det_gemm_fwd(A3, B)
    assert C3.shape == (8, 512, 4096)
    assert torch.equal(C3.reshape(4096, 4096), rlk.det_gemm_fwd(A, B))
    for b in (0, 3, 7):
        assert torch.equal(C3[b], rlk.det_gemm_fwd(A3[b], B))
    dA3 = rlk.det_gemm_da(dC3, B)
    assert torch.equal(dA3.reshape(4096, 4096), rlk.det_gemm_da(dC, B))
    assert torch.equal(dA3[5], rlk.det_gemm_da(dC3[5], B))
    assert torch.equal(rlk.det_gemm_db(A3, dC3), rlk.det_gemm_db(A, dC))


def test_run_to_run_bitwise(dev):
    A, B, dC = si.det_gemm_inputs(4096, 4096, 4096, seed=6, device=dev)
    for op in OPS:
        x, y = operands(op, A, B, dC)
        first = call(op, x, y, torch.bfloat16)
        first32 = call(op, x, y, torch.float32)
        for _ in range(4):
            assert torch.equal(call(op, x, y, torch.bfloat16), first)
            assert torch.equal(call(op, x, y, torch.float32), first32)


def test_row_chunking_bitwise(dev):
    """fwd / dA rows do not depend on which other rows are in the call."""
    A, B, dC = si.det_gemm_inputs(1000, 768, 640, seed=7, device=dev)
    full = rlk.det_gemm_fwd(A, B, out_dtype=torch.float32)
    for chunk in (1, 7, 129):
        parts = [rlk.det_gemm_fwd(A[s:s + chunk], B, out_dtype=torch.float32)
                 for s in range(0, 1000, chunk)]
        assert torch.equal(torch.cat(parts), full)
    full_da = rlk.det_gemm_da(dC, B)
    parts = [rlk.det_gemm_da(dC[s:s + 77], B) for s in range(0, 1000, 77)]
    assert torch.equal(torch.cat(parts), full_da)


def test_strided_and_misaligned_operands_bitwise(dev):
    """A leading dimension wider than the row, an odd pitch (staged through the
    workspace) and a contiguous copy all give the same bits."""
    A, B, dC = si.det_gemm_inputs(300, 200, 264, seed=8, device=dev)
    ref = rlk.det_gemm_fwd(A, B)
    wide = torch.zeros(300, 264, dtype=torch.bfloat16, device=dev)
    wide[:, :200] = A
    assert torch.equal(rlk.det_gemm_fwd(wide[:, :200], B), ref)
    odd = torch.zeros(300, 201, dtype=torch.bfloat16, device=dev)
    odd[:, :200] = A
    assert torch.equal(rlk.det_gemm_fwd(odd[:, :200], B), ref)
    oddB = torch.zeros(200, 265, dtype=torch.bfloat16, device=dev)
    oddB[:, :264] = B
    assert torch.equal(rlk.det_gemm_fwd(A, oddB[:, :264]), ref)
    ref_db = rlk.det_gemm_db(A, dC)
    oddd = torch.zeros(300, 265, dtype=torch.bfloat16, device=dev)
    oddd[:, :264] = dC
    assert torch.equal(rlk.det_gemm_db(odd[:, :200], oddd[:, :264]), ref_db)


def test_output_guard_bands(dev):
    """Writes stay inside the output: canaries around a strided output survive."""
    A, B, _ = si.det_gemm_inputs(33, 40, 33, seed=9, device=dev)
    canary = torch.full((35, 48), -7.0, dtype=torch.float32, device=dev)
    out = canary[1:34, 2:35]
    st = rlk.lib().rlk_det_gemm_fwd(
        rlk._ptr(A), 33, 40, 40, rlk._ptr(B), 33, 33, rlk._ptr(out), rlk.RLK_FP32, 48,
        None, 0, rlk._stream_ptr(None))
    # B's pitch (33) needs staging: without a workspace the call must refuse
    assert st == 5
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=dev)
    st = rlk.lib().rlk_det_gemm_fwd(
        rlk._ptr(A), 33, 40, 40, rlk._ptr(B), 33, 33, rlk._ptr(out), rlk.RLK_FP32, 48,
        rlk._ptr(ws), ws.numel(), rlk._stream_ptr(None))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out, rlk.det_gemm_fwd(A, B, out_dtype=torch.float32))
    mask = torch.ones_like(canary, dtype=torch.bool)
    mask[1:34, 2:35] = False
    assert bool((canary[mask] == -7.0).all())


def test_db_empty_reduction_is_zero(dev):
    A = torch.empty(0, 24, dtype=torch.bfloat16, device=dev)
    dC = torch.empty(0, 40, dtype=torch.bfloat16, device=dev)
    out = rlk.det_gemm_db(A, dC, out_dtype=torch.float32)
    assert out.shape == (24, 40) and bool((out == 0).all())


@pytest.mark.parametrize("dc_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(300, 200, 520), (1000, 1000, 1000), (33, 33, 33), (0, 64, 96),
                                   (4096, 4096, 4096), (3000, 2500, 2900)])
def test_two_product_backward_equals_separate_calls(dev, dc_dtype, shape):
    """rlk_det_gemm_backward (one shared BF16 rounding of an FP32 dC) and
    rlk_det_linear_backward give exactly the bits of the separate dA / dB (dX / dW)
    calls, with aligned and staged (odd-pitch) operands, and with M = 0 (empty dA,
    zero dB).  The last two shapes give each product at least a wave of tiles with
    comparable reductions, so both products run in one launch."""
    M, K, N = shape
    A, B, dC = si.det_gemm_inputs(max(M, 1), K, N, seed=M + K + N, device=dev, dc_dtype=dc_dtype)
    A, dC = A[:M], dC[:M]
    for out in (torch.float32, torch.bfloat16):
        dA, dB = rlk.det_gemm_backward(dC, A, B, out)
        assert torch.equal(dA, rlk.det_gemm_da(dC, B, out))
        assert torch.equal(dB, rlk.det_gemm_db(A, dC, out))
        W = B.T.contiguous()                                   # [N, K]
        dX, dW = rlk.det_linear_backward(dC, A, W, out)
        assert torch.equal(dX, rlk.det_linear_dx(dC, W, out))
        assert torch.equal(dW, rlk.det_linear_dw(dC, A, out))
    if M > 0:
        odd = torch.zeros(M, K + 3, dtype=torch.bfloat16, device=dev)
        odd[:, :K] = A
        dA2, dB2 = rlk.det_gemm_backward(dC, odd[:, :K], B, torch.float32)
        assert torch.equal(dA2, rlk.det_gemm_da(dC, B, torch.float32))
        assert torch.equal(dB2, rlk.det_gemm_db(A, dC, torch.float32))
        only_b = rlk.det_gemm_backward(dC, A, B, torch.float32, grad_a=False)
        assert only_b[0] is None and torch.equal(only_b[1], dB2)
    else:
        assert bool((rlk.det_gemm_backward(dC, A, B, torch.float32)[1] == 0).all())
    assert rlk.device_error() == 0


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tile_widths_give_the_same_bits(dev, out_dtype):
    """Outputs whose 256-wide tiles would leave at least half the CTA pairs idle use
    128-wide tiles.  A 256-row chunk of a 4096-row product (8 wide tiles: narrow
    tiles) must equal the same rows of the full product (128 wide tiles: wide)
    bit for bit, for the forward (MN-major right operand) and dA (K-major)."""
    M, K, N = 4096, 1024, 2048
    A, B, dC = si.det_gemm_inputs(M, K, N, seed=12, device=dev)
    full_f = rlk.det_gemm_fwd(A, B, out_dtype)
    full_a = rlk.det_gemm_da(dC, B, out_dtype)
    for r0 in (0, 256, 3840):
        rows = slice(r0, r0 + 256)
        assert torch.equal(rlk.det_gemm_fwd(A[rows], B, out_dtype), full_f[rows])
        assert torch.equal(rlk.det_gemm_da(dC[rows], B, out_dtype), full_a[rows])
    # a ragged narrow case: 33 rows x 2000 columns against the same rows of 4096
    assert torch.equal(rlk.det_gemm_fwd(A[100:133], B[:, :2000], out_dtype),
                       rlk.det_gemm_fwd(A, B[:, :2000], out_dtype)[100:133])
    assert rlk.device_error() == 0


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_mid_width_tiles_give_the_same_bits(dev, out_dtype):
    """dA and the linear forward read their right operand K-major; a 4096 x 4096 output
    runs 19 x 16 = 304 tiles 224 wide (4 full waves on 76 SM pairs) instead of 256
    tiles 256 wide.  Integer inputs give the exact product, and its rows equal the
    same rows of a 2304-row call (256-wide tiles), a 1792-row call (224) and 256-row
    calls (128-wide tiles), bit for bit."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    DA, LIN = rlk.RLK_GEMM_DA, rlk.RLK_GEMM_LINEAR_FWD
    if sms == 152:
        assert rlk.det_gemm_tile_plan(DA, 4096, 4096, 4096, sms)["tile_cols"] == 224
        assert rlk.det_gemm_tile_plan(DA, 2304, 4096, 4096, sms)["tile_cols"] == 256
        assert rlk.det_gemm_tile_plan(DA, 1792, 4096, 4096, sms)["tile_cols"] == 224
        assert rlk.det_gemm_tile_plan(LIN, 4096, 4096, 4096, sms)["tile_cols"] == 224
    g = torch.Generator(device=dev).manual_seed(22)

    def ints(r, c):
        return torch.randint(-4, 5, (r, c), generator=g, device=dev).to(torch.bfloat16)

    dC, B = ints(4096, 4096), ints(4096, 4096)     # dA = dC . B^T -> [4096, 4096]
    X, W = ints(4096, 4096), ints(4096, 4096)      # Y = X . W^T
    cases = {
        "da": (rlk.det_gemm_da(dC, B, out_dtype), dC.double() @ B.double().T,
               lambda r: rlk.det_gemm_da(dC[r], B, out_dtype)),
        "linear": (rlk.det_linear(X, W, out_dtype), X.double() @ W.double().T,
                   lambda r: rlk.det_linear(X[r], W, out_dtype)),
    }
    for name, (full, exact, part) in cases.items():
        assert torch.equal(full.double(), exact.float().to(out_dtype).double()), name
        split = torch.cat([part(slice(0, 2304)), part(slice(2304, 4096))])
        assert bits_equal(split, full), name
        small = torch.cat([part(slice(s, s + 256)) for s in range(0, 4096, 256)])
        assert bits_equal(small, full), name
    assert rlk.device_error() == 0


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_last_wave_split_gives_the_same_bits(dev, out_dtype):
    """An output of 16 x 16 wide tiles on 76 SM pairs leaves a last wave of 28
    tiles; with a long reduction (16384 here) those blocks are computed as two
    128-wide halves each in a second launch.  For all three products (outputs
    4096 x 3900, 4096 x 4000 and 4000 x 3900: a last column block of 60 columns,
    whose second half is empty, and one of 160), integer inputs give the exact
    product, and the rows equal the same rows of 1024-row calls (64 wide tiles,
    one launch) and of 256-row calls (narrow tiles throughout), bit for bit."""
    g = torch.Generator(device=dev).manual_seed(21)

    def ints(r, c):
        return torch.randint(-4, 5, (r, c), generator=g, device=dev).to(torch.bfloat16)

    R = 16384
    A, B = ints(4096, R), ints(R, 3900)                 # fwd: [4096, 3900]
    dC, Bt = ints(4096, R), ints(4000, R)               # dA: dC [4096, R] . B^T, B [4000, R]
    A2, dC2 = ints(R, 4000), ints(R, 3900)              # dB: A2^T . dC2 -> [4000, 3900]
    cases = {
        "fwd": (rlk.det_gemm_fwd(A, B, out_dtype), A.double() @ B.double(),
                lambda s, c: rlk.det_gemm_fwd(A[s:s + c], B, out_dtype), 4096),
        "da": (rlk.det_gemm_da(dC, Bt, out_dtype), dC.double() @ Bt.double().T,
               lambda s, c: rlk.det_gemm_da(dC[s:s + c], Bt, out_dtype), 4096),
        "db": (rlk.det_gemm_db(A2, dC2, out_dtype), A2.double().T @ dC2.double(),
               lambda s, c: rlk.det_gemm_db(A2[:, s:s + c], dC2, out_dtype), 4000),
    }
    for name, (full, exact, part, rows) in cases.items():
        # |sums| <= 16 * 16384 < 2^24: exact in FP32; the BF16 output is its RNE
        assert torch.equal(full.double(), exact.float().to(out_dtype).double()), name
        for chunk in (1024, 256):
            parts = torch.cat([part(s, chunk) for s in range(0, rows, chunk)])
            assert bits_equal(parts, full), (name, chunk)
    if out_dtype == torch.float32:
        # C += A . B through both launches: every block is added exactly once
        C0 = torch.randint(-8, 9, (4096, 3900), generator=g, device=dev).float()
        C = C0.clone()
        rlk.det_gemm_fwd_accum_fp32_(C, A, B)
        assert torch.equal(C, C0 + cases["fwd"][0])
    assert rlk.device_error() == 0


def test_two_product_backward_matches_the_oracle(dev, orc):
    """dA and dB from one FP32 dC (one shared BF16 rounding) against the FP64 oracle
    on the BF16 rounding of dC: relative Frobenius <= 1e-5 on sampled rows."""
    M, K, N = 1000, 768, 640
    A, B, dC = si.det_gemm_inputs(M, K, N, seed=72, device=dev, dc_dtype=torch.float32)
    dA, dB = rlk.det_gemm_backward(dC, A, B, torch.float32)
    torch.cuda.synchronize()
    d16 = orc.f32_to_bf16_rne(dC.cpu().numpy())
    ra = sample_rows(M, 24, seed=73)
    rb = sample_rows(K, 24, seed=74)
    ref_a = orc.gemm_da(d16, si.bf16_bits(B), rows=ra)
    ref_b = orc.gemm_db(si.bf16_bits(A), d16, rows=rb)
    assert rel_fro(dA.cpu().numpy()[ra].astype(np.float64), ref_a) <= GEMM_FP32_REL_FRO
    assert rel_fro(dB.cpu().numpy()[rb].astype(np.float64), ref_b) <= GEMM_FP32_REL_FRO
    assert rlk.device_error() == 0
