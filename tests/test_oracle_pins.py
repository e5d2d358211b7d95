"""Pins for the FP64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an Oracle and raises AssertionError on a
mismatch.  They are run against the real oracle, and against oracles with a
planted mistake (``ORACLE_MUTANT``) to show that every planted mistake is
caught by at least one pin.

What pins what:
  * 50-digit brute force (fractions + decimal) on tiny inputs  -> logits, lse, logp
  * torch float64 log_softmax / matmul (independent library code) -> linear_logp, GEMMs
  * hand-derived closed forms in tests/golden/closed_forms.json
  * invariants of the log-softmax definition ("feat(linear-logp): add
    batch-invariant fused SM90 operator", Walkthrough): logp <= 0,
    lse >= max z, sum_v exp(logp_v) = 1, equal rows -> -log V, V = 1 -> 0,
    bias shift -> lse shift, vocabulary permutation invariance
  * exact integer GEMMs vs numpy int64 ("feat(musa): add native deterministic
    gemm kernel", Summary: C = A B, dA = dC B^T, dB = A^T dC)
  * BF16 round-to-nearest-even vs exact rational rounding and torch's cast
"""
import json
import math
import os
import random
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _bits(x) -> np.ndarray:
    return si.bf16_bits(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def _dec(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _closed(expr: str) -> float:
    ns = {k: getattr(math, k) for k in ("log", "exp", "e", "sqrt")}
    return float(eval(expr, {"__builtins__": {}}, ns))  # fixture expressions only


# ------------------------------------------------------------------ linear-logp
def pin_closed_forms_logp(orc):
    cases = json.load(open(GOLDEN))["linear_logp"]
    for c in cases:
        h = _bits(c["hidden"])
        w = _bits(c["weight"])
        b = None if c["bias"] is None else np.asarray(c["bias"], np.float32)
        t = np.asarray(c["targets"], np.int64)
        hh = np.repeat(h, len(t), axis=0)
        logp, lse, _ = orc.linear_logp(hh, w, t, b)
        for i in range(len(t)):
            assert abs(lse[i] - _closed(c["lse"])) < 1e-13, (c["name"], i, lse[i])
            assert abs(logp[i] - _closed(c["logp"][i])) < 1e-13, (c["name"], i, logp[i])


def _brute_force(hbits, wbits, b, t):
    """Exact rational logits, then 50-digit decimal log-sum-exp."""
    getcontext().prec = 50
    H = hbits.shape[1]
    hv = [[Fraction(float(x)) for x in row] for row in _dec(hbits)]
    wv = [[Fraction(float(x)) for x in row] for row in _dec(wbits)]
    out = []
    for r, row in enumerate(hv):
        z = []
        for v, wr in enumerate(wv):
            acc = sum((row[k] * wr[k] for k in range(H)), Fraction(0))
            if b is not None:
                acc += Fraction(float(b[v]))
            z.append(acc)
        zd = [Decimal(q.numerator) / Decimal(q.denominator) for q in z]
        M = max(zd)
        s = sum(((x - M).exp() for x in zd), Decimal(0))
        lse = M + s.ln()
        out.append((float(zd[t[r]] - lse), float(lse), float(zd[t[r]])))
    return out


def pin_brute_force(orc):
    rng = np.random.default_rng(1234)
    for (N, H, V, with_bias) in [(1, 1, 1, False), (2, 3, 5, True), (4, 8, 16, True), (3, 7, 9, False)]:
        h = _bits(rng.standard_normal((N, H)))
        w = _bits(rng.standard_normal((V, H)) * 0.5)
        b = (rng.standard_normal(V) * 0.3).astype(np.float32) if with_bias else None
        t = rng.integers(0, V, N).astype(np.int64)
        logp, lse, zt = orc.linear_logp(h, w, t, b)
        ref = _brute_force(h, w, b, t)
        for i, (lp, ls, z) in enumerate(ref):
            assert abs(logp[i] - lp) < 1e-12 and abs(lse[i] - ls) < 1e-12 and abs(zt[i] - z) < 1e-12, \
                (N, H, V, i, logp[i], lp, lse[i], ls)


def pin_torch_log_softmax(orc):
    """torch float64 matmul + log_softmax on the decoded inputs (library code)."""
    hidden, weight, bias, target = si.linear_logp_inputs(16, 64, 300, bias=True, seed=3)
    h, w = si.bf16_bits(hidden), si.bf16_bits(weight)
    logp, lse, zt = orc.linear_logp(h, w, target.numpy(), bias.numpy())
    z = hidden.double() @ weight.double().T + bias.double()
    ref_lsm = torch.log_softmax(z, dim=-1)
    ref_lse = torch.logsumexp(z, dim=-1)
    ref_logp = ref_lsm.gather(1, target[:, None])[:, 0]
    assert np.allclose(logp, ref_logp.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(zt, z.gather(1, target[:, None])[:, 0].numpy(), rtol=0, atol=1e-12)


def pin_invariants(orc):
    rng = np.random.default_rng(7)
    N, H, V = 6, 24, 40
    h = _bits(rng.standard_normal((N, H)))
    w = _bits(rng.standard_normal((V, H)) / math.sqrt(H))
    # bias on a 2^-10 grid so that b + 0.75 below is exact in fp32
    b = (np.round(rng.standard_normal(V) * 0.2 * 1024) / 1024).astype(np.float32)
    t = rng.integers(0, V, N).astype(np.int64)
    logp, lse, zt = orc.linear_logp(h, w, t, b)
    z = orc.logits(h, w, b)
    # logp <= 0 and lse >= max_v z_v
    assert np.all(logp <= 0.0)
    assert np.all(lse >= z.max(axis=1))
    # the logp over every target sums (after exp) to one
    for r in range(N):
        hr = np.repeat(h[r:r + 1], V, axis=0)          # row r replicated, one copy per target
        lp_all, _, _ = orc.linear_logp(hr, w, np.arange(V, dtype=np.int64), b)
        assert abs(math.fsum(np.exp(lp_all)) - 1.0) < 1e-12
    # adding c to every bias entry shifts lse by c and leaves logp unchanged
    c = np.float32(0.75)
    logp2, lse2, _ = orc.linear_logp(h, w, t, b + c)
    assert np.array_equal((b + c).astype(np.float64), b.astype(np.float64) + 0.75)
    assert np.allclose(lse2, lse + float(c), rtol=0, atol=1e-12)
    assert np.allclose(logp2, logp, rtol=0, atol=1e-12)
    # permuting the vocabulary (W rows, bias, target ids together) changes nothing
    perm = rng.permutation(V)
    inv = np.argsort(perm)
    logp3, lse3, _ = orc.linear_logp(h, w[perm], inv[t].astype(np.int64), b[perm])
    assert np.allclose(logp3, logp, rtol=0, atol=1e-12)
    assert np.allclose(lse3, lse, rtol=0, atol=1e-12)
    # V = 1: logp = 0, lse = the single logit
    logp4, lse4, zt4 = orc.linear_logp(h, w[:1], np.zeros(N, np.int64), b[:1])
    assert np.all(logp4 == 0.0) and np.allclose(lse4, z[:, 0], rtol=0, atol=1e-12)
    # all W rows equal and zero bias: logp = -log V exactly (up to one rounding)
    weq = np.repeat(w[:1], V, axis=0)
    logp5, _, _ = orc.linear_logp(h, weq, t, None)
    assert np.allclose(logp5, -math.log(V), rtol=0, atol=1e-12)
    # out-of-range target: NaN logp, lse unaffected
    tb = t.copy()
    tb[0], tb[1] = -1, V
    logp6, lse6, zt6 = orc.linear_logp(h, w, tb, b)
    assert math.isnan(logp6[0]) and math.isnan(logp6[1]) and math.isnan(zt6[0])
    assert np.array_equal(lse6, lse)


def pin_row_subset_and_stride(orc):
    hidden, weight, bias, target = si.linear_logp_inputs(20, 32, 50, bias=True, seed=5)
    h, w = si.bf16_bits(hidden), si.bf16_bits(weight)
    full = orc.linear_logp(h, w, target.numpy(), bias.numpy())
    rows = np.array([19, 0, 7, 7, 13], np.int64)
    sub = orc.linear_logp(h, w, target.numpy(), bias.numpy(), rows=rows)
    for a, b in zip(full, sub):
        assert np.array_equal(a[rows], b)
    # target stride 0: one shared id for every row
    t0 = np.array([11], np.int64)
    lp0, _, _ = orc.linear_logp(h, w, t0, bias.numpy(), target_stride=0)
    lp1, _, _ = orc.linear_logp(h, w, np.full(20, 11, np.int64), bias.numpy())
    assert np.array_equal(lp0, lp1)


# ------------------------------------------------------------------ GEMM family
def pin_closed_forms_gemm(orc):
    for c in json.load(open(GOLDEN))["gemm"]:
        A, B, dC = _bits(c["A"]), _bits(c["B"]), _bits(c["dC"])
        assert np.array_equal(orc.gemm_fwd(A, B), np.asarray(c["C"], np.float64))
        assert np.array_equal(orc.gemm_da(dC, B), np.asarray(c["dA"], np.float64))
        assert np.array_equal(orc.gemm_db(A, dC), np.asarray(c["dB"], np.float64))


def _int_case(M, K, N, seed):
    A = si.integer_bf16((M, K), -16, 16, seed=seed)
    B = si.integer_bf16((K, N), -16, 16, seed=seed + 1)
    dC = si.integer_bf16((M, N), -16, 16, seed=seed + 2)
    return A, B, dC


def pin_integer_gemm_exact(orc):
    for (M, K, N) in [(1, 1, 1), (7, 5, 3), (33, 33, 33), (64, 40, 24), (24, 24, 24)]:
        A, B, dC = _int_case(M, K, N, seed=M + K + N)
        a = A.float().numpy().astype(np.int64)
        b = B.float().numpy().astype(np.int64)
        d = dC.float().numpy().astype(np.int64)
        Ab, Bb, dCb = si.bf16_bits(A), si.bf16_bits(B), si.bf16_bits(dC)
        assert np.array_equal(orc.gemm_fwd(Ab, Bb), (a @ b).astype(np.float64))
        assert np.array_equal(orc.gemm_da(dCb, Bb), (d @ b.T).astype(np.float64))
        assert np.array_equal(orc.gemm_db(Ab, dCb), (a.T @ d).astype(np.float64))


def pin_gemm_special_cases(orc):
    A, B, dC = si.det_gemm_inputs(12, 12, 12, seed=9)
    Ab = si.bf16_bits(A)
    eye = si.bf16_bits(torch.eye(12, dtype=torch.bfloat16))
    assert np.array_equal(orc.gemm_fwd(Ab, eye), _dec(Ab))              # A . I = A
    assert np.array_equal(orc.gemm_da(Ab, eye), _dec(Ab))               # dC . I^T = dC
    assert np.array_equal(orc.gemm_db(eye, Ab), _dec(Ab))               # I^T . dC = dC
    # K = 1: exact outer product
    A1, B1, _ = si.det_gemm_inputs(9, 1, 11, seed=10)
    a1, b1 = si.bf16_bits(A1), si.bf16_bits(B1)
    assert np.array_equal(orc.gemm_fwd(a1, b1), np.outer(_dec(a1)[:, 0], _dec(b1)[0]))


def pin_gemm_torch_f64(orc):
    A, B, dC = si.det_gemm_inputs(40, 72, 56, seed=11)
    Ab, Bb, dCb = si.bf16_bits(A), si.bf16_bits(B), si.bf16_bits(dC)
    assert np.allclose(orc.gemm_fwd(Ab, Bb), (A.double() @ B.double()).numpy(), rtol=1e-13, atol=1e-14)
    assert np.allclose(orc.gemm_da(dCb, Bb), (dC.double() @ B.double().T).numpy(), rtol=1e-13, atol=1e-14)
    assert np.allclose(orc.gemm_db(Ab, dCb), (A.double().T @ dC.double()).numpy(), rtol=1e-13, atol=1e-14)


def pin_gemm_cross_entry(orc):
    """da(dC, B) = fwd(dC, B^T) and db(A, dC) = fwd(A^T, dC), transposes materialised."""
    for (M, K, N) in [(9, 9, 9), (16, 5, 12), (7, 13, 3)]:
        A, B, dC = si.det_gemm_inputs(M, K, N, seed=M * K)
        Ab, Bb, dCb = si.bf16_bits(A), si.bf16_bits(B), si.bf16_bits(dC)
        BT = si.bf16_bits(B.T.contiguous())
        AT = si.bf16_bits(A.T.contiguous())
        assert np.array_equal(orc.gemm_da(dCb, Bb), orc.gemm_fwd(dCb, BT))
        assert np.array_equal(orc.gemm_db(Ab, dCb), orc.gemm_fwd(AT, dCb))
        rows = np.array([M - 1, 0], np.int64)
        assert np.array_equal(orc.gemm_fwd(Ab, Bb, rows=rows), orc.gemm_fwd(Ab, Bb)[rows])
        rk = np.array([K - 1, 0], np.int64)
        assert np.array_equal(orc.gemm_db(Ab, dCb, rows=rk), orc.gemm_db(Ab, dCb)[rk])


# ------------------------------------------------------------------ BF16 rounding
def _exact_rne_bf16(x: float) -> float:
    """Round a finite double to the nearest BF16 value, ties to even, by rationals."""
    q = Fraction(x)
    if q == 0:
        return 0.0
    a = abs(q)
    e = math.floor(math.log2(a)) if a > 0 else 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    qe = max(e - 7, -133)
    scaled = a / (Fraction(2) ** qe)
    n = math.floor(scaled)
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    y = Fraction(n) * Fraction(2) ** qe
    if y >= Fraction(2) ** 128:
        return math.copysign(math.inf, x)
    return math.copysign(float(y), x)


def pin_bf16_rounding(orc):
    fx = json.load(open(GOLDEN))["bf16_rne_from_f32"]
    for c in fx:
        x = np.float32(_closed(c["x"].replace("**", "**")))
        assert int(orc.f32_to_bf16_rne(np.array([x]))[0]) == int(c["bits"], 16), c
    # f32 -> bf16 against torch's cast on random and special values
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10) ** rng.integers(-30, 30, 20000).astype(np.float32),
        (np.arange(1 << 16, dtype=np.uint32) << 16 | 0x8000).view(np.float32),  # every tie pattern
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38, 1e-45], np.float32),
    ])
    vals = vals[~np.isnan(vals)]
    ours = orc.f32_to_bf16_rne(vals)
    ref = si.bf16_bits(torch.from_numpy(vals).to(torch.bfloat16))
    assert np.array_equal(ours, ref)
    # f64 -> bf16 (single rounding) against exact rational rounding
    pyr = random.Random(5)
    xs = [pyr.uniform(-1, 1) * 2.0 ** pyr.randint(-140, 130) for _ in range(3000)]
    xs += [1 + 2 ** -8, 1 + 2 ** -8 + 2 ** -40, 1 + 3 * 2 ** -8, 2 ** -134, 3 * 2 ** -135, -(1 + 2 ** -8 - 2 ** -45)]
    got = orc.f64_to_bf16_rne(np.array(xs))
    for x, g in zip(xs, got):
        want = _exact_rne_bf16(x)
        gv = float(_dec(np.array([g]))[0])
        assert gv == want or (math.isinf(want) and math.isinf(gv)), (x, gv, want)
    # a double just above a BF16 tie must round up (a detour through binary32 would tie to even)
    x = 1 + 2 ** -8 + 2 ** -40
    assert float(_dec(orc.f64_to_bf16_rne(np.array([x])))[0]) == 1 + 2 ** -7


# ------------------------------------------------------------------ backward
def _bwd_case(seed, N=7, H=12, V=30, bias=True):
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=bias, seed=seed)
    g = torch.randn(N, generator=torch.Generator().manual_seed(seed + 100), dtype=torch.float64)
    return hidden, weight, b, target, g


def pin_backward_torch_autograd(orc):
    """torch float64 autograd of sum_r g_r * log_softmax(h W^T + b)[r, t_r] (library code)."""
    hidden, weight, b, target, g = _bwd_case(21)
    target[3] = 0
    dh, dw, db, _ = orc.linear_logp_backward(si.bf16_bits(hidden), si.bf16_bits(weight),
                                             target.numpy(), g.numpy(), b.numpy())
    h = hidden.double().requires_grad_()
    w = weight.double().requires_grad_()
    bb = b.double().requires_grad_()
    lp = torch.log_softmax(h @ w.T + bb, dim=-1).gather(1, target[:, None])[:, 0]
    (g * lp).sum().backward()
    assert np.allclose(dh, h.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(dw, w.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(db, bb.grad.numpy(), rtol=0, atol=1e-12)


def pin_backward_finite_difference(orc):
    """dL/dbias_v against central differences of the (pinned) forward oracle."""
    hidden, weight, b, target, g = _bwd_case(22, N=5, H=8, V=12)
    hb, wb, t = si.bf16_bits(hidden), si.bf16_bits(weight), target.numpy()
    _, _, db, _ = orc.linear_logp_backward(hb, wb, t, g.numpy(), b.numpy())
    eps = 2.0 ** -10                       # exact in fp32 around |b| < 1
    for v in range(12):
        bp, bm = b.numpy().copy(), b.numpy().copy()
        bp[v] += eps
        bm[v] -= eps
        lp_p, _, _ = orc.linear_logp(hb, wb, t, bp)
        lp_m, _, _ = orc.linear_logp(hb, wb, t, bm)
        fd = (g.numpy() @ lp_p - g.numpy() @ lp_m) / (float(bp[v]) - float(bm[v]))
        assert abs(fd - db[v]) <= 1e-6 * max(1.0, abs(db[v])), (v, fd, db[v])


def pin_backward_invariants(orc):
    hidden, weight, b, target, g = _bwd_case(23)
    target[2] = -1                          # out of range: zero gradient row
    G = orc.grad_logits(si.bf16_bits(hidden), si.bf16_bits(weight), target.numpy(), g.numpy(),
                        b.numpy())
    live = np.ones(len(target), bool)
    live[2] = False
    assert np.all(G[2] == 0.0)
    # sum_v (onehot - softmax) = 0 for every live row
    assert np.allclose(G[live].sum(axis=1), 0.0, rtol=0, atol=1e-14)
    # the target column carries g * (1 - p) with sign(g); all other entries carry -g * p
    for r in np.flatnonzero(live):
        others = np.delete(G[r], int(target[r]))
        assert np.all(np.sign(others) != np.sign(g[r].item())) or g[r] == 0
        assert np.sign(G[r, int(target[r])]) == np.sign(g[r].item())


PINS = [pin_backward_torch_autograd, pin_backward_finite_difference, pin_backward_invariants,
        pin_closed_forms_logp, pin_brute_force, pin_torch_log_softmax, pin_invariants,
        pin_row_subset_and_stride, pin_closed_forms_gemm, pin_integer_gemm_exact,
        pin_gemm_special_cases, pin_gemm_torch_f64, pin_gemm_cross_entry, pin_bf16_rounding]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("mutant", range(1, 11))
def test_planted_mistake_is_caught(mutant):
    """Every planted oracle mistake fails at least one pin."""
    import oracle
    bad = oracle.load_mutant(mutant)
    caught = []
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
