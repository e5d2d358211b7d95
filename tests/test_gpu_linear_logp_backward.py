"""GPU parity, determinism and batch invariance of the linear-logp backward.

G = dL/dz = g * (onehot(t) - exp(z - lse)) is formed in FP32 and rounded to
BF16; grad_hidden = G.W, grad_weight = G^T.hidden, grad_bias = sum_r G.
Checks:
  * G within one BF16 ulp of the oracle's exact G (plus the FP32 error of p);
  * each product exactly as the deterministic GEMM of the GPU's own G
    (tolerance-free), and within 1e-5 relative Frobenius of the FP64 product of
    that same G (pure GEMM accuracy);
  * end to end within 1e-2 relative Frobenius of the oracle's exact gradients
    (BF16 rounding of G dominates);
  * grad_hidden rows bitwise independent of the other rows; everything
    bitwise run to run.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import bf16_ulp, cuda_or_skip, dec_bf16, rel_fro, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _case(N, H, V, bias, seed, dev):
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=bias, seed=seed)
    g = torch.randn(N, generator=torch.Generator().manual_seed(seed + 7))
    return hidden.to(dev), weight.to(dev), None if b is None else b.to(dev), target.to(dev), g.to(dev)


def _backward(hidden, weight, target, g, b, out_dtype=torch.float32):
    _, lse = rlk.linear_logp(hidden, weight, target, b)
    return rlk.linear_logp_backward(hidden, weight, target, lse, g, b, out_dtype=out_dtype,
                                    return_grad_logits=True)


@pytest.mark.parametrize("N,H,V,bias", [(300, 512, 5000, True), (130, 1024, 3001, False),
                                        (5, 64, 257, True)])
def test_backward_parity(dev, orc, N, H, V, bias):
    hidden, weight, b, target, g = _case(N, H, V, bias, seed=N + V, dev=dev)
    target[1] = -3                                    # out of range: zero gradient row
    dh, dw, db, G = _backward(hidden, weight, target, g, b)
    torch.cuda.synchronize()
    hb, wb = si.bf16_bits(hidden), si.bf16_bits(weight)
    ref_dh, ref_dw, ref_db, ref_G = orc.linear_logp_backward(
        hb, wb, target.cpu().numpy(), g.cpu().double().numpy(),
        None if b is None else b.cpu().numpy())
    # G: one BF16 ulp of the exact value, plus the FP32 error of exp(z - lse)
    Gg = dec_bf16(si.bf16_bits(G))
    slack = 1e-5 * np.abs(g.cpu().double().numpy())[:, None]
    assert np.all(np.abs(Gg - ref_G) <= bf16_ulp(ref_G) + slack)
    assert np.all(Gg[1] == 0.0)
    # the products are the deterministic GEMMs of the GPU's own BF16 G (bitwise) ...
    Gc = G.contiguous()
    assert torch.equal(dh, rlk.det_gemm_fwd(Gc, weight, out_dtype=torch.float32))
    assert torch.equal(dw, rlk.det_gemm_db(Gc, hidden, out_dtype=torch.float32))
    # ... accurate as GEMMs on that G ...
    hd, wd = dec_bf16(hb), dec_bf16(wb)
    assert rel_fro(dh.cpu().double().numpy(), Gg @ wd) <= 1e-5
    assert rel_fro(dw.cpu().double().numpy(), Gg.T @ hd) <= 1e-5
    if b is not None:
        assert rel_fro(db.cpu().double().numpy(), Gg.sum(axis=0)) <= 1e-5
    # ... and end to end close to the exact gradient (BF16 G dominates the error)
    assert rel_fro(dh.cpu().double().numpy(), ref_dh) <= 1e-2
    assert rel_fro(dw.cpu().double().numpy(), ref_dw) <= 1e-2
    if b is not None:
        assert rel_fro(db.cpu().double().numpy(), ref_db) <= 1e-2
    assert np.all(dh.cpu().numpy()[1] == 0.0)
    assert rlk.device_error() == 0


def test_backward_bf16_outputs_round_fp32(dev):
    hidden, weight, b, target, g = _case(200, 768, 4000, True, seed=3, dev=dev)
    dh32, dw32, db32, _ = _backward(hidden, weight, target, g, b, torch.float32)
    dh16, dw16, db16, _ = _backward(hidden, weight, target, g, b, torch.bfloat16)
    assert torch.equal(dh16, dh32.to(torch.bfloat16))
    assert torch.equal(dw16, dw32.to(torch.bfloat16))
    assert torch.equal(db16, db32)                    # grad_bias is always FP32


def test_backward_rows_invariant_and_deterministic(dev):
    N, H, V = 700, 1024, 9000
    hidden, weight, b, target, g = _case(N, H, V, True, seed=4, dev=dev)
    dh, dw, db, G = _backward(hidden, weight, target, g, b)
    for _ in range(2):
        dh2, dw2, db2, G2 = _backward(hidden, weight, target, g, b)
        assert torch.equal(dh, dh2) and torch.equal(dw, dw2) and torch.equal(db, db2)
        assert torch.equal(G, G2)
    _, lse = rlk.linear_logp(hidden, weight, target, b)
    for chunk in (1, 129):
        parts = [rlk.linear_logp_backward(hidden[s:s + chunk], weight, target[s:s + chunk],
                                          lse[s:s + chunk], g[s:s + chunk], b, grad_weight=False,
                                          grad_bias=False, out_dtype=torch.float32)[0]
                 for s in range(0, N, chunk)]
        assert torch.equal(torch.cat(parts), dh), f"chunk {chunk}"


def test_backward_mid_shape_runs_deterministically(dev):
    w = si.MID
    hidden, weight, b, target = si.workload_inputs(w, seed=5, device=dev)
    hidden, target = hidden[:1024], target[:1024]
    g = torch.randn(1024, device=dev)
    dh, dw, db, _ = _backward(hidden, weight, target, g, b, torch.bfloat16)
    dh2, dw2, _, _ = _backward(hidden, weight, target, g, b, torch.bfloat16)
    assert torch.equal(dh, dh2) and torch.equal(dw, dw2)
    assert bool(torch.isfinite(dh.float()).all()) and bool(torch.isfinite(dw.float()).all())
    assert rlk.device_error() == 0


def test_backward_mid_rows_equal_across_tilings(dev):
    """At the mid vocabulary grad_hidden = G . W reduces over V = 151936.  A 4096-row
    call has 16 x 16 output tiles, whose last wave runs as half tiles in a second
    launch; 1024- and 600-row calls run wide tiles in one launch, 256-row calls
    narrow tiles throughout.  The rows of all of them are the same bits."""
    w = si.MID
    hidden, weight, _, target = si.workload_inputs(w, seed=6, device=dev)
    g = torch.randn(w.N, device=dev, generator=torch.Generator(device=dev).manual_seed(13))
    _, lse = rlk.linear_logp(hidden, weight, target)

    def dh(rows):
        return rlk.linear_logp_backward(hidden[rows], weight, target[rows], lse[rows], g[rows],
                                        grad_weight=False, grad_bias=False,
                                        out_dtype=torch.float32)[0]

    full = dh(slice(0, w.N))
    for chunk in (1024, 600, 256):
        parts = torch.cat([dh(slice(s, min(s + chunk, w.N))) for s in range(0, w.N, chunk)])
        assert torch.equal(parts.view(torch.int32), full.view(torch.int32)), chunk
    assert rlk.device_error() == 0


def test_backward_zero_rows(dev):
    weight = torch.randn(50, 64, device=dev).to(torch.bfloat16)
    e = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    dh, dw, db = rlk.linear_logp_backward(e, weight, torch.empty(0, dtype=torch.int64, device=dev),
                                          torch.empty(0, device=dev), torch.empty(0, device=dev),
                                          torch.zeros(50, device=dev), out_dtype=torch.float32)
    assert dh.numel() == 0 and bool((dw == 0).all()) and bool((db == 0).all())


def test_backward_bias_alignment_paths(dev):
    """An aligned bias is read four floats at a time, any other one float at a time:
    G and all three gradients agree bit for bit."""
    N, H, V = 300, 512, 5003
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=True, seed=41, device=dev)
    g = torch.randn(N, generator=torch.Generator(device=dev).manual_seed(42), device=dev)
    _, lse = rlk.linear_logp(hidden, weight, target, b)
    store = torch.empty(V + 4, dtype=torch.float32, device=dev)
    store[1:V + 1] = b
    shifted = store[1:V + 1]
    assert b.data_ptr() % 16 == 0 and shifted.data_ptr() % 16 == 4
    ref = rlk.linear_logp_backward(hidden, weight, target, lse, g, b, return_grad_logits=True)
    got = rlk.linear_logp_backward(hidden, weight, target, lse, g, shifted, return_grad_logits=True)
    for x, y in zip(ref, got):
        assert torch.equal(x, y)


def test_backward_mid_parity_sampled(dev, orc):
    """The bench's backward step at the full mid shape (N=4096, H=4096, V=151936):
    sampled rows of G and grad_hidden and sampled rows of grad_weight against the
    FP64 oracle and against float64 products of the GPU's own G.  grad_hidden
    reduces over K = V = 151,936 terms, one large (the target's) and the rest
    tiny, so its FP32 accumulation error exceeds the 1e-5 used for the K = 4096
    GEMMs: it is held to the FP32 summation bound |gpu - exact| <= K 2^-23
    sum |G W| elementwise, and to 1e-3 relative Frobenius."""
    w = si.MID
    hidden, weight, b, target = si.workload_inputs(w, seed=6, device=dev)
    g = torch.randn(w.N, generator=torch.Generator(device=dev).manual_seed(7), device=dev)
    dh, dw, _, G = _backward(hidden, weight, target, g, b, torch.float32)
    torch.cuda.synchronize()
    rows = sample_rows(w.N, 10, seed=8, must=(255, 256, 4095))
    hb_rows, wb = si.bf16_bits(hidden[rows]), si.bf16_bits(weight)
    ref_G = orc.grad_logits(hb_rows, wb, target[rows].cpu().numpy(), g[rows].cpu().double().numpy())
    Gg = dec_bf16(si.bf16_bits(G[rows]))
    slack = 1e-5 * np.abs(g[rows].cpu().double().numpy())[:, None]
    assert np.all(np.abs(Gg - ref_G) <= bf16_ulp(ref_G) + slack)
    wd = dec_bf16(wb)
    got = dh[rows].cpu().double().numpy()
    exact = Gg @ wd
    assert np.all(np.abs(got - exact) <= w.V * 2.0 ** -23 * (np.abs(Gg) @ np.abs(wd)))
    assert rel_fro(got, exact) <= 1e-3
    assert rel_fro(got, ref_G @ wd) <= 1e-2
    # grad_weight rows (vocabulary ids) need G's whole column: use the GPU's own G
    vs = np.array([0, 1, 255, 256, 75967, 151935], dtype=np.int64)
    Gcols = dec_bf16(si.bf16_bits(G[:, vs].contiguous()))            # [N, len(vs)]
    hd = dec_bf16(si.bf16_bits(hidden))
    assert rel_fro(dw[vs].cpu().double().numpy(), Gcols.T @ hd) <= 1e-5
    assert rlk.device_error() == 0


def test_backward_full_vocabulary_grad_weight_vs_oracle(dev, orc):
    """grad_weight at the full mid vocabulary (V = 151,936, H = 4096) tied back to
    the FP64 oracle end to end: N = 256 rows, the oracle's G by definition on
    every row, and sampled vocabulary rows of grad_weight = G^T . hidden (the
    tile edges 0 / 255 / 256, the last id, and ids that some row targets) against
    the exact product, within the end-to-end 1e-2 relative Frobenius bound (the
    BF16 rounding of G dominates); the same rows within 1e-5 of the float64
    product of the GPU's own G."""
    w = si.MID
    N = 256
    hidden, weight, b, target = si.workload_inputs(w, seed=9, device=dev)
    hidden, target = hidden[:N].contiguous(), target[:N].contiguous()
    g = torch.randn(N, generator=torch.Generator(device=dev).manual_seed(10), device=dev)
    dh, dw, _, G = _backward(hidden, weight, target, g, b, torch.float32)
    torch.cuda.synchronize()
    hb, wb = si.bf16_bits(hidden), si.bf16_bits(weight)
    tgt = target.cpu().numpy()
    ref_G = orc.grad_logits(hb, wb, tgt, g.cpu().double().numpy())          # [N, V]
    vs = np.array(sorted({0, 1, 255, 256, 75968, w.V - 1, int(tgt[0]), int(tgt[1]),
                          int(tgt[N - 1])}), dtype=np.int64)
    hd = dec_bf16(hb)
    got = dw[vs].cpu().double().numpy()
    assert rel_fro(got, ref_G[:, vs].T @ hd) <= 1e-2
    for i, v in enumerate(vs):                        # row by row as well
        assert rel_fro(got[i], ref_G[:, v] @ hd) <= 1e-2, f"vocabulary row {v}"
    Gcols = dec_bf16(si.bf16_bits(G[:, vs].contiguous()))
    assert rel_fro(got, Gcols.T @ hd) <= 1e-5
    # G itself on every row: one BF16 ulp of the exact value (+ the FP32 error of exp)
    Gg = dec_bf16(si.bf16_bits(G))
    slack = 1e-5 * np.abs(g.cpu().double().numpy())[:, None]
    assert np.all(np.abs(Gg - ref_G) <= bf16_ulp(ref_G) + slack)
    assert rlk.device_error() == 0


def test_backward_layouts_staged_operands(dev):
    """A wider-pitch view, an odd-pitch (staged) hidden and an odd-pitch (staged)
    weight give the same G and gradients bit for bit as contiguous operands."""
    N, H, V = 300, 1000, 5003
    hidden, weight, b, target, g = _case(N, H, V, True, seed=43, dev=dev)
    _, lse = rlk.linear_logp(hidden, weight, target, b)

    def bwd(h, w):
        return rlk.linear_logp_backward(h, w, target, lse, g, b, out_dtype=torch.float32,
                                        return_grad_logits=True)

    ref = bwd(hidden, weight)
    for name, pad_h, pad_w in (("wide pitch", 64, 0), ("odd hidden pitch", 1, 0),
                               ("odd weight pitch", 0, 3), ("both odd", 5, 7)):
        h = torch.zeros(N, H + pad_h, dtype=torch.bfloat16, device=dev)
        h[:, :H] = hidden
        w = torch.zeros(V, H + pad_w, dtype=torch.bfloat16, device=dev)
        w[:, :H] = weight
        got = bwd(h[:, :H], w[:, :H])
        for x, y, what in zip(ref, got, ("grad_hidden", "grad_weight", "grad_bias", "G")):
            assert torch.equal(x, y), f"{name}: {what} bits differ"
    # a hidden whose base is 2 bytes past a 16-byte boundary is staged as well
    store = torch.zeros(N * H + 8, dtype=torch.bfloat16, device=dev)
    shifted = store[1:1 + N * H].view(N, H)
    shifted.copy_(hidden)
    assert shifted.data_ptr() % 16 == 2
    got = bwd(shifted, weight)
    for x, y in zip(ref, got):
        assert torch.equal(x, y)
    assert rlk.device_error() == 0


def test_backward_fails_closed_on_a_misaligned_output(dev):
    """An FP32 grad_weight that is not 4-byte aligned is refused before anything
    launches: grad_hidden and the workspace keep every byte."""
    import ctypes
    N, H, V = 64, 256, 1000
    hidden, weight, b, target, g = _case(N, H, V, False, seed=44, dev=dev)
    _, lse = rlk.linear_logp(hidden, weight, target, b)
    lib = rlk.lib()
    n = lib.rlk_linear_logp_backward_workspace_size_for(rlk._ptr(hidden), N, H, H, rlk._ptr(weight),
                                                        V, H)
    ws = torch.full((n,), 0x5A, dtype=torch.uint8, device=dev)
    gh = torch.full((N, H), -7.0, device=dev)
    gw_store = torch.zeros(V * H + 4, dtype=torch.float32, device=dev)
    bad_gw = ctypes.c_void_p(gw_store.data_ptr() + 2)
    torch.cuda.synchronize()
    st = lib.rlk_linear_logp_backward(
        rlk._ptr(hidden), N, H, H, rlk._ptr(weight), V, H, None, rlk._ptr(target), 1,
        rlk._ptr(lse), rlk._ptr(g), rlk._ptr(gh), rlk.RLK_FP32, H, bad_gw, rlk.RLK_FP32, H, None,
        rlk._ptr(ws), n, rlk._stream_ptr(None))
    assert st == 4                                                     # RLK_ERR_ALIGN
    torch.cuda.synchronize()
    assert bool((gh == -7.0).all()) and bool((ws == 0x5A).all()) and bool((gw_store == 0).all())
    # a grad_hidden pitch below H is refused the same way
    st = lib.rlk_linear_logp_backward(
        rlk._ptr(hidden), N, H, H, rlk._ptr(weight), V, H, None, rlk._ptr(target), 1,
        rlk._ptr(lse), rlk._ptr(g), rlk._ptr(gh), rlk.RLK_FP32, H - 1, None, rlk.RLK_FP32, H, None,
        rlk._ptr(ws), n, rlk._stream_ptr(None))
    assert st == 2                                                     # RLK_ERR_SHAPE
    torch.cuda.synchronize()
    assert bool((gh == -7.0).all()) and bool((ws == 0x5A).all())
    assert rlk.device_error() == 0


@pytest.mark.parametrize("want", ["all", "hidden", "weight"])
def test_trainable_autograd_matches_the_backward_entry(dev, want):
    """linear_logp_trainable under autograd: forward bitwise equal to linear_logp,
    gradients bitwise equal to linear_logp_backward with the same grad_logp, and
    only the requested gradients are formed; lse carries no gradient."""
    hidden, weight, b, target, g = _case(200, 512, 3001, True, seed=11, dev=dev)
    h = hidden.clone().requires_grad_(want in ("all", "hidden"))
    w = weight.clone().requires_grad_(want in ("all", "weight"))
    bb = b.clone().requires_grad_(want == "all")
    logp, lse = rlk.linear_logp_trainable(h, w, target, bb)
    assert not lse.requires_grad and logp.requires_grad
    ref_logp, ref_lse = rlk.linear_logp(hidden, weight, target, b)
    assert torch.equal(logp.detach(), ref_logp) and torch.equal(lse, ref_lse)
    (logp * g).sum().backward()
    dh, dw, db = rlk.linear_logp_backward(hidden, weight, target, ref_lse, g, b)
    torch.cuda.synchronize()
    if want in ("all", "hidden"):
        assert h.grad.dtype == torch.bfloat16 and torch.equal(h.grad, dh)
    else:
        assert h.grad is None
    if want in ("all", "weight"):
        assert w.grad.dtype == torch.bfloat16 and torch.equal(w.grad, dw)
    else:
        assert w.grad is None
    if want == "all":
        assert bb.grad.dtype == torch.float32 and torch.equal(bb.grad, db)
    else:
        assert bb.grad is None
    with pytest.raises(RuntimeError):                 # the forward-only entry fails closed
        if h.requires_grad:
            rlk.linear_logp(h, weight, target)
        else:
            rlk.linear_logp(hidden, w, target)
