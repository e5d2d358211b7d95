"""Bitwise determinism and batch invariance of the fused linear-logp.

The page "feat(linear-logp): add batch-invariant fused SM90 operator" fixes the
contract: the same row with the same V gives the same bits whatever the batch
(author notes: full-batch bits == concatenation of the chunks' bits, checked
with exact equality, never allclose; PR body: batch size, row position,
neighbouring rows, chunking, layouts, vocabulary boundaries and CUDA streams).
Every check here compares bit patterns (signed zeros and NaN payloads included).
"""
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import bits_equal, cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


@pytest.fixture(scope="module")
def mid(dev):
    return si.workload_inputs(si.MID, seed=11, device=dev)


def lp(hidden, weight, target, bias=None, stream=None):
    return rlk.linear_logp(hidden, weight, target, bias, return_target_logit=True, stream=stream)


def chunked(hidden, weight, target, bias, chunk):
    outs = [lp(hidden[s:s + chunk], weight, target[s:s + chunk], bias)
            for s in range(0, hidden.size(0), chunk)]
    return tuple(torch.cat([o[i] for o in outs]) for i in range(3))


def assert_same(a, b, what):
    for x, y, name in zip(a, b, ("logp", "lse", "target_logit")):
        assert bits_equal(x, y), f"{what}: {name} bits differ"


def test_run_to_run_mid(mid):
    hidden, weight, bias, target = mid
    first = lp(hidden, weight, target, bias)
    for _ in range(9):
        assert_same(lp(hidden, weight, target, bias), first, "run-to-run")
    assert rlk.device_error() == 0


@pytest.mark.parametrize("chunk", [1, 7, 512])
def test_chunking_mid(mid, chunk):
    hidden, weight, bias, target = mid
    full = lp(hidden, weight, target, bias)
    assert_same(chunked(hidden, weight, target, bias, chunk), full, f"chunk {chunk}")


def test_chunking_large(dev):
    hidden, weight, bias, target = si.workload_inputs(si.LARGE, seed=12, device=dev)
    full = lp(hidden, weight, target, bias)
    for chunk in (7, 2048):
        assert_same(chunked(hidden, weight, target, bias, chunk), full, f"large chunk {chunk}")


def test_row_position_and_neighbours(dev):
    H, V, N = 1024, 40000, 300
    hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=13, device=dev)
    row, t = hidden[5].clone(), target[5].clone()
    ref = lp(row[None], weight, t[None], bias)
    g = torch.Generator(device=dev).manual_seed(99)
    for pos in (0, 127, 128, N - 1):
        h = torch.randn(N, H, generator=g, device=dev).to(torch.bfloat16)   # fresh neighbours
        tt = torch.randint(0, V, (N,), generator=g, device=dev)
        h[pos], tt[pos] = row, t
        out = lp(h, weight, tt, bias)
        assert_same(tuple(o[pos:pos + 1] for o in out), ref, f"position {pos}")


def test_vocab_boundary_targets(dev):
    """Targets on tile / split edges and the last id of a ragged vocabulary."""
    H, V = 512, 32003
    hidden, weight, bias, _ = si.linear_logp_inputs(16, H, V, bias=True, seed=14, device=dev)
    edges = torch.tensor([0, 255, 256, 511, 512, 31999, 32000, 32002, 1, 254, 257, 1023, 1024,
                          16383, 16384, 32001], device=dev)
    full = lp(hidden, weight, edges, bias)
    for i in range(16):
        one = lp(hidden[i:i + 1], weight, edges[i:i + 1], bias)
        assert_same(tuple(o[i:i + 1] for o in full), one, f"edge target {int(edges[i])}")


def test_streams(mid):
    hidden, weight, bias, target = mid
    ref = lp(hidden[:1000], weight, target[:1000], bias)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        a = lp(hidden[:1000], weight, target[:1000], bias, stream=s1)
    with torch.cuda.stream(s2):
        b = lp(hidden[:1000], weight, target[:1000], bias, stream=s2)
    torch.cuda.synchronize()
    assert_same(a, ref, "stream 1")
    assert_same(b, ref, "stream 2")


def test_layouts(dev):
    """Contiguous, wider-pitch view and odd-pitch (staged) hidden give the same bits."""
    N, H, V = 257, 2048, 32003
    hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, seed=15, device=dev)
    ref = lp(hidden, weight, target, bias)
    wide = torch.zeros(N, H + 64, dtype=torch.bfloat16, device=dev)
    wide[:, :H] = hidden
    assert_same(lp(wide[:, :H], weight, target, bias), ref, "wide pitch")
    odd = torch.zeros(N, H + 1, dtype=torch.bfloat16, device=dev)
    odd[:, :H] = hidden
    assert_same(lp(odd[:, :H], weight, target, bias), ref, "odd pitch (staged)")
    wodd = torch.zeros(V, H + 3, dtype=torch.bfloat16, device=dev)
    wodd[:, :H] = weight
    assert_same(lp(hidden, wodd[:, :H], target, bias), ref, "odd weight pitch (staged)")
    t_strided = torch.stack([target, target], dim=1)[:, 0]           # stride 2
    assert_same(lp(hidden, weight, t_strided, bias), ref, "strided target")


@pytest.mark.parametrize("n_small", [1, 17, 32, 100, 128, 129, 200, 255, 256])
def test_small_call_loops_match_the_pair_loop(dev, n_small):
    """Calls of at most 128 rows run on the one-CTA loop (M=128 per CTA; at most
    32 rows: a thin ring staging only those rows); larger calls on the 2-SM loop
    (M=256 over a pair, rows split between the pair's CTAs).  A row's bits are the
    same in all of them: the rows of a small call equal the same rows inside 33-,
    129-, 257- and 300-row calls (other row blocks and pair halves), for a ragged
    vocabulary with bias, and with a staged (odd-pitch) hidden or weight."""
    H, V = 2048, 32003
    hidden, weight, bias, target = si.linear_logp_inputs(300, H, V, bias=True, seed=16, device=dev)
    for start in (0, 5, 44):
        rows = slice(start, start + n_small)
        small = lp(hidden[rows], weight, target[rows], bias)
        for big_n in (33, 129, 257, 300):
            if big_n <= n_small:
                continue
            s0 = max(0, min(start, big_n - n_small))
            h_big, t_big = hidden[:big_n].clone(), target[:big_n].clone()
            h_big[s0:s0 + n_small], t_big[s0:s0 + n_small] = hidden[rows], target[rows]
            big = lp(h_big, weight, t_big, bias)
            assert_same(tuple(o[s0:s0 + n_small] for o in big), small,
                        f"{n_small} rows at {start} vs a {big_n}-row call")
    odd = torch.zeros(n_small, H + 1, dtype=torch.bfloat16, device=dev)
    odd[:, :H] = hidden[:n_small]
    ref = lp(hidden[:n_small], weight, target[:n_small], bias)
    assert_same(lp(odd[:, :H], weight, target[:n_small], bias), ref, "small call, staged hidden")
    wodd = torch.zeros(V, H + 3, dtype=torch.bfloat16, device=dev)
    wodd[:, :H] = weight
    assert_same(lp(hidden[:n_small], wodd[:, :H], target[:n_small], bias), ref,
                "small call, staged weight")
    assert rlk.device_error() == 0


@pytest.mark.parametrize("N", [17, 300])
def test_bias_alignment_paths(dev, N):
    """A 16-byte-aligned bias is read as two 4-float vectors per lane, any other one
    float at a time (and the 3-id tail tile of V = 32003 always so); both add the same
    FP32 values, so the bits agree (one-CTA and 2-SM loops)."""
    H, V = 1024, 32003
    hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=17, device=dev)
    assert bias.data_ptr() % 16 == 0
    store = torch.empty(V + 4, dtype=torch.float32, device=dev)
    store[1:V + 1] = bias
    shifted = store[1:V + 1]
    assert shifted.data_ptr() % 16 == 4
    assert_same(lp(hidden, weight, target, shifted), lp(hidden, weight, target, bias),
                "bias read one float at a time vs four at a time")


@pytest.mark.parametrize("H", [64, 320, 2112])
def test_zero_rows_keep_their_signed_zero_across_loops(dev, H):
    """A hidden row of zeros against an all-negative weight makes every product -0.
    Calls of more than 256 rows stage 128 reduction columns at a time, smaller ones
    64; with an odd number of 64-wide blocks the last 128-wide stage holds one
    block and zero fill, and only that block's MMAs run, so the logits (and the
    target logit read out as is) keep the same zero sign as in a 1-row call (one-CTA
    loop) or a 200-row call (2-SM loop, 64-wide stages)."""
    V = 1000
    hidden, weight, _, target = si.linear_logp_inputs(300, H, V, bias=False, seed=18, device=dev)
    weight = -(weight.abs() + 2.0 ** -8).to(torch.bfloat16)
    hidden = hidden.clone()
    zero_rows = (0, 7, 255, 256, 299)
    hidden[list(zero_rows)] = 0
    big = lp(hidden, weight, target)
    mid_call = lp(hidden[:200], weight, target[:200])
    for r in zero_rows:
        one = lp(hidden[r:r + 1], weight, target[r:r + 1])
        assert_same(tuple(o[r:r + 1] for o in big), one, f"zero row {r}: 300-row vs 1-row call")
        if r < 200:
            assert_same(tuple(o[r:r + 1] for o in mid_call), one, f"zero row {r}: 200-row call")
    assert_same(tuple(o[:200] for o in big), mid_call, "300-row vs 200-row call")
    assert rlk.device_error() == 0
