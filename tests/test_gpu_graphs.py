"""The operators run inside CUDA graphs.

Every call is stream-ordered, allocates nothing and never synchronises the
host, so a captured sequence (the counter zeroing of a long launch, the
programmatic-dependent launches, staging copies) replays with the same bits as
eager calls.
"""
import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


@pytest.mark.parametrize("N", [17, 300, 4096])
def test_linear_logp_graph_replay(dev, N):
    w = si.MID
    hidden, weight, bias, target = si.workload_inputs(w, seed=51, device=dev)
    hidden, target = hidden[:N].contiguous(), target[:N].contiguous()
    call = rlk.LinearLogpCall(hidden, weight, target, bias, target_logit=True)
    call()
    torch.cuda.synchronize()
    eager = (call.logp.clone(), call.lse.clone(), call.zt.clone())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):            # warm-up on the capture stream
        call(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        call.logp.zero_(), call.lse.zero_(), call.zt.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip((call.logp, call.lse, call.zt), eager):
            assert torch.equal(a, b)
    # new inputs copied into the captured buffers are picked up by the replay
    h2 = torch.randn(N, w.H, device=dev, generator=torch.Generator(device=dev).manual_seed(52))
    hidden.copy_(h2.to(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    ref = rlk.linear_logp(hidden, weight, target, bias)
    assert torch.equal(call.logp, ref[0]) and torch.equal(call.lse, ref[1])
    assert rlk.device_error() == 0


def test_backward_and_det_gemm_graph_replay(dev):
    N, H, V = 300, 512, 5003
    hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=53, device=dev)
    gl = torch.randn(N, device=dev, generator=torch.Generator(device=dev).manual_seed(54))
    A, B, dC = si.det_gemm_inputs(1000, 768, 640, seed=55, device=dev)
    _, lse = rlk.linear_logp(hidden, weight, target, bias)

    def step():
        grads = rlk.linear_logp_backward(hidden, weight, target, lse, gl, bias)
        return grads + (rlk.det_gemm_fwd(A, B), rlk.det_gemm_da(dC.float(), B),
                        rlk.det_gemm_db(A, dC, out_dtype=torch.float32))

    eager = step()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = step()
    for _ in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, eager):
            assert torch.equal(a, b)
    assert rlk.device_error() == 0


def test_det_gemm_last_wave_split_graph_replay(dev):
    """A product whose last wave runs as half tiles in a second launch (16 x 16 wide
    tiles, reduction 16384) replays from a graph with the eager bits, after a torch
    kernel that rewrites its input inside the same graph."""
    A, B, _ = si.det_gemm_inputs(4096, 16384, 3900, seed=58, device=dev)
    A0 = A.clone()

    def step():
        A.copy_(A0)
        return rlk.det_gemm_fwd(A, B, out_dtype=torch.float32)

    eager = step()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = step()
    for _ in range(2):
        out.zero_()
        A.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), eager.view(torch.int32))
    assert rlk.device_error() == 0


@pytest.mark.parametrize("N", [17, 1000])
def test_calls_see_inputs_written_just_before(dev, N):
    """Each library kernel may start while the previous kernel in the stream is
    finishing (programmatic dependent launch) and waits for it before touching
    memory: a torch kernel that rewrites the inputs right before every call, with
    no synchronisation in between, is always seen."""
    H, V = 1024, 20000
    hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=56, device=dev)
    A, B, _ = si.det_gemm_inputs(N, H, 768, seed=57, device=dev)
    want = {}
    for sign in (1.0, -1.0):
        want[sign] = (rlk.linear_logp(hidden * sign, weight, target, bias),
                      rlk.det_gemm_fwd(A * sign, B, out_dtype=torch.float32))
    torch.cuda.synchronize()
    got = []
    sign = 1.0
    for _ in range(8):
        hidden.mul_(-1.0)            # torch kernels, immediately followed by the library's
        A.mul_(-1.0)
        sign = -sign
        got.append((sign, rlk.linear_logp(hidden, weight, target, bias),
                    rlk.det_gemm_fwd(A, B, out_dtype=torch.float32)))
    torch.cuda.synchronize()
    for sign, lp, c in got:
        (wl, wc) = want[sign]
        assert torch.equal(lp[0], wl[0]) and torch.equal(lp[1], wl[1]) and torch.equal(c, wc)
    assert rlk.device_error() == 0


def test_vocabulary_shards_and_two_product_backward_graph_replay(dev):
    """Shard partials (two shards, one staged through its workspace), the merge over
    the gathered shards, and the two-product det_gemm backward with an FP32 dC
    (one shared BF16 rounding) captured in one graph replay with the eager bits."""
    N, H, V = 300, 1002, 32003                      # pitch 1002: hidden and W shards staged
    hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=57, device=dev)
    S, vps, _ = rlk.vocab_split_policy(V)
    cut = 50
    offsets = [0, cut, S]
    v_cut = cut * vps * 256
    shards = [(weight[:v_cut].contiguous(), bias[:v_cut].contiguous(), 0, cut),
              (weight[v_cut:].contiguous(), bias[v_cut:].contiguous(), cut, S)]
    A, B, dC = si.det_gemm_inputs(520, 300, 264, seed=58, device=dev, dc_dtype=torch.float32)

    def run():
        parts, zts = [], []
        for w_, b_, j0, j1 in shards:
            p, z = rlk.linear_logp_shard_partials(hidden, w_, target, V, j0, j1, b_,
                                                  ld_partials=S - cut)
            parts.append(p)
            zts.append(z)
        out = rlk.linear_logp_combine_shards(torch.stack(parts), torch.stack(zts), offsets, target,
                                             V, return_target_logit=True)
        return out + rlk.det_gemm_backward(dC, A, B, torch.float32)

    eager = [t.clone() for t in run()]
    ref = rlk.linear_logp(hidden, weight, target, bias, return_target_logit=True)
    for a, b in zip(eager[:3], ref):
        assert torch.equal(a, b)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = run()
    for _ in range(2):
        for t in outs:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, eager):
            assert torch.equal(a, b)
    assert rlk.device_error() == 0
