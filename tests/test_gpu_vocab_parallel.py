"""Vocabulary-parallel linear-logp: merged shards equal the one-device operator bit for bit.

"feat(linear-logp): add batch-invariant fused SM90 operator", author notes: the
split count comes from V alone and the merge takes the splits' partials in a
fixed order.  Dividing the vocabulary at split boundaries therefore changes only
where each split is computed: every split's (m, s) partial and every target
logit are the same bits, and the fixed-order merge over the gathered shards
reproduces logp, lse and the target logit exactly (compared as bit patterns,
torch.equal on int32 views, so NaN rows compare too).
"""
import os
import socket
import sys
import tempfile

import pytest
import torch
import torch.multiprocessing as mp

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


def run_shards(hidden, weight, target, bias, V, offsets):
    """Each shard's partials from its own weight rows, gathered and merged."""
    S, vps, _ = rlk.vocab_split_policy(V)
    widest = max(b - a for a, b in zip(offsets[:-1], offsets[1:]))
    parts, zts = [], []
    for j0, j1 in zip(offsets[:-1], offsets[1:]):
        v0, v1 = min(j0 * vps * 256, V), min(j1 * vps * 256, V)
        w = weight[v0:v1].clone()                       # the shard holds only its own rows
        b = None if bias is None else bias[v0:v1].clone()
        p, z = rlk.linear_logp_shard_partials(hidden, w, target, V, j0, j1, b, ld_partials=widest)
        parts.append(p)
        zts.append(z)
    return rlk.linear_logp_combine_shards(torch.stack(parts), torch.stack(zts), offsets, target, V,
                                          return_target_logit=True)


CASES = [
    # (N, H, V, bias, shard split offsets as fractions of S)
    (1000, 4096, 151936, False, (0.0, 0.17, 1.0)),
    (1000, 4096, 151936, False, (0.0, 0.002, 0.5, 1.0)),
    (17, 4096, 151936, True, (0.0, 0.6, 1.0)),               # one-CTA loop
    (300, 1024, 300007, True, (0.0, 0.013, 0.7, 1.0)),       # two 256-id tiles per split
    (300, 1024, 300007, True, (0.0, 0.5, 1.0)),
]


@pytest.mark.parametrize("N,H,V,bias,fr", CASES)
def test_merged_shards_equal_the_whole_vocabulary_call(dev, N, H, V, bias, fr):
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=bias, seed=N + V, device=dev)
    target[0], target[N - 1] = V - 1, 0
    if N > 4:
        target[2] = -1                                   # out of range: NaN in both
    S = rlk.vocab_split_policy(V)[0]
    offsets = sorted({0, S, *[min(S, max(0, round(f * S))) for f in fr]})
    ref = rlk.linear_logp(hidden, weight, target, b, return_target_logit=True)
    got = run_shards(hidden, weight, target, b, V, offsets)
    for x, y, name in zip(ref, got, ("logp", "lse", "target_logit")):
        assert bits_equal(x, y), f"offsets {offsets}: {name} bits differ"
    assert rlk.device_error() == 0


def test_balanced_shards_and_empty_ones(dev):
    """The balanced partition for 2, 3 and 8 shards, and a partition with empty shards."""
    N, H, V = 129, 1024, 32003
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=True, seed=5, device=dev)
    ref = rlk.linear_logp(hidden, weight, target, b, return_target_logit=True)
    S = rlk.vocab_split_policy(V)[0]
    for R in (2, 3, 8):
        offsets = [rlk.vocab_shard_range(V, R, q)[0] for q in range(R)] + [S]
        got = run_shards(hidden, weight, target, b, V, offsets)
        for x, y in zip(ref, got):
            assert bits_equal(x, y), f"{R} balanced shards"
    got = run_shards(hidden, weight, target, b, V, [0, 0, 50, 50, S, S])
    for x, y in zip(ref, got):
        assert bits_equal(x, y), "empty shards"


def test_shard_partials_are_the_whole_calls_partials(dev):
    """A shard's (m, s) pairs equal the matching columns of the whole call's [N][S]
    partials, and its target logits those of the rows whose target it holds."""
    N, H, V = 300, 2048, 151936
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, seed=21, device=dev)
    call = rlk.LinearLogpCall(hidden, weight, target, b)
    call.partials()
    S, vps, _ = rlk.vocab_split_policy(V)
    whole = call.ws[:N * S * 8].view(torch.float32).view(N, S, 2)
    off_zt = -(-N * S * 8 // 256) * 256
    whole_zt = call.ws[off_zt:off_zt + 4 * N].view(torch.float32)
    for j0, j1 in ((0, 1), (100, 333), (590, 594)):
        v0, v1 = j0 * 256, min(j1 * 256, V)
        p, z = rlk.linear_logp_shard_partials(hidden, weight[v0:v1].clone(), target, V, j0, j1)
        assert bits_equal(p[:, :j1 - j0], whole[:, j0:j1])
        held = (target >= v0) & (target < v1)
        assert bits_equal(z[held], whole_zt[held])
        assert bool(torch.isnan(z[~held]).all())
    assert rlk.device_error() == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _vp_rank(rank, world, port, outdir, N, H, V):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    import deterministic_invariant_gemm_linear_gb300 as rlk_
    import seeded_inputs as si_
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    hidden, weight, b, target = si_.linear_logp_inputs(N, H, V, bias=True, seed=77, device=dev)
    _, _, v0, v1 = rlk_.vocab_shard_range(V, world, rank)
    w_shard, b_shard = weight[v0:v1].clone(), b[v0:v1].clone()
    del weight, b
    out = rlk_.vocab_parallel_linear_logp(hidden, w_shard, target, V, b_shard,
                                          return_target_logit=True)
    torch.cuda.synchronize()
    torch.save([o.cpu() for o in out], os.path.join(outdir, f"rank{rank}.pt"))
    dist.destroy_process_group()


@pytest.mark.parametrize("N,H,V", [(300, 1024, 32003), (64, 2048, 151936)])
def test_two_ranks_exchange_through_gloo(dev, N, H, V):
    """Two processes (gloo, world size 2), each holding half of the vocabulary's
    weight rows, exchange their partials as host tensors and merge: both ranks
    get the one-device bits.  Both run on this one GPU; their kernels never wait
    on each other (the exchange is on the host)."""
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=True, seed=77, device=dev)
    ref = [o.cpu() for o in rlk.linear_logp(hidden, weight, target, b, return_target_logit=True)]
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with tempfile.TemporaryDirectory() as d:
        procs = [ctx.Process(target=_vp_rank, args=(r, world, port, d, N, H, V))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        for r in range(world):
            got = torch.load(os.path.join(d, f"rank{r}.pt"))
            for x, y in zip(ref, got):
                assert bits_equal(x, y), f"rank {r}"


def test_merged_shards_match_the_oracle(dev, orc):
    """The merged shards against the FP64 oracle directly (|delta| <= 1e-3 on logp and
    lse, target logit within 1e-4), V = 300,007 (two 256-id tiles per split), three
    uneven shards, bias, every row."""
    from helpers import assert_logp_close
    N, H, V = 200, 512, 300007
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=True, seed=71, device=dev)
    S = rlk.vocab_split_policy(V)[0]
    logp, lse, zt = run_shards(hidden, weight, target, b, V, [0, 3, 401, S])
    torch.cuda.synchronize()
    rlp, rls, rzt = orc.linear_logp(si.bf16_bits(hidden), si.bf16_bits(weight),
                                    target.cpu().numpy(), b.cpu().numpy())
    assert_logp_close(logp.cpu().numpy(), lse.cpu().numpy(), rlp, rls, "merged shards")
    assert float((zt.cpu().double() - torch.from_numpy(rzt)).abs().max()) <= 1e-4
    assert rlk.device_error() == 0


def test_shard_partials_are_batch_invariant(dev):
    """A shard's partials for a chunk of rows equal the same rows of the shard's
    partials for the whole batch (1-, 7- and 129-row chunks; one-CTA and 2-SM loops)."""
    N, H, V = 300, 1024, 151936
    hidden, weight, b, target = si.linear_logp_inputs(N, H, V, bias=True, seed=75, device=dev)
    j0, j1 = 100, 250
    v0, v1 = j0 * 256, j1 * 256
    w, bb = weight[v0:v1].contiguous(), b[v0:v1].contiguous()
    full_p, full_z = rlk.linear_logp_shard_partials(hidden, w, target, V, j0, j1, bb)
    for chunk in (1, 7, 129):
        for s0 in range(0, N, chunk * 11):
            rows = slice(s0, min(N, s0 + chunk))
            p, z = rlk.linear_logp_shard_partials(hidden[rows], w, target[rows], V, j0, j1, bb)
            assert bits_equal(p, full_p[rows]), f"chunk {chunk} at {s0}"
            assert bits_equal(z, full_z[rows])
    assert rlk.device_error() == 0
