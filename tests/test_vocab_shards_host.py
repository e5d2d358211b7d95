"""Host logic of the vocabulary-parallel linear-logp (no GPU needed).

The split policy of "feat(linear-logp): add batch-invariant fused SM90 operator"
(author notes: V -> split count -> contiguous ranges -> ordered merge) lets the
vocabulary be divided at split boundaries.  Checked here on the CPU:
  * rlk_vocab_shard_range partitions the S splits into contiguous runs that
    cover every split and every vocabulary id exactly once;
  * the shard entry points validate their arguments before touching a device;
  * the exchange step (exchange_shard_partials) gathers every rank's padded
    partials and target logits in rank order over gloo, world size 2.
"""
import ctypes
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

import deterministic_invariant_gemm_linear_gb300 as rlk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P16 = ctypes.c_void_p(0x10000)          # never dereferenced: validation fails first


@pytest.fixture(scope="module")
def lib():
    from deterministic_invariant_gemm_linear_gb300 import build as b
    b.build()
    return rlk.lib()


@pytest.mark.parametrize("V", [1, 255, 1024, 32003, 151936, 152064, 300007])
@pytest.mark.parametrize("R", [1, 2, 3, 8, 64])
def test_shard_ranges_partition_the_splits(lib, V, R):
    S, vps, vt = rlk.vocab_split_policy(V)
    ranges = [rlk.vocab_shard_range(V, R, q) for q in range(R)]
    assert ranges[0][0] == 0 and ranges[-1][1] == S
    assert ranges[0][2] == 0 and ranges[-1][3] == V
    for q in range(R):
        j0, j1, v0, v1 = ranges[q]
        assert j0 <= j1 and v0 <= v1
        if q + 1 < R:
            assert ranges[q + 1][0] == j1 and ranges[q + 1][2] == v1    # contiguous
        assert v0 == min(j0 * vps * 256, V) and v1 == min(j1 * vps * 256, V)
        assert (j1 - j0) in (S // R, -(-S // R))                         # balanced
        if j1 > j0:
            assert v1 > v0                                               # every split holds ids


def test_shard_range_rejects(lib):
    x = ctypes.c_int64()
    r = ctypes.byref(x)
    assert lib.rlk_vocab_shard_range(1000, 0, 0, r, r, r, r) == 2
    assert lib.rlk_vocab_shard_range(1000, 65, 0, r, r, r, r) == 2
    assert lib.rlk_vocab_shard_range(1000, 2, 2, r, r, r, r) == 2
    assert lib.rlk_vocab_shard_range(0, 1, 0, r, r, r, r) == 2
    assert lib.rlk_vocab_shard_range(1000, 1, 0, None, r, r, r) == 1


def test_shard_partials_validates_before_any_device_use(lib):
    f = lib.rlk_linear_logp_shard_partials
    V, S = 151936, 594
    # split range outside [0, S], reversed, or wider than ld_partials
    for j0, j1, ld in ((0, S + 1, S + 1), (5, 4, 8), (-1, 3, 8), (0, 10, 9)):
        assert f(P16, 8, 64, 64, P16, V, j0, j1, 64, None, P16, 1, P16, ld, P16, P16, 1 << 20,
                 None) == 2
    # a weight pitch below H
    assert f(P16, 8, 64, 64, P16, V, 0, 2, 63, None, P16, 1, P16, 2, P16, P16, 1 << 20, None) == 2
    # no rows or an empty shard: nothing to do
    assert f(P16, 0, 64, 64, P16, V, 0, 2, 64, None, P16, 1, P16, 2, P16, P16, 1 << 20, None) == 0
    assert f(P16, 8, 64, 64, P16, V, 3, 3, 64, None, P16, 1, P16, 1, P16, P16, 1 << 20, None) == 0
    # missing outputs
    assert f(P16, 8, 64, 64, P16, V, 0, 2, 64, None, P16, 1, None, 2, P16, P16, 1 << 20, None) == 1
    # workspace size: 256 bytes of counter when nothing is staged, 0 for bad arguments
    ws = lib.rlk_linear_logp_shard_workspace_size
    assert ws(P16, 8, 64, 64, P16, V, 0, 2, 64) == 256
    assert ws(P16, 8, 64, 64, P16, V, 0, S + 1, 64) == 0
    staged = ws(ctypes.c_void_p(0x10002), 8, 64, 64, P16, V, 0, 2, 64)
    assert staged == 256 + 8 * 64 * 2


def test_combine_shards_validates_before_any_device_use(lib):
    f = lib.rlk_linear_logp_combine_shards
    V, S, N = 151936, 594, 8
    Offs = ctypes.c_int64 * 3

    def call(offs, R=2, ld=300, shard_stride=N * 300, zt_stride=N):
        return f(N, V, P16, 1, R, offs, P16, ld, shard_stride, P16, zt_stride, P16, P16, None, None)

    assert call(Offs(1, 300, S)) == 2             # must start at 0
    assert call(Offs(0, 300, S - 1)) == 2         # must end at S
    assert call(Offs(0, 400, 300)) == 2           # decreasing
    assert call(Offs(0, 300, S), ld=299) == 2     # a shard wider than ld
    assert call(Offs(0, 300, S), shard_stride=N * 300 - 1) == 2   # shard blocks overlap
    assert call(Offs(0, 300, S), zt_stride=N - 1) == 2
    assert call(Offs(0, 300, S), R=0) == 2
    assert f(N, V, P16, 1, 2, None, P16, 300, N * 300, P16, N, P16, P16, None, None) == 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _exchange_rank(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import deterministic_invariant_gemm_linear_gb300 as rlk_
    dist.init_process_group("gloo", rank=rank, world_size=world)
    N, ld = 5, 7
    # rank r's partials hold (r, row, column) codes; its target logits hold (r, row)
    p = torch.tensor([[[rank * 1000 + r * 10 + c, -c] for c in range(ld)] for r in range(N)],
                     dtype=torch.float32)
    z = torch.tensor([rank * 100 + r for r in range(N)], dtype=torch.float32)
    gp, gz = rlk_.exchange_shard_partials(p, z)
    out[rank] = (gp.tolist(), gz.tolist())
    dist.destroy_process_group()


def test_exchange_gathers_in_rank_order_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_exchange_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    N, ld = 5, 7
    want_p = [[[[q * 1000 + r * 10 + c, -c] for c in range(ld)] for r in range(N)]
              for q in range(world)]
    want_z = [[q * 100 + r for r in range(N)] for q in range(world)]
    for rank in range(world):
        gp, gz = out[rank]
        assert gp == want_p and gz == want_z


def test_ordered_sum_validates_before_any_device_use(lib):
    f = lib.rlk_sum_partials_ordered
    assert f(P16, 0, 4, 4, 4, 16, P16, 1, 4, None) == 2          # no parts
    assert f(P16, 2, 4, 4, 4, 15, P16, 1, 4, None) == 2          # parts overlap
    assert f(P16, 2, 4, 4, 3, 16, P16, 1, 4, None) == 2          # pitch below the columns
    assert f(P16, 2, 4, 4, 4, 16, P16, 5, 4, None) == 3          # unknown dtype
    assert f(ctypes.c_void_p(0x10002), 2, 4, 4, 4, 16, P16, 1, 4, None) == 4
    assert f(P16, 2, 0, 4, 4, 0, P16, 1, 4, None) == 0           # no rows: nothing to do
