"""dB with its rows divided between devices: per-device partial products, then a
fixed-order sum (rlk_sum_partials_ordered).

"feat(musa): add native deterministic gemm kernel", Summary: dB = A^T dC reduces
over the batch rows in a fixed order.  When those rows are spread over devices,
each device forms its FP32 partial over its own rows and the partials are added
in a fixed device order, never by a ring all-reduce whose order depends on the
ring.  Checked here on one GPU:
  * the ordered sum equals float32 additions in the same order, bit for bit;
  * a row-sharded dB is run-to-run bitwise, within the FP32 bound of the FP64
    oracle, and its BF16 output is the rounding of its FP32 output;
  * two processes exchanging their partials through gloo get the same bits as
    the one-process computation.
"""
import os
import socket
import sys
import tempfile

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import GEMM_FP32_REL_FRO, cuda_or_skip, rel_fro, sample_rows

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


@pytest.mark.parametrize("P,rows,cols", [(1, 1, 1), (2, 33, 100), (3, 1000, 257), (5, 64, 4096)])
def test_ordered_sum_is_float32_addition_in_part_order(dev, P, rows, cols):
    g = torch.Generator(device=dev).manual_seed(P * rows + cols)
    parts = torch.randn(P, rows, cols, generator=g, device=dev) * \
        torch.logspace(-3, 3, P, device=dev)[:, None, None]
    want = parts[0].clone()
    for q in range(1, P):
        want = want + parts[q]
    got = rlk.sum_partials_ordered(parts, torch.float32)
    assert torch.equal(got, want)
    assert torch.equal(rlk.sum_partials_ordered(parts, torch.bfloat16), want.to(torch.bfloat16))
    assert rlk.device_error() == 0


def _sharded_db(A, dC, cuts, out_dtype):
    parts = [rlk.det_gemm_db(A[a:b], dC[a:b], out_dtype=torch.float32)
             for a, b in zip(cuts[:-1], cuts[1:])]
    return rlk.sum_partials_ordered(torch.stack(parts), out_dtype), parts


def test_row_sharded_db(dev, orc):
    M, K, N = 4096, 1024, 768
    A, _, dC = si.det_gemm_inputs(M, K, N, seed=61, device=dev)
    cuts = [0, 1000, 2500, M]                                  # three uneven row shards
    db32, parts = _sharded_db(A, dC, cuts, torch.float32)
    want = parts[0] + parts[1] + parts[2]
    assert torch.equal(db32, want)
    again, _ = _sharded_db(A, dC, cuts, torch.float32)
    assert torch.equal(again, db32)                           # run to run
    db16, _ = _sharded_db(A, dC, cuts, torch.bfloat16)
    assert torch.equal(db16, db32.to(torch.bfloat16))
    rows = sample_rows(K, 24, seed=62, must=(255, 256, 1023))
    ref = orc.gemm_db(si.bf16_bits(A), si.bf16_bits(dC), rows=rows)
    assert rel_fro(db32.cpu().numpy()[rows].astype(np.float64), ref) <= GEMM_FP32_REL_FRO
    whole = rlk.det_gemm_db(A, dC, out_dtype=torch.float32)   # one device, one order
    assert rel_fro(db32.cpu().double().numpy(), whole.cpu().double().numpy()) <= GEMM_FP32_REL_FRO
    assert rlk.device_error() == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _db_rank(rank, world, port, outdir, M, K, N):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import deterministic_invariant_gemm_linear_gb300 as rlk_
    import seeded_inputs as si_
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    A, _, dC = si_.det_gemm_inputs(M, K, N, seed=63, device=dev)
    half = M // 2
    rows = slice(0, half) if rank == 0 else slice(half, M)
    db = rlk_.det_gemm_db_row_sharded(A[rows].contiguous(), dC[rows].contiguous(), torch.float32)
    torch.cuda.synchronize()
    torch.save(db.cpu(), os.path.join(outdir, f"rank{rank}.pt"))
    dist.destroy_process_group()


def test_two_ranks_exchange_through_gloo(dev):
    M, K, N = 2048, 512, 640
    A, _, dC = si.det_gemm_inputs(M, K, N, seed=63, device=dev)
    want, _ = _sharded_db(A, dC, [0, M // 2, M], torch.float32)
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with tempfile.TemporaryDirectory() as d:
        procs = [ctx.Process(target=_db_rank, args=(r, world, port, d, M, K, N))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        for r in range(world):
            assert torch.equal(torch.load(os.path.join(d, f"rank{r}.pt")), want.cpu())
