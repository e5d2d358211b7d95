"""Concurrent callers: the library keeps no per-call state outside the caller's
workspace (host caches are mutex-guarded; each call's unit counter lives in its
own workspace; no kernel waits on another grid's blocks), so calls from several
host threads on their own streams run side by side and still give the serial
bits.  ctypes releases the GIL around each library call, so the host calls
overlap too.
"""
import threading

import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def test_threads_on_their_own_streams_give_the_serial_bits(dev):
    hidden, weight, bias, target = si.linear_logp_inputs(300, 1024, 32003, bias=True, seed=9,
                                                         device=dev)
    small = (hidden[:40], target[:40])                     # one-CTA loop
    A, B, dC = si.det_gemm_inputs(1000, 1000, 1000, seed=9, device=dev)
    ref = {
        "lp": rlk.linear_logp(hidden, weight, target, bias),
        "lp_small": rlk.linear_logp(small[0], weight, small[1], bias),
        "fwd": rlk.det_gemm_fwd(A, B),
        "two": rlk.det_gemm_backward(dC.float(), A, B),
    }
    torch.cuda.synchronize()
    out, errors = {}, []

    def worker(k):
        try:
            s = torch.cuda.Stream(device=dev)
            with torch.cuda.stream(s):
                got = []
                for _ in range(4):
                    got.append({
                        "lp": rlk.linear_logp(hidden, weight, target, bias),
                        "lp_small": rlk.linear_logp(small[0], weight, small[1], bias),
                        "fwd": rlk.det_gemm_fwd(A, B),
                        "two": rlk.det_gemm_backward(dC.float(), A, B),
                    })
            s.synchronize()
            out[k] = got
        except Exception as e:                              # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert sorted(out) == [0, 1, 2, 3]
    for got in out.values():
        for g in got:
            for name in ("lp", "lp_small", "two"):
                for a, b in zip(g[name], ref[name]):
                    assert torch.equal(a, b), name
            assert torch.equal(g["fwd"], ref["fwd"])
    assert rlk.device_error() == 0
