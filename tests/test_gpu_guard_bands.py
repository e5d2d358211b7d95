"""Sanitizer substitutes on the GPU (compute-sanitizer is closed on this machine).

1. Guard-band canaries (tests/guard_bands.py) around every output and workspace
   buffer of linear-logp, its backward, the det_gemm products and the shard
   partials, at N in {1, 33, 129}, H in {1, 8, 100}, V in {1, 257, 32003}:
   nothing outside the documented bytes is written.
2. The debug build (librlk_debug.so, -DRLK_DEBUG) runs the same shapes in a child
   process: every kernel checks each global store's index against its buffer's
   extent, so the error word must stay 0; its own selftest (a store declared
   out of range, skipped without touching memory) must raise RLK_DEVERR_BOUNDS;
   and the per-CTA phase trace of a linear-logp call must be ordered in time.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import guard_bands
from helpers import cuda_or_skip

pytestmark = pytest.mark.gpu
TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def test_guard_bands_release_build(dev):
    fails = guard_bands.run_all(dev)
    assert not fails, fails[:10]
    assert rlk.device_error() == 0


CHILD = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import numpy as np
import torch
import deterministic_invariant_gemm_linear_gb300 as rlk
import guard_bands
import seeded_inputs as si
dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
res = {{"debug": rlk.is_debug_build(), "lib": rlk.LIB_PATH}}
res["fails"] = guard_bands.run_all(dev)
res["error_word"] = rlk.device_error()
res["selftest_status"] = rlk.lib().rlk_selftest_store_check(rlk._stream_ptr(None))
res["selftest_word"] = rlk.device_error()
res["after"] = rlk.device_error()
ordered = []
for N in (17, 300):
    hidden, weight, bias, target = si.linear_logp_inputs(N, 2048, 32003, seed=1, device=dev)
    rlk.linear_logp(hidden, weight, target, bias)
    rlk.debug_trace()                                   # clears
    rlk.linear_logp(hidden, weight, target, bias)
    tr = rlk.debug_trace().astype(np.int64)
    used = tr[tr[:, 4] > 0]
    # the fields a CTA recorded (the second CTA of a pair issues no MMAs: no field 2)
    times = used[:, :6]                             # fields 6 and 7 are cycle counts
    # role counters: every MMA issuer issued tiles, and no wait exceeds its role's span
    mma = used[used[:, 10] > 0]
    roles_ok = bool(len(mma) > 0 and np.all(mma[:, 11] > 0) and
                    np.all(mma[:, 8] + mma[:, 9] <= mma[:, 10]) and
                    np.all(used[:, 12] <= used[:, 13]) and np.all(used[:, 13] > 0))
    ordered.append([int(len(used)), all(bool(np.all(np.diff(r[r > 0]) >= 0)) for r in times),
                    roles_ok, int(len(mma))])
res["trace"] = ordered
res["final_word"] = rlk.device_error()
print(json.dumps(res))
"""


def test_debug_build_store_checks_and_trace(dev):
    from deterministic_invariant_gemm_linear_gb300 import build as b
    b.build(flavors=("debug",))
    env = dict(os.environ, RLK_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, tests=TESTS)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["debug"] == 1 and res["lib"].endswith("librlk_debug.so")
    assert res["fails"] == [], res["fails"][:10]
    assert res["error_word"] == 0                     # no store outside its buffer
    assert res["selftest_status"] == 0
    assert res["selftest_word"] == rlk.RLK_DEVERR_BOUNDS and res["after"] == 0
    # 17 rows: one CTA per vocabulary tile (126); 300 rows: persistent CTA pairs
    (n17, ok17, roles17, mma17), (n300, ok300, roles300, mma300) = res["trace"]
    assert n17 == 126 and ok17
    assert n300 > 0 and ok300
    # one-CTA loop: every CTA issues its own MMAs; 2-SM loop: one issuer per pair
    assert roles17 and mma17 == 126
    assert roles300 and mma300 == n300 // 2
    assert res["final_word"] == 0


def test_release_build_has_no_debug_entry_points(dev):
    if os.environ.get("RLK_LIBRARY") == "debug":
        pytest.skip("the whole suite is running against the debug build (RLK_LIBRARY=debug)")
    assert not rlk.is_debug_build()
    assert rlk.lib().rlk_selftest_store_check(rlk._stream_ptr(None)) == 10  # NOT_DEBUG_BUILD
    assert rlk.device_error() == 0
