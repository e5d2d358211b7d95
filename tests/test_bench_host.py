"""Host-side pieces of bench.py's output contract (no GPU): the headline metric
string, and the config that both arms (GPU and reference) print for a workload."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import seeded_inputs as si  # noqa: E402


def test_mid_metric_is_the_headline_metric():
    assert bench.linear_logp_metric(si.MID) == bench.METRIC


def test_config_states_workload_batch_and_l2_rule():
    mid = bench.linear_logp_config(si.MID, 1)
    assert mid["global_batch"] == 4096 and mid["parallelism"] == "replicas x1"
    assert "N=4096 H=4096 V=151936" in mid["workload"]
    assert mid["l2"].startswith("inputs larger than L2")        # 1.245 GB weight streams from HBM
    tiny = bench.linear_logp_config(si.TINY, 2)
    assert tiny["global_batch"] == 2 * 64 and tiny["parallelism"] == "replicas x2"
    assert "+bias" in tiny["workload"] and tiny["l2"].startswith("L2 flushed")
    assert bench.linear_logp_config(si.MID, 1) == mid             # pure: both arms get equal dicts
