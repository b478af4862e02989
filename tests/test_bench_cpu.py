"""Host-only parts of bench.py: the planner timing reported beside the
device numbers (fi_plan runs on the CPU before every serving step)."""
import os
import sys

import pytest

pytest.importorskip("torch")
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from paged_kv_attention_27_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("name,items", [("tiny_decode", None), ("llama7b_decode", 2048)])
def test_plan_timing_reports_the_plan_the_step_runs(name, items):
    b = bench.make_workload(name)
    t = bench.time_plan(b, 152, calls=20)
    assert t["calls"] == 20 and t["median_us"] > 0
    if items is not None:
        assert t["items"] == items


def test_plan_timing_of_a_prefill_batch_uses_a_prefill_plan():
    b = synth.causal_prefill(1024, batch=1)
    t = bench.time_plan(b, 152, calls=5)
    # 8 row tiles of 128 x 64 query heads
    assert t["items"] == 8 * 64
