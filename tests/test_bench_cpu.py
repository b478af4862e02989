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


def _brute_pairs(b):
    total = 0
    for qo, kv in zip(b.qo_lens.tolist(), b.kv_lens.tolist()):
        for i in range(qo):
            pos = kv - qo + i
            for t in range(kv):
                if b.causal and t > pos:
                    continue
                if b.window_left >= 0 and t < pos - b.window_left:
                    continue
                total += 1
    return total


@pytest.mark.parametrize("seed", range(8))
def test_visible_pairs_count_the_mask(seed):
    import numpy as np
    g = np.random.default_rng(seed)
    kv = g.integers(0, 90, size=5)
    qo = np.minimum(g.integers(1, 40, size=5), np.maximum(kv, 1))
    qo[kv == 0] = 0
    causal = bool(seed % 2)
    b = synth.make_batch("pairs", kv, qo, 2, 1, 64, 16, synth.NHD, None, causal, seed,
                         window_left=int(g.choice([-1, 0, 5, 31])))
    assert bench.visible_pairs(b) == _brute_pairs(b)


def test_square_causal_prefill_counts_the_triangle():
    b = synth.make_batch("tri", [300, 17], [300, 17], 2, 1, 64, 16, synth.NHD, None, True, 0)
    assert bench.visible_pairs(b) == 300 * 301 // 2 + 17 * 18 // 2
    assert bench.attention_flops(b) == 4 * 64 * 2 * bench.visible_pairs(b)


def test_kv_bytes_count_shared_prefix_pages_once():
    kv = [100, 70, 40, 33]
    b = synth.make_batch("shared", kv, [1, 1, 1, 1], 4, 2, 64, 16, synth.NHD, None, False, 1,
                         shared_prefix_requests=3, shared_prefix_tokens=32)
    unique = sum(kv) - 2 * 32                         # three requests share two full pages
    assert bench.kv_bytes(b) == unique * 2 * 2 * 64 * 2


def test_default_line_covers_every_configuration():
    names = [n for n, _ in bench.SECONDARY]
    assert all(n in bench.WORKLOADS for n in names)
    # the 70B GQA decode, prefill at 1K/4K/16K/32K, the ragged and the mixed batch
    for n in ("llama70b_gqa_decode", "causal_prefill_1k", "causal_prefill_4k",
              "causal_prefill_16k", "causal_prefill_32k", "ragged_prefill",
              "mixed_chunk_decode"):
        assert n in names
    assert all(cap >= 5 for _, cap in bench.SECONDARY)


def test_clock_summary_reads_each_timed_window():
    c = bench.ClockSampler(0)
    row = lambda mhz, cap: ["0", str(mhz), "2070", "500", "0x0", "Not Active", "Not Active",
                            "Not Active", "Active" if cap else "Not Active"]
    c.samples = [(10.0, row(2070, False)), (10.5, row(2070, False)),
                 (20.0, row(1500, True)), (20.5, row(1600, True))]
    c.windows = [(9.9, 10.6), (19.9, 20.6)]
    first, second = c.summary(0), c.summary(1)
    assert first["sm_mhz"] == 2070 and first["reasons"] == []
    assert second["sm_mhz"] == 1550 and second["reasons"] == ["sw_power_cap"]
    assert second["window"] == "timed region"
