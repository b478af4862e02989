"""The multi-rank plumbing of bench.py on CPU with two gloo ranks: every rank
learns the slowest rank's step time, and the whole-job rate counts every
rank's units over that time (weak scaling, no data exchange between ranks)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = [2.0, 5.0][rank]
    ms = bench.reduce_max(my_ms, dist, "cpu")
    rate = bench.whole_job_rate(1e9, world, ms)
    out.put((rank, ms, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    # two ranks x 1e9 units in the slowest rank's 5 ms
    assert res[0][2] == pytest.approx(2 * 1e9 / 5e-3)


def test_single_rank_is_the_identity():
    import bench
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.whole_job_rate(10, 1, 1000.0) == pytest.approx(10.0)
