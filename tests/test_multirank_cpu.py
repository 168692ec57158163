"""The N > 1 replica path of bench.py on CPU: two gloo ranks, each with its own step time; both must
report the slowest rank's time and the whole-job value (units of both ranks over that time)."""
import os
import socket
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_replica_aggregation():
    mp = pytest.importorskip("torch.multiprocessing")
    import multirank_worker
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=multirank_worker.run, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, step_ms in got:
        assert step_ms == 5.0
        assert value == pytest.approx(2 * 1000 / 5e-3)


def test_workload_seed_differs_per_rank():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import types

    import bench
    args = types.SimpleNamespace(n=256, decode_steps=2, sketch="2bit")
    w0, w1 = bench.workload(args, 0), bench.workload(args, 1)
    assert not (w0.K == w1.K).all()
