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


def test_traffic_figures_are_gated_by_the_kernel_source_hash(tmp_path, monkeypatch):
    """bench.py reports ncu DRAM bytes only while the kernel source they were taken on is unchanged."""
    import json
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import hashlib
    import types

    import bench
    src = tmp_path / "k.cu"
    src.write_text("kernel source\n")
    (tmp_path / "profiles").mkdir()
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    rec = {"source": "k.cu", "source_sha256": sha, "dram_bytes_per_launch": {"attn": 123}}
    (tmp_path / "profiles" / "traffic_qwen3-4b-32k-2bit.txt").write_text("# header\n" + json.dumps(rec) + "\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    w = types.SimpleNamespace(n=32768, sketch="2bit")
    assert bench.measured_traffic(w) == {"attn": 123}
    src.write_text("kernel source, changed\n")
    assert bench.measured_traffic(w) == {}
    assert bench.measured_traffic(types.SimpleNamespace(n=32768, sketch="int8")) == {}
