"""CPU test of the benchmark's multi-rank path (replicas on N GPUs, one process
each): two gloo ranks agree on the slowest rank's time and on the whole-job
throughput, and the reference arm's non-zero ranks exit without work."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        t = bench.slowest_rank_ms(ms, world)
        q.put((rank, t, bench.job_tops(2e12, 4, world, t)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_throughput():
    torch = pytest.importorskip("torch")
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expected = 2e12 * 4 * 2 / (15.0 * 1e-3) / 1e12   # both ranks' work over the slowest time
    for rank, t, v in results:
        assert t == 15.0
        assert v == pytest.approx(expected)


def test_single_rank_is_unchanged():
    import bench
    assert bench.slowest_rank_ms(12.5, 1) == 12.5
    assert bench.job_tops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(argparse.Namespace(workload="tiny", steps=1, warmup=3))
    assert out.getvalue() == ""
