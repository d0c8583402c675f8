"""The bench's multi-rank path on CPU: two gloo ranks (no GPU).

Under torchrun every rank runs the same workload on its own GPU (replicas: the
projection has no exchange step at TP1); the line reports the bytes of all
ranks over the slowest rank's time, and only rank 0 prints.  These tests run
the rank-aggregation helpers and the reference arm's rank handling on two CPU
processes with the gloo backend.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        slowest = bench.reduce_max(10.0 + 5.0 * rank)  # rank 1 is the slower one
        tdist.barrier()
        gbs = bench.whole_job_gbs(1_000_000, 100, world, slowest)
        out.put((rank, slowest, gbs))
    finally:
        tdist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_all_bytes():
    port = free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=10) for _ in range(2))
    for rank, slowest, gbs in res:
        assert slowest == 15.0  # the max over ranks, on every rank
        assert gbs == pytest.approx(2 * 1_000_000 * 100 / 15e-3 / 1e9)


def test_reduce_max_without_process_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_gbs(2_000_000_000, 10, 1, 1000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Ranks other than 0 leave the reference arm at once, without work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus, workload = 5, 3, 2, "oproj_sweep"
    assert bench.run_reference(Args()) == 0
