"""bench.py's multi-rank plumbing on CPU: two gloo ranks, no GPU.

The benchmark's N > 1 path runs one rank per GPU, each on its own batch, with
no collective on the data path; the ranks only meet at barriers around the
timed region and in a max over their times.  These tests run that plumbing
as two local processes on the gloo backend.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        t = bench.max_over_ranks(10.0 + 3.0 * r, w)      # each rank's own step time
        bench.barrier(w)
        out.put((r, local, w, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    assert [g[1] for g in got] == [0, 1]
    assert all(g[2] == world for g in got)
    assert all(g[3] == 13.0 for g in got)   # max over ranks, the same on every rank


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(4.5, 1) == 4.5
    bench.barrier(1)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        warmup, steps, ref_seconds = 3, 1, 0.1
    bench.run_reference(Args())          # rank 1: returns at once, prints nothing
    assert capsys.readouterr().out == ""
