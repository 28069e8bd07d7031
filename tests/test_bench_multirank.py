"""Host logic of bench.py's multi-rank path, on CPU with gloo ranks: the
step time is the slowest rank's, the value aggregates every rank's bytes,
and the reference arm does its work on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        q.put((rank, ms, bench.whole_job_gbs(1_000_000_000, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    # spawned ranks import torch first, which takes a while on a loaded host
    for p in procs:
        p.join(timeout=600)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.terminate()
        p.join(timeout=30)
    assert not alive, "a gloo rank did not finish"
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=60) for _ in range(world))
    for rank, ms, gbs in got:
        assert ms == 2.5                          # slowest rank's time on every rank
        assert gbs == pytest.approx(2 * 1e9 / 2.5e-3 / 1e9)


def test_single_rank_passthrough():
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.whole_job_gbs(6_700_000_000, 1, 1.0) == pytest.approx(6700.0)


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 3, 3, 2

    assert bench.run_reference(A()) == 0      # returns before touching the workload
