"""The bench's multi-rank host logic on CPU: two gloo ranks, each an independent replica.
No GPU: the block has no data-parallel exchange, so the only cross-rank steps are the
barrier and the max-over-ranks of the timed region; whole-job throughput counts every
rank's tokens over the slowest rank's time.  The reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_setup()
        dist.barrier()
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slow replica
        slowest = bench.max_over_ranks(ms, got_ws, "cpu")
        value = bench.job_throughput(4256, 100, got_ws, slowest)
        q.put((rank, got_ws, got_rank, got_local, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_over_ranks_and_job_throughput():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, got_ws, got_rank, got_local, slowest, value in res:
        assert (got_ws, got_rank, got_local) == (2, rank, rank)
        assert slowest == 15.0                       # every rank reports the slowest replica
        # 2 ranks x 100 steps x 4256 tokens in 15 ms per step
        assert value == pytest.approx(2 * 100 * 4256 / 0.015)


def test_single_rank_is_local():
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_throughput(4256, 10, 1, 2.0) == pytest.approx(4256 * 10 / 0.002)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 0, 2
    # rank 1 returns before touching the oracle (which would take minutes at this size)
    assert bench.run_reference(Args) is None
    assert capsys.readouterr().out == ""
