"""CPU, world size 2 over gloo: the bench's multi-rank timing takes the slowest rank and sums
the replicas' work (the forward itself needs no exchange between GPUs)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        local_ms = 100.0 if rank == 0 else 250.0      # rank 1 is the slow one
        value, elapsed = bench.aggregate_tflops(1e12, 4, local_ms, ws)
        q.put((rank, value, elapsed))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, value, elapsed in got:
        assert elapsed == pytest.approx(250.0)
        # 2 ranks × 1e12 FLOP × 4 steps in 0.25 s = 32 TFLOP/s
        assert value == pytest.approx(32.0)


def test_single_rank_aggregate_is_plain():
    import bench
    value, elapsed = bench.aggregate_tflops(2e12, 5, 1000.0, 1)
    assert elapsed == 1000.0 and value == pytest.approx(10.0)
