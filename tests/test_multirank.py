"""The N > 1 host logic of bench.py on CPU with the gloo backend (world
size 2): every rank runs its own replica of the step (the path shards by
rows, no data-path collective), timing is the max over ranks and the
reported value aggregates all ranks' work."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 2.0 + rank            # rank 1 is the slow one
        got = bench.reduce_max_over_ranks(local_ms, world)
        value = bench.aggregate_value(1e12, world, got)
        queue.put((rank, got, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_is_max_and_value_is_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in results:
        assert got == 3.0                      # max over ranks
        assert value == pytest.approx(2 * 1e12 / 3e-3 / 1e12)   # both ranks' FLOPs / slowest time


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_over_ranks(1.5, 1) == 1.5
    assert bench.aggregate_value(2e12, 1, 1.0) == pytest.approx(2000.0)
