"""The bench's multi-replica bookkeeping on CPU: two gloo ranks (the path runs one independent replica
per GPU with no collective on the data path; only the timing is reduced, max over ranks)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [5.25, 7.5][rank]           # the second replica is the slower one
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        gbs, pos = bench.job_rates(14227333120, 5, ms, world)
        out.put((rank, ms, gbs, pos))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
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
    for rank, ms, gbs, pos in res:
        assert ms == 7.5
        assert gbs == pytest.approx(2 * 14227333120 / 7.5e-3 / 1e9)
        assert pos == pytest.approx(2 * 5 / 7.5e-3)


def test_one_replica_needs_no_process_group():
    assert bench.max_over_ranks(3.0, None, "cpu") == 3.0
    gbs, pos = bench.job_rates(1e9, 5, 2.0, 1)
    assert gbs == pytest.approx(500.0) and pos == pytest.approx(2500.0)
