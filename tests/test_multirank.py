"""The benchmark's multi-rank timing on CPU: two gloo ranks, max over ranks,
whole-job rate = units of all ranks / slowest rank's time."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + rank)            # rank 1 is the slow one
        q.put((rank, t, bench.whole_job_rate(100.0, world, t)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [11.0, 11.0]
    assert all(abs(g[2] - 200.0 / 11.0) < 1e-12 for g in got)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
