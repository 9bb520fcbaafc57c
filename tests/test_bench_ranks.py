"""bench.py's multi-rank path (N independent replicas, no collective on the
data path): the step time reported is the slowest rank's, and the value is
the work of all ranks over that time.  Runs two gloo ranks on the CPU."""

import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]                     # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms)          # CPU tensor under gloo
        value = bench.aggregate_throughput(2.0e12, ms_max / 1e3, world)
        bench.barrier()
        q.put((rank, ms_max, value, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value, env in out:
        assert ms_max == 5.0                      # max over ranks
        assert abs(value - 2 * 2.0e12 / 5e-3) < 1  # all ranks' work / slowest time
        assert env[0] == rank and env[1] == 2


def test_single_process_is_identity():
    assert bench.max_over_ranks(4.5) == 4.5
    assert bench.aggregate_throughput(1.0e12, 0.5, 1) == 2.0e12
