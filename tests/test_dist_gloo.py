"""The N > 1 path of bench.py ("replicas only": every rank runs the whole
workload on its own GPU) on CPU ranks with the gloo backend: whole-job
throughput is all ranks' work over the slowest rank's time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench

    ws, r = bench.init_dist("gloo")
    assert (ws, r) == (world, rank)
    bench.barrier()
    # rank r did (r + 1) units in (r + 1) * 0.5 seconds
    thr, tmax = bench.aggregate_throughput(float(rank + 1), (rank + 1) * 0.5)
    mx = bench.reduce_max(float(10 * rank))
    q.put((rank, thr, tmax, mx))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_aggregation_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    total_units = sum(r + 1 for r in range(world))
    slowest = world * 0.5
    for rank, thr, tmax, mx in res:
        assert tmax == pytest.approx(slowest)
        assert thr == pytest.approx(total_units / slowest)
        assert mx == 10.0 * (world - 1)


def test_single_rank_is_identity():
    import bench

    assert bench.reduce_max(3.5) == 3.5
    thr, t = bench.aggregate_throughput(6.0, 2.0)
    assert (thr, t) == (3.0, 2.0)
