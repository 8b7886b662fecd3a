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
    # each rank sizes its batches from its own estimate; all time the same count
    nb = bench.uniform_count(bench.batches_for(1e-3 * (rank + 1), 20, min_timed_s=2.0))
    ks = bench.uniform_count(bench.steps_for(10e-6 * (rank + 1), 20))
    q.put((rank, thr, tmax, mx, nb, ks))
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
    import bench

    want_nb = max(bench.batches_for(1e-3 * (r + 1), 20, min_timed_s=2.0) for r in range(world))
    want_ks = max(bench.steps_for(10e-6 * (r + 1), 20) for r in range(world))
    for rank, thr, tmax, mx, nb, ks in res:
        assert tmax == pytest.approx(slowest)
        assert thr == pytest.approx(total_units / slowest)
        assert mx == 10.0 * (world - 1)
        assert (nb, ks) == (want_nb, want_ks)


def test_single_rank_is_identity():
    import bench

    assert bench.reduce_max(3.5) == 3.5
    thr, t = bench.aggregate_throughput(6.0, 2.0)
    assert (thr, t) == (3.0, 2.0)


def test_batch_and_step_counts():
    import bench

    assert bench.batches_for(1e-3, 20) == 25          # 0.5 s of 20 ms batches
    assert bench.batches_for(1.0, 20) == 7            # at least 7 batches
    assert bench.batches_for(1e-9, 20) == 400         # at most 400
    assert bench.steps_for(10e-6, 20) == 200          # about 2 ms per batch
    assert bench.steps_for(1e-3, 20) == 20            # at least K_min
    assert bench.steps_for(1e-9, 20) == 2000          # at most K_max
