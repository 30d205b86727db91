"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank
runs an independent batch (weak scaling); the whole-job value is every
rank's bytes over the slowest rank's time."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    # rank r: (r + 1) seconds for 10 * (r + 1) GB
    value, tmax, total = bench.aggregate(float(rank + 1), 10.0 * (rank + 1), w)
    bench.barrier(w)
    q.put((rank, value, tmax, total))
    dist.destroy_process_group()


def test_weak_scaling_aggregate_two_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, tmax, total in results:
        assert tmax == 2.0 and total == 30.0 and abs(value - 15.0) < 1e-12


def test_single_rank_aggregate():
    import bench
    assert bench.aggregate(2.0, 10.0, 1) == (5.0, 2.0, 10.0)
