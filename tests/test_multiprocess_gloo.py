"""The multi-rank host path of bench.py on CPU: two gloo ranks, barrier, and the
max-over-ranks time that sets the whole-job throughput."""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    t = bench.dist_max(1.5 + rank, w)  # each rank's own time; the slowest one counts
    out[rank] = t
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.dist_max(3.0, 1) == 3.0
    bench.barrier(1)
