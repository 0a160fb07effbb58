"""The host logic of a several-GPU run, on CPU with two gloo ranks: each rank
is an independent replica (own pool, own batch), the timed region reports the
slowest rank and the aggregate rate counts every rank's work.  The update
itself has no exchange step, so there is no collective on the data path."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    # every rank builds its own replica of the workload, seeded by its rank
    w = workloads.random_problem(100 + rank, kind="onetoken", slots=16, heads=2, dim=4, dstate=16,
                                 groups=1, nseq=4)
    slowest = bench.max_over_ranks(10.0 + rank, torch.device("cpu"))
    rate = bench.aggregate_rate(w.rows, world, 5, slowest)
    first_x = float(w.x.float()[0, 0, 0])
    gathered = [None] * world
    dist.all_gather_object(gathered, first_x)
    out[rank] = (slowest, rate, gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # no fork of a process that may hold threads
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, rate, xs = res[rank]
        assert slowest == 11.0                      # max over ranks
        assert rate == pytest.approx(4 * 2 * 5 / 11.0e-3)
        assert xs[0] != xs[1]                       # replicas are seeded independently
