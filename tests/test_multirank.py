"""The N>1 bench path on CPU: two gloo ranks, each timing its own replica of
the workload; the job figures are the max of the elapsed times and the sum of
the units (weak scaling, no collective in the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    elapsed = [0.5, 0.8][rank]
    units = [100.0, 300.0][rank]
    t, u = bench.aggregate(elapsed, units, world, device=None)
    out[rank] = (t, u)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_gloo():
    pytest.importorskip("torch.distributed")
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        assert out[r] == (0.8, 400.0)


def test_single_rank_aggregate_is_identity():
    import bench
    assert bench.aggregate(1.5, 10.0, 1) == (1.5, 10.0)
