"""The N>1 path on CPU: world-size-2 gloo process group, no GPU.

The training path has no exchange step; N GPUs run N independent replicas
and the benchmark reports the whole job's tokens/s over the slowest rank.
This checks that aggregation across two ranks with the gloo backend.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t_local = [0.25, 0.40][rank]  # rank 1 is the slow replica
    value, t = bench.aggregate(t_local, 8192, world, dist, "cpu")
    out[rank] = (value, t)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replica_aggregation_gloo():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            value, t = out[r]
            assert t == pytest.approx(0.40)
            assert value == pytest.approx(2 * 8192 / 0.40)


def test_single_rank_aggregation_without_group():
    import bench
    value, t = bench.aggregate(0.5, 1000, 1)
    assert (value, t) == (2000.0, 0.5)
