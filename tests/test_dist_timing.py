"""The benchmark's multi-rank timing: every rank runs its own sequence and the
reported time is the maximum over ranks.  Exercised with two gloo ranks on CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, _ = bench.dist_env()
    assert (w, r) == (world, rank)
    local = 10.0 + 5.0 * rank          # rank 1 is the slow one
    got = bench.max_over_ranks(local)
    bench.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == 15.0 and out[1] == 15.0


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
