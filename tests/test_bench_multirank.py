"""The benchmark's multi-rank host logic on CPU with the gloo backend,
world size 2: replicas report their own time, the job takes the slowest
rank's, and the whole-job rate counts every rank's parameters."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 100.0 + 25.0 * rank                     # rank 1 is the slow one
    got = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    rate = bench.whole_job_rate(world, 1000, 4, got)
    out[rank] = (got, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 125.0
    assert res[0][1] == pytest.approx(2 * 1000 * 4 / 0.125)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.whole_job_rate(1, 10, 2, 1000.0) == 20.0
