"""The multi-rank path of bench.py on CPU: two gloo ranks (127.0.0.1), each a
replica with its own step time; both must see the slowest rank's time and the
same whole-job throughput.  No GPU and no collective on the data path."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [2.5, 4.0][rank]
    ms = bench.combine_over_ranks(local, dist, "cpu")
    out[rank] = (ms, bench.job_throughput(7, world, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    ms, value = out[0]
    assert ms == 4.0
    assert abs(value - 2 * 7 / 4.0e-3) < 1e-9


def test_single_rank_is_local():
    import bench
    assert bench.combine_over_ranks(3.0, None, "cpu") == 3.0
    assert bench.job_throughput(1, 1, 2.0) == 500.0
