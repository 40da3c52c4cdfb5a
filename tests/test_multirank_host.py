"""The benchmark's multi-rank path on CPU: world_size 2 over gloo.  Every
rank runs an independent replica (no collective on the data path); the only
exchange is the max over ranks of the timed region, and the reported value
is the bytes all ranks processed over that slowest time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [120.0, 150.0][rank]          # rank 1 is the slower replica
    ms, gbs = bench.aggregate_ranks(local_ms, 10, 2e9, world, torch.device("cpu"))
    out[rank] = (ms, gbs)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    os.environ["PYTHONPATH"] = root + os.pathsep + os.environ.get("PYTHONPATH", "")
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in (0, 1):
        ms, gbs = out[rank]
        assert ms == pytest.approx(15.0)                       # 150 ms / 10 steps, on every rank
        assert gbs == pytest.approx(2 * 2e9 / 15e-3 / 1e9)     # both replicas' bytes


def test_single_rank_aggregation_is_local():
    import bench
    ms, gbs = bench.aggregate_ranks(50.0, 5, 1e9, 1, torch.device("cpu"))
    assert ms == 10.0 and gbs == pytest.approx(100.0)
