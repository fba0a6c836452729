"""Multi-rank host logic of the benchmark on CPU: two gloo processes take the
max of their step times, combine weak-scaling throughput, and the reference
arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 11.0][rank]
    m = bench.reduce_max(ms, "cpu")
    v = bench.replica_throughput(world, 1_000_000, m)
    out[rank] = (m, v)
    # the reference arm: ranks other than 0 return 0 without work or output
    if rank != 0:
        class A:
            workload = "decoder_1p3b"
            n_ranks = None
            steps = 1
            warmup = 0
            gpus = world
        out[10 + rank] = bench.run_reference(A())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 12.5
    assert out[0][1] == pytest.approx(2 * 1_000_000 / 0.0125)
    assert out[11] == 0
