"""The bench's multi-rank host logic on CPU: two gloo ranks, each a replica with
its own batch; the step time is the max over ranks and the job throughput sums
the ranks' tokens.  No data-path collective exists to test."""
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
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    t = bench.max_over_ranks(1.0 + rank, world, device="cpu")   # rank 1 is the slowest
    out[rank] = t
    out[2 + rank] = bench.job_tokens_per_s(t, world)
    # replicas draw different batches (seed per rank)
    import synth
    d = synth.qdelta_inputs(1, 4, 1, 8, 8, seed=1 + rank)
    out[4 + rank] = float(d["q"].sum())
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_throughput():
    world, port = 2, _free_port()
    out = torch.zeros(6, dtype=torch.float64).share_memory_()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    import bench
    assert out[0] == out[1] == 2.0
    assert out[2] == out[3] == pytest.approx(bench.B * bench.T * 2 / 2e-3)
    assert out[4] != out[5]
