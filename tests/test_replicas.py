"""The N > 1 path of bench.py is replicas only: each rank runs its own copy of the
workload; the job time is the slowest rank's and the throughput sums every rank's
tokens.  Checked with two gloo ranks on the CPU."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
    tokens = 1000 * (rank + 1)
    res = bench.aggregate_ranks(ms, tokens, dist, "cpu")
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_max_time_and_sums_tokens():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0] == out[1] == (15.0, 3000, 2)


def test_single_process_aggregation_is_identity():
    import bench
    assert bench.aggregate_ranks(7.5, 128, None, "cpu") == (7.5, 128, 1)
