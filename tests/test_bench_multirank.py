"""The benchmark's multi-rank logic on the CPU with two gloo ranks.

One process per GPU is how bench.py runs under torchrun; the path shards by
(batch, head) with no data-path collective, so the only cross-rank steps are
the barrier, the max-over-ranks of the timed region and the whole-job
aggregate.  These run here with the gloo backend on two CPU processes.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synthetic


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.0, 30.0][rank]                   # rank 1 is the slow one
        m = bench.max_over_ranks(torch, dist, ms, "cpu")
        dist.barrier()
        # each rank's shard differs; every rank uses the same case shape
        case = synthetic.CASES["C1"]
        seed = bench.shard_seed(case.seed, rank)
        q = synthetic.make_inputs(synthetic.custom_case(1, 1, 8, 8, 64, False, seed=seed))["q"]
        digest = torch.tensor([float(q.float().sum())])
        gathered = [torch.zeros(1) for _ in range(world)]
        dist.all_gather(gathered, digest)
        out[rank] = (m, bench.job_tflops(1e12, 10, world, m), [float(g) for g in gathered])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_aggregate():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    for rank in range(world):
        m, tflops, digests = out[rank]
        assert m == 30.0                          # max over ranks
        assert tflops == pytest.approx(2 * 1e12 * 10 / 0.030 / 1e12)
        assert digests[0] != digests[1]           # different shards per rank


def test_single_rank_helpers_without_a_process_group():
    assert bench.max_over_ranks(torch, dist, 5.0, "cpu") == 5.0
    assert bench.job_tflops(2e12, 4, 1, 8.0) == pytest.approx(1000.0)
    assert bench.shard_seed(1004, 0) == 1004 and bench.shard_seed(1004, 3) == 1304
