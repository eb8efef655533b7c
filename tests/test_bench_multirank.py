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


def test_launch_and_flop_counts():
    """The counts the JSON line's gpu_launches and value are built from."""
    C4, C5 = bench.case_by_name("C4"), bench.case_by_name("C5")
    # C4 (bf16): one attention kernel; C5 (e4m3, d 128): the V widening pass and
    # the attention kernel (attn_fwd_fp8_ws); split-KV adds the combine kernel;
    # the backward pass is three kernels; d = 256 e4m3 widens on chip (one)
    assert bench.launches_per_call(C4, 1) == 1
    assert bench.launches_per_call(C5, 1) == 2
    assert bench.launches_per_call(bench.case_by_name("LKV"), 9) == 2
    assert bench.launches_per_call(bench.case_by_name("BWD"), 1) == 3
    assert bench.launches_per_call(bench.case_by_name("D256F"), 1) == 1
    # 4 B H N_q N_k d FLOPs, halved under the causal mask; the backward counts 2.5x
    assert bench.work_flops(C4) == 4 * 1 * 16 * 16384 * 16384 * 128 / 2
    assert bench.work_flops(C5) == 4 * 2 * 16 * 8192 * 8192 * 128
    bwd = bench.case_by_name("BWD")
    assert bench.work_flops(bwd) == 2.5 * 4 * 2 * 16 * 4096 * 4096 * 128 / 2
