"""The benchmark's multi-GPU host logic on CPU with two gloo ranks.

Several GPUs only replicate the problem: every rank runs an independent instance with its
own seed (weak scaling), no collective touches the data path, and the job's throughput is
all ranks' work over the slowest rank's time.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.rank_workload(synth.Workload("t", 8, 16, 64, "NN", "normal_sqrtk", 1), rank)
        A_bits, _ = synth.make_inputs(w)
        local_ms = 10.0 + 5.0 * rank
        slowest = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        digests = [None] * world
        dist.all_gather_object(digests, (w.seed, A_bits.tobytes()))
        out[rank] = (slowest, digests)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        slowest, digests = out[r]
        assert slowest == 15.0
        seeds = [d[0] for d in digests]
        assert seeds == [1, 1001]
        assert digests[0][1] != digests[1][1]
    flops = 2.0 * 2048 * 2432 * 4096
    assert np.isclose(bench.job_tflops(2, flops, 10, 15.0), 2 * 10 * flops / 0.015 / 1e12)
    assert bench.max_over_ranks(3.5, None, None) == 3.5
