"""The benchmark's multi-GPU host logic on CPU with two gloo ranks.

On several GPUs the job is one GEMM whose rows (of A and C) are split over the ranks, with B
replicated (output tiles are independent, so no collective touches the data path). Checked
here without a GPU: the row shards tile [0, M) in rank order; every rank's row block of A is
bit-identical to the same rows of the whole matrix and every rank holds the same B; the rows
each rank computes (the FP64 oracle stands in for the kernel) reassemble into the oracle's
full C; the job's throughput is all ranks' work over the slowest rank's time.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth
from oracle import gemm as og

BASE = synth.Workload("t", 40, 24, 64, "NN", "normal_sqrtk", 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wg = bench.sharded_workload(BASE, world)
        r0, rows = bench.m_shard(wg.M, world, rank)
        A_bits, B_bits = synth.make_row_block(wg, r0, r0 + rows)
        C_rows = og.ref_gemm(A_bits, B_bits, wg.layout)
        local_ms = 10.0 + 5.0 * rank
        slowest = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        parts = [None] * world
        dist.all_gather_object(parts, (r0, rows, A_bits.tobytes(), B_bits.tobytes(), C_rows))
        out[rank] = (slowest, parts)
    finally:
        dist.destroy_process_group()


def test_two_rank_m_split():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    wg = bench.sharded_workload(BASE, world)
    A_all, B_all = synth.make_inputs(wg)
    C_all = og.ref_gemm(A_all, B_all, wg.layout)
    for r in range(world):
        slowest, parts = out[r]
        assert slowest == 15.0
        assert [(p[0], p[1]) for p in parts] == [(0, BASE.M), (BASE.M, BASE.M)]
        for r0, rows, a, b, c in parts:
            assert a == A_all[r0:r0 + rows].tobytes()
            assert b == B_all.tobytes()
            assert np.array_equal(c, C_all[r0:r0 + rows])
    flops = 2.0 * 2048 * 2432 * 4096
    assert np.isclose(bench.job_tflops(2, flops, 10, 15.0), 2 * 10 * flops / 0.015 / 1e12)
    assert bench.max_over_ranks(3.5, None, None) == 3.5


def test_m_shard_tiles_rows():
    # Divmod split, the first M % world shards one row longer, in rank order.
    for M in range(1, 70):
        for world in range(1, 9):
            shards = [bench.m_shard(M, world, r) for r in range(world)]
            assert shards[0][0] == 0
            assert all(shards[i][0] + shards[i][1] == shards[i + 1][0] for i in range(world - 1))
            assert shards[-1][0] + shards[-1][1] == M
            assert max(s[1] for s in shards) - min(s[1] for s in shards) <= 1
    assert bench.m_shard(10, 4, 0) == (0, 3) and bench.m_shard(10, 4, 3) == (8, 2)


def test_row_blocks_match_whole_inputs():
    for w in (synth.Workload("u", 33, 8, 24, "NT", "uniform", 2),
              synth.Workload("v", 20, 8, 16, "NT", "normal", 5, zero_first_row=True, scale_last_row=4.0),
              synth.Workload("s", 48, 16, 64, "NN", "normal_sqrtk", 3)):
        A, B = synth.make_inputs(w)
        for r0, r1 in ((0, w.M), (0, 7), (5, 19), (w.M - 3, w.M), (4, 4)):
            a, b = synth.make_row_block(w, r0, r1)
            assert np.array_equal(a, A[r0:r1]) and np.array_equal(b, B)
