"""bench.py's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank of a replicated run times its own steps; the job time is the
maximum over ranks and the whole-job value counts every rank's FLOPs.
Also the paper's FLOP count (FlashAttention-3, zenmind.me summary §7.1).
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [10.0 + rank, 50.0 - 7.0 * rank]
    out[rank] = bench.max_over_ranks(local, world)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [11.0, 50.0]


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.5], 1) == [3.0, 4.5]


def test_job_value_counts_every_rank():
    f = bench.fwd_flops(2, 16, 8192, 128, False) * 4.5
    one = bench.job_tflops(f, 10, 1, 100.0)
    assert bench.job_tflops(f, 10, 2, 100.0) == pytest.approx(2 * one)   # weak scaling: twice the work
    assert bench.job_tflops(f, 10, 2, 200.0) == pytest.approx(one)       # the slowest rank sets the time


def test_flop_formula_of_the_pages():
    # 4 * seqlen^2 * head_dim * heads per batch element, halved when causal
    assert bench.fwd_flops(4, 16, 8448, 128, False) == 4 * 4 * 16 * 8448 ** 2 * 128
    assert bench.fwd_flops(1, 1, 1000, 64, True) == 2 * 1000 ** 2 * 64
