"""The multi-GPU host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

With N GPUs every rank runs its own batch of the workload (the (b, h) problems
are independent: no data-path collective); the only collectives are the barrier
and the max over ranks of the measured time, and rank 0 reports the job's
tokens (weak scaling).  These tests run those steps with two CPU processes.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from mamba_ssd_chunked_02_gb300 import workloads as W

TINY = W.Workload("r b1 T64 H2 P8 N8 G1 L16 f32", 1, 64, 2, 8, 8, 1, 16, dtype="f32", seed=77)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.rank_workload(TINY, rank)
        inp = W.make_inputs(w)
        y, f = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)      # this rank's own problem
        # every rank's inputs and outputs differ: no two ranks compute the same batch
        sums = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, torch.tensor([float(inp["x"].double().sum()), float(np.sum(y))],
                                           dtype=torch.float64))
        t_local = 1.0 + rank                                        # ms, a stand-in timing
        t_job = bench.max_over_ranks(t_local, dist, "cpu")
        dist.barrier()
        out[rank] = (float(sums[0][0]), float(sums[1][0]), float(sums[0][1]), float(sums[1][1]),
                     t_job, bench.job_tokens(w, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_independent_batches_and_report_the_slowest():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        r0, r1 = out[0], out[1]
    assert r0[0] != r0[1] and r0[2] != r0[3]           # distinct inputs and outputs per rank
    assert r0[:4] == r1[:4]                             # both ranks saw the same gathered values
    assert r0[4] == r1[4] == 2.0                        # job time = the slowest rank's
    assert r0[5] == r1[5] == 2 * TINY.tokens            # weak scaling: tokens of both ranks


def test_single_process_helpers():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.rank_workload(TINY, 0) == TINY
    assert bench.rank_workload(TINY, 3).seed == TINY.seed + 3
    assert bench.job_tokens(TINY, 4) == 4 * TINY.tokens
