"""The bench's multi-rank path on CPU: two gloo ranks, each with its own
batch (requests are independent, no data-path collective), whole-job timing
as the maximum over ranks and token counts summed."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from gen import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times = [1.0 + rank, 10.0 - rank, 5.0 * (rank + 1)]
    w = wl.make_config(2, batch=2, seed=bench.rank_seed(2, rank), prompt_scale=0.01,
                       cache_fill="zeros")
    tokens = int(w["cu_nodes"][-1]) + rank
    got_times, got_tokens = bench.reduce_over_ranks(times, tokens, world, torch.device("cpu"))
    gathered = [None] * world
    dist.all_gather_object(gathered, (tokens, w["prompt_len"].tolist()))
    out[rank] = (got_times, got_tokens, gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_bench():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    (t0, n0, g0), (t1, n1, g1) = out[0], out[1]
    assert t0 == t1 == [2.0, 10.0, 10.0]                 # maxima over ranks
    assert n0 == n1 == sum(tok for tok, _ in g0)
    assert g0[0][1] != g0[1][1]                          # ranks verify different batches


def test_single_rank_is_identity():
    assert bench.reduce_over_ranks([1.5, 2.5], 7, 1, torch.device("cpu")) == ([1.5, 2.5], 7.0)
