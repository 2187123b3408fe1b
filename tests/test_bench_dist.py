"""The bench's multi-rank host logic on CPU (gloo, world size 2).

Heads are independent, so N GPUs run N replicas: each rank compresses its own
cache (its own seed) and no collective touches the data path. The only
collectives are the bench's timing ones: the step time is the max over ranks
and the token count the sum. Those are checked here with gloo ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        ms = 1.0 + rank            # rank 1 is the slow one
        tokens = 100.0 * (rank + 1)
        bench.barrier()
        out[rank] = (bench.max_over_ranks(ms), bench.sum_over_ranks(tokens), bench.rank_seed(0, rank))
    finally:
        dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 2.0
    assert out[0][1] == out[1][1] == 300.0
    assert out[0][2] != out[1][2]   # every rank compresses its own cache


def test_single_process_reductions_are_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.sum_over_ranks(7.0) == 7.0
    assert bench.rank_seed(5, 0) == 5


def test_path_bytes_follow_the_stated_formula():
    pytest.importorskip("geometric_kv_cache_gb300")
    nb = bench.path_bytes([16384] * 32, 8, 0.5)
    heads, T, d, keep = 256, 16384, 128, 8192
    assert nb["tokens"] == heads * T
    assert nb["path"] == heads * (4 * T * d + 8 * keep * d)
    assert nb["gather"] == heads * 8 * keep * d
    assert nb["piece_sums"] == heads * 2 * T * d
    assert nb["piece_scores"] == heads * (2 * T * d + 4 * T)
    assert bench.path_bytes([16384] * 32, 8, 0.5, k_reads=1)["piece_sums"] == heads * (2 * T * d + 4 * T)
