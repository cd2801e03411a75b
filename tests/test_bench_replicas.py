"""bench.py's multi-process plumbing on CPU: two gloo ranks, the barrier and the
max-over-ranks reduction that turns per-rank times into the job's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["CUDA_VISIBLE_DEVICES"] = ""  # CPU ranks (gloo) even on a GPU machine
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench._dist()
    assert (w, r, local) == (world, rank, rank)
    bench._barrier(w)
    got = bench._max_over_ranks(float(10 * (rank + 1)), w)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_single_process_needs_no_process_group():
    import bench
    assert bench._max_over_ranks(3.5, 1) == 3.5
