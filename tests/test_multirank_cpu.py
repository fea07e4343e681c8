"""Host logic of bench.py's multi-GPU (replica) mode on CPU: two gloo ranks,
each with its own batch, reduce to the slowest rank's time and the sum of
all ranks' active tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from entropy_active_span_gb300 import workloads as W
    w = W.WORKLOADS["rl_16k"]
    mask = W.make_mask(w.replace(seed=w.seed + 1000 * rank))   # bench's per-rank batch
    ms_local = 10.0 + 5.0 * rank
    ms, tokens = bench.aggregate_ranks(ms_local, float(mask.sum()), "cpu")
    out[rank] = (ms, tokens, int(mask.sum()))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    ms0, tok0, own0 = out[0]
    ms1, tok1, own1 = out[1]
    assert ms0 == ms1 == 15.0                 # slowest rank
    assert tok0 == tok1 == own0 + own1        # every rank's tokens
    assert own0 != own1                       # independent batches


def test_single_process_passthrough():
    import bench
    assert bench.aggregate_ranks(3.5, 7.0, "cpu") == (3.5, 7.0)
