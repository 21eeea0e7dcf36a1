"""The N > 1 bench path on CPU: two gloo ranks on 127.0.0.1.

Each rank decodes its own batch (a different seed, same shape: weak
scaling, no collective on the data path); the timed region's length is the
maximum over ranks.  Checked without a GPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from query_aware_sparse_kv_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        spec = bench.shard_spec(W.spec_for("tiny"), r)
        inp = W.make_inputs(spec)
        bench.barrier(w)
        t = bench.max_over_ranks(1.5 + r, w)
        results[r] = (w, r, lr, spec.seed, float(inp["q"].sum()), t)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_take_the_max_time():
    port = _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
    r0, r1 = results[0], results[1]
    assert (r0[0], r0[1]) == (2, 0) and (r1[0], r1[1]) == (2, 1)
    assert r0[3] != r1[3] and r0[4] != r1[4]  # different batches
    assert r0[5] == r1[5] == 2.5  # both see the slowest rank's time


def test_single_rank_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.0, 1) == 3.0
