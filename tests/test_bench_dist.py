"""bench.py's multi-rank logic on CPU (gloo, world size 2).

Under torchrun every rank drafts its own batch (weak scaling, no exchange of
data); the only collective is the host-side maximum of the ranks' step times.
These tests run that logic in two CPU processes over gloo on 127.0.0.1.
"""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    d = bench.dist_init(w, "gloo")
    try:
        bench.barrier(d)
        step_ms = [3.0, 5.0][rank]                 # rank 1 is the slower one
        out[rank] = bench.max_over_ranks(step_ms, d)
        out[2 + rank] = bench.rank_seed(2, rank)
        bench.barrier(d)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank_seeds_on_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Array("d", 4)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert list(out[:2]) == [5.0, 5.0]           # every rank sees the slowest rank's time
    assert out[2] != out[3]                       # each rank drafts its own batch


def test_single_rank_needs_no_process_group():
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(7.5, None) == 7.5
