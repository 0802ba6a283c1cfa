"""The multi-rank bench plumbing on CPU: two gloo ranks (spawned processes)
take the maximum of their per-rank step times the way bench.py does under
torchrun, and draw distinct replica seeds (rank 0 draws the published
workload's seed)."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 1.5 + 2.0 * rank                     # rank 1 is the slower one
        out[rank] = (bench.max_over_ranks(local_ms), bench.rank_seed(rank))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert out[0][0] == pytest.approx(3.5) and out[1][0] == pytest.approx(3.5)
    assert out[0][1] == 1 and out[1][1] != out[0][1]


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(2.25) == 2.25
