"""Host logic of bench.py's multi-rank path on CPU: two gloo ranks, each with its own elapsed
time; every rank must see the maximum, and the job throughput counts both replicas."""
from __future__ import annotations

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank
    m = bench.max_over_ranks(ms, device="cpu")
    out[rank] = (m, bench.job_rows_per_s(4608, 100, world, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_job_value():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    m, v = res[0]
    assert m == 15.0
    assert v == pytest.approx(4608 * 100 * 2 / 0.015)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, device="cpu") == 3.5
    assert bench.job_rows_per_s(10, 2, 1, 1000.0) == pytest.approx(20.0)
