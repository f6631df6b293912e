"""Host logic of the multi-rank path on CPU (two gloo ranks): bench.py's max-over-ranks timing,
job throughput and agreement on the number of timed windows; and the row partition
(fp8_quant_row_gb300.row_pieces), whose pieces, computed rank by rank through the oracle and
gathered, must reproduce the single call's outputs bit for bit."""
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
    # the ranks' first windows differ (0.34 ms vs 0.5 ms): each wants a different number of
    # windows, and they must agree on the larger one (else one rank waits in a barrier)
    first = 0.34 if rank == 0 else 0.5
    want = bench.windows_needed(first, 10, 0.3)
    agreed = int(bench.max_over_ranks(float(want), device="cpu"))
    out[rank] = (m, bench.job_rows_per_s(4608, 100, world, m), want, agreed)
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
    assert res[0][:2] == res[1][:2]
    m, v, _, _ = res[0]
    assert m == 15.0
    assert v == pytest.approx(4608 * 100 * 2 / 0.015)
    assert res[0][2] != res[1][2], "the two ranks should want different window counts"
    assert res[0][3] == res[1][3] == max(res[0][2], res[1][2])


def test_windows_needed():
    import bench
    assert bench.windows_needed(0.34, 10, 0.3) == 883      # ceil(0.3 s / 0.34 ms)
    assert bench.windows_needed(100.0, 10, 0.3) == 10       # long windows: the repeat floor
    assert bench.windows_needed(1e-6, 10, 0.3) == 2000      # capped


def test_row_pieces_cover_every_row_once_inside_one_group():
    import fp8_quant_row_gb300 as fq
    for rows, mod_rows, world in ((9216, 4608, 8), (4608, 0, 3), (13, 5, 4), (7, 3, 7), (2, 1, 4),
                                  (0, 0, 2), (1000, 300, 6)):
        seen = []
        for rank in range(world):
            for r0, r1, g in fq.row_pieces(rows, mod_rows, world, rank):
                assert r0 < r1
                if mod_rows:
                    assert g == r0 // mod_rows == (r1 - 1) // mod_rows
                else:
                    assert g == 0
                seen.extend(range(r0, r1))
        assert seen == list(range(rows)), (rows, mod_rows, world)
    with pytest.raises(ValueError):
        fq.row_pieces(4, 0, 2, 2)


def _partition_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    import fp8_quant_row_gb300 as fq
    import oracle
    import workloads as W
    rows, cols, mod_rows, s = 13, 64, 5, 0.05
    n_mod = (rows + mod_rows - 1) // mod_rows
    inp = W.nss_inputs(rows, cols, seed=11, n_mod=n_mod)
    res = W.residual_inputs(rows, cols, seed=12, n_mod=n_mod)
    mine = []
    for r0, r1, g in fq.row_pieces(rows, mod_rows, world, rank):
        y, q = oracle.nss_fp8(inp["x"][r0:r1], inp["scale"][g:g + 1], inp["shift"][g:g + 1], s)
        ro, y2, q2 = oracle.scale_residual_nss_fp8(
            res["x"][r0:r1], res["residual"][r0:r1], res["bias"], res["gate"][g:g + 1],
            res["scale"][g:g + 1], res["shift"][g:g + 1], s)
        mine.append((r0, y, q, ro, y2, q2))
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        pieces = sorted((p for part in gathered for p in part), key=lambda p: p[0])
        cat = [np.concatenate([p[i] for p in pieces]) for i in range(1, 6)]
        y, q = oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], s, mod_rows=mod_rows)
        ro, y2, q2 = oracle.scale_residual_nss_fp8(res["x"], res["residual"], res["bias"],
                                                   res["gate"], res["scale"], res["shift"], s,
                                                   mod_rows=mod_rows)
        out["ok"] = all(np.array_equal(a, b) for a, b in zip(cat, (y, q, ro, y2, q2)))
        out["pieces"] = len(pieces)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_row_pieces_reproduce_the_single_call():
    """Rank 0 gets rows 0-6 (groups 0 and 1: two pieces), rank 1 rows 7-12 (groups 1 and 2)."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_partition_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        assert out["pieces"] == 4
        assert out["ok"], "gathered pieces differ from the single call"


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, device="cpu") == 3.5
    assert bench.job_rows_per_s(10, 2, 1, 1000.0) == pytest.approx(20.0)
