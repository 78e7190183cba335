"""Host logic of the multi-rank bench path (replicas: one rank per GPU, no
exchange of data) on CPU with two gloo ranks: the job time is the slowest
rank's, the whole-job value counts every replica, and the reference arm
runs on rank 0 only."""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        per_rank_ms = [12.5, 20.0][rank]
        job_ms = bench.max_over_ranks(per_rank_ms, ws)
        value = bench.job_value(ws, 1e12, job_ms)
        printed = None
        if rank == 1:  # the reference arm: rank 0 alone runs and prints
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                bench.run_reference(None, None, "jagged_self")
            printed = buf.getvalue()
        q.put((rank, bench._dist(), job_ms, value, printed))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    try:
        res = {}
        for _ in range(ws):
            rank, d, job_ms, value, printed = q.get(timeout=120)
            res[rank] = (d, job_ms, value, printed)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for r in range(ws):
        d, job_ms, value, _ = res[r]
        assert d == (ws, r, r)
        assert job_ms == 20.0                     # the slowest rank's time
        assert value == pytest.approx(2 * 1e12 / 20e-3 / 1e12)  # both replicas' work
    assert res[1][3] == ""                        # rank 1 runs no reference and prints nothing


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_value(1, 2e12, 4.0) == pytest.approx(500.0)
