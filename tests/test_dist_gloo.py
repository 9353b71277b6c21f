"""The benchmark's multi-rank host logic on CPU: two gloo processes on
127.0.0.1.  Each rank times its own copy of the workload; the job's time is
the slowest rank's and its throughput counts every rank's bytes; the
reference arm runs on rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    got_ws, got_rank = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    local_ms = 10.0 * (rank + 1)                     # rank 1 is the slower one
    t_max, value = bench.aggregate(bytes_per_step=1_000_000, steps=100, local_ms=local_ms, ws=got_ws)
    # the reference arm prints on rank 0 only; other ranks return at once
    out = io.StringIO()
    if got_rank != 0:
        with contextlib.redirect_stdout(out):
            bench.run_reference(bench.parse(["--impl", "reference"]), got_ws, got_rank)
    bench.barrier(got_ws)
    q.put((got_rank, got_ws, t_max, value, out.getvalue()))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_summed_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, t_max, value, printed in res:
        assert ws == 2
        assert t_max == pytest.approx(20.0)                       # the slowest rank's time
        assert value == pytest.approx(2 * 1e6 * 100 / 20e-3 / 1e9)  # both ranks' bytes over it
        if rank == 1:
            assert printed == ""
