"""The N > 1 path of bench.py on CPU: two gloo ranks (the path has no exchange
step; the ranks are independent replicas joined only by the timing
reduction), so what is tested is the host logic around them: every rank sees
the slowest rank's time, the whole-job value counts every rank's bytes, and the
reference arm runs on rank 0 only."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    import io
    import contextlib
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        local_ms = [12.5, 17.0][rank]
        tmax = bench.max_over_ranks(local_ms, "cpu")
        value = bench.job_value(1_000_000, 10, tmax, ws)
        # reference arm: rank 0 alone prints its line
        buf = io.StringIO()

        class A:
            workload = "tiny"
            steps = 1
            warmup = 0
            cpu_seconds = 0.05

        with contextlib.redirect_stdout(buf):
            bench.run_reference(A)
        q.put((rank, tmax, value, buf.getvalue()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_aggregate_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r, tmax, value, printed = q.get(timeout=300)
        res[r] = (tmax, value, printed)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 17.0                       # the slowest rank's time
    assert res[0][1] == pytest.approx(2 * 1_000_000 * 10 / 0.017 / 1e9)
    assert '"impl": "reference"' in res[0][2]                   # rank 0 prints the line
    assert res[1][2] == ""                                      # rank 1 runs nothing


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_value(2_000_000_000, 5, 1000.0, 1) == pytest.approx(10.0)
