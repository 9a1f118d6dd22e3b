"""Multi-rank logic of the benchmark on CPU (gloo, world size 2): the step time
is the max over ranks, the throughput counts every replica's work, and the
reference arm runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    assert bench.dist_env() == (ws, rank, rank)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    step_ms = bench.max_over_ranks(local_ms, ws)
    value = bench.whole_job_tflops(ws, 1e12, step_ms)
    # reference arm: only rank 0 prints
    args = type("A", (), {"workload": 2, "seq": 1024, "steps": 1, "warmup": 0})()
    buf = io.StringIO()
    if rank != 0:
        with redirect_stdout(buf):
            bench.reference_arm(args)
    dist.barrier()
    q.put((rank, step_ms, value, buf.getvalue()))
    dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, step_ms, value, out in res:
        assert step_ms == 15.0                       # max over ranks
        assert value == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
        if rank == 1:
            assert out == ""                         # the reference arm ran on rank 0 only
