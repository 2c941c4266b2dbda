"""The multi-process bench path on the CPU (gloo, world size 2): every rank runs its own replica of
the workload (the layer's (batch, head) pairs are independent, so there is no data-path
collective); the ranks meet at a barrier before and after the timed region, the timing is the
maximum over ranks, and the whole-job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    mx = bench.max_over_ranks(1.0 + rank, w)
    value, ms = bench.whole_job(0.5 + rank, 100, 10, w)
    bench.barrier(w)
    q.put((r, w, mx, value, ms))
    torch.distributed.destroy_process_group()


def test_two_ranks_barrier_max_timing_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ws, mx, value, ms in res:
        assert ws == 2
        assert mx == 2.0                               # max over ranks of 1 + rank
        assert value == pytest.approx(100 * 2 * 10 / 1.5)  # both ranks' tokens over the slowest time
        assert ms == pytest.approx(1e3 * 1.5 / 10)
    assert [r[0] for r in res] == [0, 1]


def test_single_process_needs_no_collective():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.whole_job(2.0, 50, 4, 1)
    assert value == pytest.approx(50 * 4 / 2.0) and ms == pytest.approx(500.0)
