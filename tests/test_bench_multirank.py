"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, the timed region's max
over ranks and the whole-job tokens/s (replicas, weak scaling).  No GPU involved."""
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


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [0.25, 0.75][rank]            # seconds each rank spent in the timed steps
    dist.barrier()
    m = bench.max_over_ranks(local, dist)
    q.put((rank, m, bench.job_tokens_per_s(1024, 20, world, m)))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [0.75, 0.75]
    assert res[0][2] == pytest.approx(1024 * 20 * 2 / 0.75)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, None) == 1.5
    assert bench.job_tokens_per_s(64, 10, 1, 0.5) == 1280
