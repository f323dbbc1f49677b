"""The N > 1 path of the benchmark (independent replicas, one per GPU): the job's time is the
slowest rank's and the value counts every rank's windows. Two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [3.0, 5.5][rank]  # the second rank is slower
    total = bench.job_ms(local, world, "cpu")
    value = bench.us_per_window(total, 8, world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, total, value))


def test_two_replicas_take_the_slowest_rank():
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
    assert [r[1] for r in res] == [5.5, 5.5]
    # 2 ranks x 8 windows in 5.5 ms: 343.75 us per window
    assert all(abs(r[2] - 5.5e3 / 16) < 1e-9 for r in res)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_ms(4.25, 1, "cpu") == 4.25
    assert bench.us_per_window(4.25, 17, 1) == pytest.approx(4250 / 17)
