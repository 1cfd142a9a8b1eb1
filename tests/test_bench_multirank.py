"""The multi-rank path of bench.py on CPU with the gloo backend (world size 2).

On GPUs every rank runs its own replica of the workload (heads are
independent problems; there is no data-path collective); the ranks meet only
for the barrier and for the max-over-ranks step time.  These tests run that
host logic in two spawned processes.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from tests.conftest import ROOT  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.5][rank]  # rank 1 is the slow one
    dist.barrier()
    got = bench.dist_max(ms, dist)
    value = bench.weak_scaling_value(1e12, world, got)
    out.put((rank, got, value))
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
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
    assert [r[1] for r in res] == [5.5, 5.5]  # every rank sees the slowest rank's time
    # two replicas of 1e12 flop each in 5.5 ms
    assert all(abs(r[2] - 2e12 / 5.5e-3 / 1e12) < 1e-9 for r in res)


def test_single_process_helpers():
    import bench
    assert bench.dist_max(2.5) == 2.5
    assert abs(bench.weak_scaling_value(4e12, 1, 2.0) - 2000.0) < 1e-9
    assert abs(bench.weak_scaling_value(4e12, 8, 2.0) - 16000.0) < 1e-9
