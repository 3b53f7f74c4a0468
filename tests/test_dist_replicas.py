"""The multi-GPU path is independent replicas (sequences are independent; no exchange on the
hot path).  What the ranks share is the timing: every rank times its own steps, the job's time
is the slowest rank's and the throughput counts the units of all ranks.  Checked here with two
gloo ranks on the CPU."""
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


def _worker(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    ms, value = bench.aggregate(world, local_ms[rank], units_per_step=64, K=5)
    q.put((rank, ms, value))
    dist.destroy_process_group()


@pytest.mark.parametrize("local_ms", [(10.0, 12.5), (7.0, 3.0)])
def test_two_rank_timing_is_max_and_throughput_sums(local_ms):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(local_ms)
    for rank, ms, value in res:
        assert ms == slowest
        assert value == pytest.approx(2 * 64 * 5 / (slowest / 1e3))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(1, 4.0, units_per_step=1, K=8)
    assert ms == 4.0 and value == pytest.approx(2000.0)
