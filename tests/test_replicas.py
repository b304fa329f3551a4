"""The N-replica path of the benchmark on the CPU: two gloo ranks, each with
its own time and term count, must both see the slowest rank's time and every
rank's terms (bench.job_rate, the whole-job rate of independent replicas)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, queue):
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    rate, ms = bench.job_rate(1.0 + rank, 1000 * (rank + 1), 2, "cpu")
    queue.put((rank, rate, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_all_terms():
    ctx = torch.multiprocessing.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, ms in got:
        assert ms == 2.0                                  # the slower rank's 2 ms per step
        assert rate == pytest.approx(3000 / 2e-3 / 1e9)   # 1000 + 2000 terms over that time
