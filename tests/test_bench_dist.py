"""The multi-rank host logic of bench.py on CPU: two gloo ranks (one process
each, 127.0.0.1 rendezvous) take the max of their timings and report the
whole-job throughput of both replicas."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.dist_barrier(world)
    ms_local = [40.0, 50.0][rank]          # rank 1 is the slower one
    ms_step, value = bench.aggregate_throughput(10**9, ms_local, 10, world)
    bench.dist_barrier(world)
    dist.destroy_process_group()
    q.put((rank, ms_step, value))


def test_two_gloo_ranks_report_whole_job_throughput_at_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms_step, value in out:
        assert ms_step == pytest.approx(5.0)                      # max(40, 50) ms / 10 steps
        assert value == pytest.approx(2 * 10**9 / 5e-3 / 1e9)     # both replicas' bytes
