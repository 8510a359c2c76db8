"""The bench's multi-process path (one process per GPU, replicas with a
barrier and max-over-ranks timing) exercised with world_size 2 on the gloo
backend, on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    import bench
    os.environ["WORLD_SIZE"], os.environ["RANK"], os.environ["LOCAL_RANK"] = str(world), str(rank), str(rank)
    w, r, l = bench.dist_env()
    bench.barrier(world)
    slowest = bench.max_over_ranks(1.5 + rank, world)          # rank 1 is the slower one
    value = bench.whole_job_throughput(3.0e12, slowest, world)
    out.put((rank, w, r, l, slowest, value))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_rank_replicas_aggregate_over_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, r, l, slowest, value in results:
        assert (w, r, l) == (2, rank, rank)
        assert slowest == 2.5
        # 2 ranks x 3e12 units in 2.5 ms = 2400 (x 1e12 per second)
        assert value == pytest.approx(2.0 * 3.0e12 / 2.5e-3 / 1e12)
