"""The benchmark's multi-rank aggregation on CPU (gloo, world size 2).

The GEMM runs as independent replicas, one per rank; the only cross-rank step
is the max-over-ranks time that turns per-rank work into whole-job throughput.
"""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q) -> None:
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t, rate = bench.aggregate(1.0 + rank, 100.0, world, dist)
    q.put((rank, t, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_throughput_uses_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, t, rate in out:
        assert t == 2.0                  # slowest rank's time
        assert rate == 100.0             # (100 + 100) units / 2.0 s


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.aggregate(0.5, 10.0, 1, None) == (0.5, 20.0)
