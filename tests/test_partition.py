"""The partitioned GEMM's host side (no GPU): gemm_partition's slices and the
all-gather of C on CPU ranks (gloo, world size 2).

A GEMM split over devices by output rows or columns ("rank offset": each
device takes different output blocks) needs no exchange to compute.  The
slices must cover the split axis exactly once, in rank order, balanced to one
128-wide unit, with boundaries that keep operand offsets 16-byte aligned; the
one collective, gathering C where every device needs all of it, must place
each rank's slice where it belongs.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import dense_gemm_05_gb300 as g


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


SHAPES = [(0, 5, 7), (1, 1, 1), (16, 14336, 4096), (64, 1000, 10), (65, 1000, 10),
          (1023, 1029, 1000), (8192, 8192, 8192), (129, 3000, 64), (5000, 17, 33)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8, 64])
@pytest.mark.parametrize("axis", [g.GEMM_SPLIT_AUTO, g.GEMM_SPLIT_M, g.GEMM_SPLIT_N])
def test_slices_cover_the_output_once(M, N, K, world, axis):
    slices = [g.gemm_partition(M, N, K, world, r, axis) for r in range(world)]
    want_axis = axis if axis != g.GEMM_SPLIT_AUTO else (g.GEMM_SPLIT_N if M <= 64 else g.GEMM_SPLIT_M)
    cover = np.zeros((M, N), dtype=np.int32) if M * N <= 4_000_000 else None
    starts, sizes = [], []
    for r, sl in enumerate(slices):
        assert (sl["axis"], sl["rank"], sl["world"]) == (want_axis, r, world)
        if want_axis == g.GEMM_SPLIT_M:
            assert (sl["col0"], sl["cols"]) == (0, N)
            starts.append(sl["row0"])
            sizes.append(sl["rows"])
        else:
            assert (sl["row0"], sl["rows"]) == (0, M)
            starts.append(sl["col0"])
            sizes.append(sl["cols"])
        if cover is not None:
            cover[sl["row0"]:sl["row0"] + sl["rows"], sl["col0"]:sl["col0"] + sl["cols"]] += 1
    extent = M if want_axis == g.GEMM_SPLIT_M else N
    # contiguous, in rank order, covering [0, extent)
    pos = 0
    for st, sz in zip(starts, sizes):
        assert st == pos and sz >= 0
        pos += sz
    assert pos == extent
    # boundaries on 128-element units, sizes within one unit of each other
    assert all(st % 128 == 0 or st == extent for st in starts)
    units = [-(-sz // 128) for sz in sizes]
    assert max(units) - min(units) <= 1
    if cover is not None:
        assert (cover == 1).all()


def test_partition_argument_errors():
    for args in [(-1, 5, 5, 2, 0, -1), (5, 5, 5, 0, 0, -1), (5, 5, 5, 2, 2, -1),
                 (5, 5, 5, 2, -1, -1), (5, 5, 5, 2, 0, 3)]:
        with pytest.raises(g.GemmError):
            g.gemm_partition(*args)
    assert g.lib().gemm_partition(5, 5, 5, 2, 0, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_run_slice(None, g.gemm_partition(5, 5, 5, 1, 0), 0, 5, 0, 5, 0, 5, 5, 5, 5,
                            g.GEMM_BF16) == g.GEMM_ERR_INVALID_ARG


# ---------------------------------------------------------------- gloo ranks

def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, M: int, N: int, K: int, axis: int, q) -> None:
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import dense_gemm_05_gb300 as gg
        import oracle
        import workloads
        A, B = workloads.custom(M, K, N, "bf16", seed=M + N + K, dist="int4")
        sl = gg.gemm_partition(M, N, K, world, rank, axis)
        # this rank's slice, computed by the oracle (the CPU stands in for a device)
        a = A[sl["row0"]:sl["row0"] + sl["rows"]]
        b = B[:, sl["col0"]:sl["col0"] + sl["cols"]]
        local = torch.from_numpy(oracle.gemm(a, b)).to(torch.float32) if sl["rows"] and sl["cols"] \
            else torch.zeros(sl["rows"], sl["cols"])
        full = gg.gather_c(local, M, N, K, axis)
        ref = oracle.gemm(A, B)
        q.put((rank, bool(np.array_equal(full.double().numpy(), ref)), sl))
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("M,N,K,axis", [(300, 200, 64, g.GEMM_SPLIT_M),
                                         (16, 700, 96, g.GEMM_SPLIT_AUTO),
                                         (130, 129, 40, g.GEMM_SPLIT_N)])
def test_gather_assembles_c_on_every_rank(M, N, K, axis):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, M, N, K, axis, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, same, sl in out:
        assert same, (rank, sl)
