"""The partitioned GEMM on one GPU (GPU): every rank's slice, run one after
another through gemm_run_slice on the whole matrices' layouts, must assemble C.

On one device the slices stand in for the ranks of a multi-GPU run (each rank
would run its own slice on its own device with its own copies of the operands;
the slices need no exchange).  Integer-valued inputs must match the oracle and
the unpartitioned gemm_run bit for bit; normal inputs the oracle within the
suite's tolerance.  Guard cells around C must survive.
"""
import numpy as np
import pytest
import torch

import dense_gemm_05_gb300 as g
import oracle
import workloads

pytestmark = pytest.mark.gpu

SENTINEL = 1234.5
REL, ABS = 1e-3, 1e-5


@pytest.fixture(scope="module")
def plan():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    p = g.Plan(0)
    yield p
    p.close()


def run_sliced(plan, a, b, M, N, K, world, axis, ldc):
    c = torch.full((M + 2, ldc), SENTINEL, dtype=torch.float32, device=a.device)
    for r in range(world):
        sl = g.gemm_partition(M, N, K, world, r, axis)
        plan.run_slice(a, b, c[:M, :N], sl)
    torch.cuda.synchronize()
    return c.cpu().double().numpy()


@pytest.mark.parametrize("M,K,N,world,axis", [
    (1023, 1000, 1029, 2, g.GEMM_SPLIT_M),     # the ragged workload over 2 ranks by rows
    (1023, 1000, 1029, 3, g.GEMM_SPLIT_N),     # ... over 3 by columns
    (16, 4096, 14336, 8, g.GEMM_SPLIT_AUTO),   # the M = 16 workload: columns, 1792 each
    (4096, 512, 4096, 8, g.GEMM_SPLIT_M),      # 512 rows each
    (300, 300, 3000, 64, g.GEMM_SPLIT_N),      # more ranks than units: empty slices
    (1, 64, 1, 4, g.GEMM_SPLIT_M),
])
def test_slices_assemble_c_bit_exact(plan, M, K, N, world, axis):
    A, B = workloads.custom(M, K, N, "bf16", seed=M + K + N + world, dist="int4")
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    got = run_sliced(plan, a, b, M, N, K, world, axis, ldc=N + 3)
    assert np.all(got[:M, N:] == SENTINEL) and np.all(got[M:, :] == SENTINEL)
    ref = oracle.gemm(A, B)
    assert np.array_equal(got[:M, :N], ref), f"max diff {np.abs(got[:M, :N] - ref).max()}"
    whole = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    plan.run(a, b, whole)
    torch.cuda.synchronize()
    assert np.array_equal(got[:M, :N], whole.cpu().double().numpy())


@pytest.mark.parametrize("M,K,N,world,axis", [
    (2048, 2048, 2048, 4, g.GEMM_SPLIT_M),
    (64, 8192, 5000, 3, g.GEMM_SPLIT_AUTO),
])
def test_slices_within_tolerance(plan, M, K, N, world, axis):
    A, B = workloads.custom(M, K, N, "bf16", seed=world, dist="normal")
    dev = torch.device("cuda:0")
    got = run_sliced(plan, A.to(dev), B.to(dev), M, N, K, world, axis, ldc=N)
    ref = oracle.gemm(A, B)
    bnd = oracle.absbound(A, B)
    ok = np.abs(got[:M, :N] - ref) <= REL * bnd + ABS
    assert ok.all(), f"{int((~ok).sum())} entries outside tolerance"


def test_slice_outside_the_matrix_is_rejected(plan):
    dev = torch.device("cuda:0")
    a = torch.zeros(256, 64, dtype=torch.bfloat16, device=dev)
    b = torch.zeros(64, 256, dtype=torch.bfloat16, device=dev)
    c = torch.zeros(256, 256, dtype=torch.float32, device=dev)
    bad = dict(g.gemm_partition(256, 256, 64, 2, 1, g.GEMM_SPLIT_M), rows=200)
    st = g.gemm_run_slice(plan.handle, bad, a.data_ptr(), 64, b.data_ptr(), 256, c.data_ptr(),
                          256, 256, 256, 64, g.GEMM_BF16)
    assert st == g.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
