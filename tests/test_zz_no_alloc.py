"""gemm_run_noalloc against gemm_run (GPU).

gemm_run_noalloc serves callers that cannot allocate device memory (a process
that has handed all free HBM to its own pool, or a loop that cannot take the
synchronisation cudaMalloc/cudaFree may cause): it runs the small-M split-K
kernel with its scratch in a static device array instead of a plan's
workspace.  Its output must agree with the plan-based entry point within the
suite's tolerance, on two calls in a row (the second call sees the scratch as
the first one left it).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import dense_gemm_05_gb300 as g
import oracle
import workloads

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-5


@pytest.fixture(scope="module")
def plan():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    torch.cuda.set_device(0)
    p = g.Plan(0)
    yield p
    p.close()


@pytest.mark.parametrize("M,K,N,dtype,dist,seed", [
    (16, 4096, 14336, "bf16", "normal", 4),     # the M=16 decode-shaped workload's shape
    (40, 1000, 3000, "f16", "uniform", 17),     # ragged K and N, MMA N = 64
    (5, 64, 104, "bf16", "uniform", 23),        # a single K block: no split
])
def test_noalloc_matches_gemm_run_on_two_calls(plan, M, K, N, dtype, dist, seed):
    if (M, K, N) == (16, 4096, 14336):
        A, B = workloads.make_inputs("skinny16x4096x14336_bf16")
    else:
        A, B = workloads.custom(M, K, N, dtype, seed=seed, dist=dist)
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    code = g.GEMM_BF16 if dtype == "bf16" else g.GEMM_F16
    stream = torch.cuda.current_stream().cuda_stream

    c_ref = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    plan.run(a, b, c_ref)
    torch.cuda.synchronize()
    ref = c_ref.cpu().double().numpy()
    bound = oracle.absbound(A, B)

    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        st = g.gemm_run_noalloc(a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, M, N, K, code,
                                stream)
        assert st == g.GEMM_OK, g.status_string(st)
        torch.cuda.synchronize()
        got = c.cpu().double().numpy()
        ok = np.abs(got - ref) <= REL * bound + ABS
        assert ok.all(), f"call {call}: {int((~ok).sum())} entries differ from gemm_run"


def test_noalloc_rejects_sizes_beyond_its_limits(plan):
    dev = torch.device("cuda:0")
    a = torch.zeros(128, 64, dtype=torch.bfloat16, device=dev)
    c = torch.zeros(128, 64, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    U = g.GEMM_ERR_UNSUPPORTED
    # M above the limit
    assert g.gemm_run_noalloc(a.data_ptr(), 64, a.data_ptr(), 64, c.data_ptr(), 64,
                              g.GEMM_NOALLOC_MAX_M + 1, 64, 64, g.GEMM_BF16, s) == U
    # N above the limit (rejected before any pointer is touched)
    assert g.gemm_run_noalloc(a.data_ptr(), 64, a.data_ptr(), g.GEMM_NOALLOC_MAX_N + 8,
                              c.data_ptr(), g.GEMM_NOALLOC_MAX_N + 8, 16,
                              g.GEMM_NOALLOC_MAX_N + 8, 64, g.GEMM_BF16, s) == U
    # pitch that TMA cannot use
    assert g.gemm_run_noalloc(a.data_ptr(), 63, a.data_ptr(), 64, c.data_ptr(), 64, 16, 64, 63,
                              g.GEMM_BF16, s) == U
    torch.cuda.synchronize()
