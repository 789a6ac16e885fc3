"""gemm_run_noalloc (GPU): the entry point for callers that cannot allocate.

Some callers cannot allocate device memory when they multiply: a serving
process that hands all free HBM to its own memory pool at start-up has none
left for a library's workspace, and a loop that shares the GPU with other
streams cannot take the device-wide synchronisation that cudaMalloc/cudaFree
may cause.  gemm_run_noalloc runs the small-M split-K kernel with its scratch
in a static device array instead of a plan's workspace.  Its output is checked
against the fp64 oracle within the suite's tolerance -- and against the
plan-based entry point -- on two calls in a row (the second call sees the
scratch as the first one left it).  This file is collected last on purpose.
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


def _inputs(M, K, N, dtype, dist, seed):
    if (M, K, N) == (16, 4096, 14336):
        return workloads.make_inputs("skinny16x4096x14336_bf16")
    return workloads.custom(M, K, N, dtype, seed=seed, dist=dist)


def test_noalloc_setup_call_launches_nothing_and_allocates_nothing(plan):
    # A call with M = 0 only does the device set-up (loads the kernels and the
    # static array); callers that will give all free memory to their own pool
    # make it first.  After it, a real call changes no allocation.
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_run_noalloc(0, 0, 0, 0, 0, 0, 0, 0, 0, g.GEMM_BF16, s) == g.GEMM_OK
    dev = torch.device("cuda:0")
    A, B = workloads.custom(16, 512, 1024, "bf16", seed=31, dist="uniform")
    a, b = A.to(dev), B.to(dev)
    c = torch.empty(16, 1024, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert g.gemm_run_noalloc(a.data_ptr(), 512, b.data_ptr(), 1024, c.data_ptr(), 1024, 16,
                                  1024, 512, g.GEMM_BF16, s) == g.GEMM_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


@pytest.mark.parametrize("M,K,N,dtype,dist,seed", [
    (16, 4096, 14336, "bf16", "normal", 4),     # the M=16 decode-shaped workload's shape
    (40, 1000, 3000, "f16", "uniform", 17),     # ragged K and N, MMA N = 64
    (5, 64, 104, "bf16", "uniform", 23),        # a single K block: no split
    (64, 1024, 2048, "bf16", "uniform", 29),    # 16 tiles: split shares whose partials fit
])
def test_noalloc_matches_the_oracle_on_two_calls(plan, M, K, N, dtype, dist, seed):
    A, B = _inputs(M, K, N, dtype, dist, seed)
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    code = g.GEMM_BF16 if dtype == "bf16" else g.GEMM_F16
    stream = torch.cuda.current_stream().cuda_stream
    ref = oracle.gemm(A, B)
    bound = oracle.absbound(A, B)

    c_plan = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    plan.run(a, b, c_plan)
    torch.cuda.synchronize()
    via_plan = c_plan.cpu().double().numpy()

    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        st = g.gemm_run_noalloc(a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, M, N, K, code,
                                stream)
        assert st == g.GEMM_OK, g.status_string(st)
        torch.cuda.synchronize()
        got = c.cpu().double().numpy()
        ok = np.abs(got - ref) <= REL * bound + ABS
        assert ok.all(), f"call {call}: {int((~ok).sum())} entries outside the oracle tolerance"
        # and the same result as the plan-based entry point, within the same tolerance
        ok = np.abs(got - via_plan) <= REL * bound + ABS
        assert ok.all(), f"call {call}: {int((~ok).sum())} entries differ from gemm_run"


def test_noalloc_falls_back_to_whole_tiles_when_partials_do_not_fit(plan):
    # M = 64, K = 16384, N = 11520: the automatic split (270 shares over 90
    # tiles, up to 5 partial tiles each) would need about 14.7 MB of partial
    # tiles, more than the static array holds, so every tile is computed whole
    # by one CTA.  Checked on sampled entries plus every edge of C against the
    # oracle.
    M, K, N = 64, 16384, 11520
    A, B = workloads.custom(M, K, N, "bf16", seed=37, dist="uniform")
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    s = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(37)
    rows = np.concatenate([rng.integers(0, M, 2048), [0, M - 1] * 64, np.arange(M)])
    cols = np.concatenate([rng.integers(0, N, 2048), rng.integers(0, N, 128),
                           np.full(M, N - 1)])
    ref, bound = oracle.gemm_entries(A, B, rows, cols)
    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        assert g.gemm_run_noalloc(a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, M, N, K,
                                  g.GEMM_BF16, s) == g.GEMM_OK
        torch.cuda.synchronize()
        cc = c.cpu()
        assert not torch.isnan(cc).any(), "an entry of C was not written"
        got = cc.double().numpy()[rows, cols]
        ok = np.abs(got - ref) <= REL * bound + ABS
        assert ok.all(), f"call {call}: {int((~ok).sum())} sampled entries outside tolerance"


def test_noalloc_uses_every_counter_at_the_largest_n(plan):
    # N = GEMM_NOALLOC_MAX_N: 1024 column tiles, one counter each.
    M, K, N = 16, 256, g.GEMM_NOALLOC_MAX_N
    A, B = workloads.custom(M, K, N, "bf16", seed=41, dist="int4")
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    s = torch.cuda.current_stream().cuda_stream
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    assert g.gemm_run_noalloc(a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, M, N, K,
                              g.GEMM_BF16, s) == g.GEMM_OK
    torch.cuda.synchronize()
    # small-integer inputs: every sum is exact, so the result equals the oracle's bits
    np.testing.assert_array_equal(c.cpu().double().numpy(), oracle.gemm(A, B))


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
