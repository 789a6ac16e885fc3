"""Seeded random shapes through gemm_run_ex against the fp64 oracle.

Each case draws M, N, K log-uniformly (1 .. 3000, at most 4e9 multiply-adds),
the input type, both operand layouts, the output type and a padded or tight C
pitch, then runs the automatic choice and one forced kernel that can take the
arguments (pair tiles, one-CTA tiles, the generic producer, the split-K cluster
kernel, the swap-AB stream-K kernel).  Tolerance as in test_layouts_gpu: the
task's 1e-3 * sum|A||B| + 1e-5, plus the one rounding of a 16-bit output.
Guard cells right of N and below M must survive.
"""
import numpy as np
import pytest
import torch

import dense_gemm_05_gb300 as g
import oracle
import workloads

pytestmark = pytest.mark.gpu

SENTINEL = 77.0
REL, ABS = 1e-3, 1e-5
U_OUT = {g.GEMM_OUT_F32: 0.0, g.GEMM_OUT_F16: 2.0 ** -11, g.GEMM_OUT_BF16: 2.0 ** -8}
TORCH_OUT = {g.GEMM_OUT_F32: torch.float32, g.GEMM_OUT_F16: torch.float16,
             g.GEMM_OUT_BF16: torch.bfloat16}
N_, T_ = g.GEMM_OP_N, g.GEMM_OP_T


@pytest.fixture(scope="module")
def plan():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    p = g.Plan(0)
    yield p
    p.close()


def draw(seed):
    rng = np.random.default_rng(seed)
    while True:
        M, N, K = (int(np.exp(rng.uniform(0.0, np.log(3000.0)))) for _ in range(3))
        if M * N * K <= 4e9:
            break
    if rng.random() < 0.3:                      # small M is its own family of kernels
        M = int(rng.integers(1, 65))
    dtype = "bf16" if rng.random() < 0.5 else "f16"
    op_a = T_ if rng.random() < 0.3 else N_
    op_b = T_ if rng.random() < 0.4 else N_
    out = [g.GEMM_OUT_F32, g.GEMM_OUT_F16, g.GEMM_OUT_BF16][int(rng.integers(0, 3))]
    ldc = N + int(rng.integers(0, 9)) if rng.random() < 0.5 else N
    return M, N, K, dtype, op_a, op_b, out, ldc, rng


def candidates(M, N, K, op_a):
    ks = [g.GEMM_KERNEL_PAIR, g.GEMM_KERNEL_TMA, g.GEMM_KERNEL_GENERIC]
    if op_a == N_ and K >= 128:
        ks.append(g.GEMM_KERNEL_SPLIT_PAIR)
    if op_a == N_ and M <= 64:
        ks.append(g.GEMM_KERNEL_SKINNY)
    return ks


def run(plan, A_st, B_st, op_a, op_b, M, N, K, out, ldc, kernel):
    dev = torch.device("cuda:0")
    a, b = A_st.to(dev), B_st.to(dev)
    # row pitch of the stored operands (torch reports any stride for a dimension of size 1)
    lda, ldb = max(a.stride(0), a.size(1)), max(b.stride(0), b.size(1))
    cbuf = torch.full((M + 2, ldc), SENTINEL, dtype=TORCH_OUT[out], device=dev)
    plan.force(kernel, 0, 0)
    try:
        dt = g.GEMM_BF16 if a.dtype == torch.bfloat16 else g.GEMM_F16
        cfg = g.gemm_query_ex(plan.handle, op_a, op_b, a.data_ptr(), lda, b.data_ptr(), ldb,
                              cbuf.data_ptr(), ldc, out, M, N, K, dt)
        st = g.gemm_run_ex(plan.handle, op_a, op_b, a.data_ptr(), lda, b.data_ptr(), ldb,
                           cbuf.data_ptr(), ldc, out, M, N, K, dt,
                           torch.cuda.current_stream().cuda_stream)
        assert st == g.GEMM_OK, g.status_string(st)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
    return cfg, cbuf.float().cpu().double().numpy()


@pytest.mark.parametrize("seed", range(200))
def test_random_shape(plan, seed):
    M, N, K, dtype, op_a, op_b, out, ldc, rng = draw(1000 + seed)
    A, B = workloads.custom(M, K, N, dtype, seed=seed, dist="normal")
    A_st = A.contiguous() if op_a == N_ else A.t().contiguous()
    B_st = B.contiguous() if op_b == N_ else B.t().contiguous()
    ref = oracle.gemm(A, B)
    bnd = oracle.absbound(A, B)
    tol = REL * bnd + ABS + U_OUT[out] * (np.abs(ref) + REL * bnd)
    ks = candidates(M, N, K, op_a)
    for kernel in (0, ks[int(rng.integers(0, len(ks)))]):
        try:
            cfg, got = run(plan, A_st, B_st, op_a, op_b, M, N, K, out, ldc, kernel)
        except g.GemmError as e:
            # a forced kernel may refuse arguments it cannot take (e.g. two unaligned
            # operands too large for the staging buffer); the automatic choice never may
            assert kernel != 0 and e.status == g.GEMM_ERR_UNSUPPORTED, str(e)
            continue
        what = (f"seed {seed}: {M}x{N}x{K} {dtype} ops {op_a}{op_b} out {out} ldc {ldc} "
                f"forced {kernel} ran {cfg['kernel_name']}")
        assert np.all(got[:M, N:] == SENTINEL) and np.all(got[M:] == SENTINEL), what + ": guards"
        err = np.abs(got[:M, :N] - ref)
        bad = err > tol
        assert not bad.any(), f"{what}: {int(bad.sum())} entries outside tolerance"
