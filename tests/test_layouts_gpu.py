"""GPU parity of gemm_run_ex: transposed operand storage and fp16/bf16 output.

The oracle always sees the logical operands: a transposed stored operand is
turned back into its logical M x K / K x N matrix on the CPU (a transpose moves
the 16-bit values without changing them) before the fp64 product.

Tolerance.  fp32 output: the suite's |C - C_ref| <= 1e-3 * sum|A||B| + 1e-5.
fp16 / bf16 output adds the one rounding of the fp32 accumulator to the output
type (round-to-nearest-even: relative error at most u = 2^-11 for fp16 and
2^-8 for bf16), i.e. + u * (|C_ref| + 1e-3 * sum|A||B|).  Integer inputs with
|C| <= 256 are exact in every output type and must match bit for bit.
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


def stored(A_logical, op):
    """Row-major storage of a logical operand for the given op."""
    return A_logical.contiguous() if op == N_ else A_logical.t().contiguous()


def run_ex(plan, A_st, B_st, op_a, op_b, M, N, K, out, kernel=0, ldc=None, expect=None):
    dev = torch.device("cuda:0")
    a, b = A_st.to(dev), B_st.to(dev)
    ldc = N if ldc is None else ldc
    cbuf = torch.full((M + 2, ldc), SENTINEL, dtype=TORCH_OUT[out], device=dev)
    plan.force(kernel, 0, 0)
    try:
        if expect is not None:
            cfg = g.gemm_query_ex(plan.handle, op_a, op_b, a.data_ptr(), a.stride(0),
                                  b.data_ptr(), b.stride(0), cbuf.data_ptr(), ldc, out, M, N, K,
                                  g.GEMM_BF16 if a.dtype == torch.bfloat16 else g.GEMM_F16)
            assert cfg["kernel"] == expect, cfg
        st = g.gemm_run_ex(plan.handle, op_a, op_b, a.data_ptr(), a.stride(0), b.data_ptr(),
                           b.stride(0), cbuf.data_ptr(), ldc, out, M, N, K,
                           g.GEMM_BF16 if a.dtype == torch.bfloat16 else g.GEMM_F16,
                           torch.cuda.current_stream().cuda_stream)
        assert st == g.GEMM_OK, g.status_string(st)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
    return cbuf.float().cpu().double().numpy()


def check(got, A, B, M, N, out, what):
    assert np.all(got[:M, N:] == SENTINEL) and np.all(got[M:] == SENTINEL), f"{what}: guard cells"
    ref = oracle.gemm(A, B)
    bnd = oracle.absbound(A, B)
    tol = REL * bnd + ABS + U_OUT[out] * (np.abs(ref) + REL * bnd)
    err = np.abs(got[:M, :N] - ref)
    assert np.all(err <= tol), f"{what}: {int((err > tol).sum())} entries outside tolerance"


KERNELS = [g.GEMM_KERNEL_PAIR, g.GEMM_KERNEL_TMA, g.GEMM_KERNEL_GENERIC]
OPS = [(N_, N_), (N_, T_), (T_, N_), (T_, T_)]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("op_a,op_b", OPS)
def test_operand_layouts(plan, kernel, op_a, op_b):
    M, K, N = 328, 200, 264          # ragged against every tile; 16-byte pitches either way
    A, B = workloads.custom(M, K, N, "bf16", seed=31 + 2 * op_a + op_b, dist="normal")
    got = run_ex(plan, stored(A, op_a), stored(B, op_b), op_a, op_b, M, N, K, g.GEMM_OUT_F32,
                 kernel=kernel, ldc=N + 8, expect=kernel)
    check(got, A, B, M, N, g.GEMM_OUT_F32, f"kernel {kernel} ops {op_a}{op_b}")


@pytest.mark.parametrize("op_b", [N_, T_])
@pytest.mark.parametrize("kernel,shares,block_n", [(g.GEMM_KERNEL_SKINNY, 0, 0),
                                                   (g.GEMM_KERNEL_SKINNY, 7, 0),
                                                   (g.GEMM_KERNEL_SPLIT_PAIR, 0, 128),
                                                   (g.GEMM_KERNEL_SPLIT_PAIR, 0, 192),
                                                   (g.GEMM_KERNEL_SPLIT_PAIR, 0, 256)])
def test_skinny_weight_layout(plan, op_b, kernel, shares, block_n):
    """M <= 64 with B stored N x K (the weight layout): swap-AB reads it K-major,
    the cluster kernel as a K-major MMA B operand."""
    M, K, N = 40, 520, 392
    A, B = workloads.custom(M, K, N, "f16", seed=5 + op_b, dist="normal")
    dev = torch.device("cuda:0")
    a, b = A.to(dev), stored(B, op_b).to(dev)
    c = torch.full((M + 2, N), SENTINEL, dtype=torch.float32, device=dev)
    plan.force(kernel, shares, block_n)
    try:
        st = g.gemm_run_ex(plan.handle, N_, op_b, a.data_ptr(), K, b.data_ptr(), b.stride(0),
                           c.data_ptr(), N, g.GEMM_OUT_F32, M, N, K, g.GEMM_F16,
                           torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
    assert st == g.GEMM_OK, g.status_string(st)
    check(c.cpu().double().numpy(), A, B, M, N, g.GEMM_OUT_F32, f"skinny op_b {op_b}")


@pytest.mark.parametrize("out", [g.GEMM_OUT_F16, g.GEMM_OUT_BF16])
@pytest.mark.parametrize("kernel,shape", [(g.GEMM_KERNEL_PAIR, (600, 320, 520)),
                                          (g.GEMM_KERNEL_TMA, (300, 256, 264)),
                                          (g.GEMM_KERNEL_GENERIC, (130, 96, 72)),
                                          (g.GEMM_KERNEL_SKINNY, (16, 1024, 1000)),
                                          (g.GEMM_KERNEL_SPLIT_PAIR, (16, 1024, 1000)),
                                          (g.GEMM_KERNEL_SPLIT_PAIR, (300, 1024, 520))])
def test_16bit_outputs(plan, out, kernel, shape):
    M, K, N = shape
    A, B = workloads.custom(M, K, N, "bf16", seed=M + out, dist="normal")
    got = run_ex(plan, A, B, N_, N_, M, N, K, out, kernel=kernel, ldc=N + 8, expect=kernel)
    check(got, A, B, M, N, out, f"kernel {kernel} out {out}")


@pytest.mark.parametrize("out", [g.GEMM_OUT_F32, g.GEMM_OUT_F16, g.GEMM_OUT_BF16])
@pytest.mark.parametrize("op_a,op_b", OPS)
def test_integer_exact_every_layout_and_output(plan, out, op_a, op_b):
    M, K, N = 264, 16, 200           # |C| <= 16 * 16 = 256: exact in fp16 and bf16
    gen = torch.Generator().manual_seed(3 * out + 2 * op_a + op_b)
    A = torch.randint(-4, 5, (M, K), generator=gen).to(torch.bfloat16)
    B = torch.randint(-4, 5, (K, N), generator=gen).to(torch.bfloat16)
    ref = oracle.gemm(A, B)
    for kernel in (g.GEMM_KERNEL_TMA, g.GEMM_KERNEL_PAIR, g.GEMM_KERNEL_GENERIC):
        got = run_ex(plan, stored(A, op_a), stored(B, op_b), op_a, op_b, M, N, K, out,
                     kernel=kernel)
        assert np.array_equal(got[:M, :N], ref), f"kernel {kernel}"


@pytest.mark.parametrize("out", [g.GEMM_OUT_F32, g.GEMM_OUT_F16, g.GEMM_OUT_BF16])
@pytest.mark.parametrize("op_a,op_b", [(N_, N_), (T_, T_)])
@pytest.mark.parametrize("M,K,N", [(2048, 2048, 5120), (2560, 2048, 4864)])
def test_pair_stream_k_layouts_and_outputs(plan, out, op_a, op_b, M, K, N):
    """Pair tiles with a stream-K phase (160 tiles of 256 columns, two shares per
    split tile; 190 tiles, 2-3 shares per split tile): the fix-up
    writes every output type and reads every operand layout.  Integer inputs:
    the fp32 sums stay below 2^24 and are exact, so each output is the oracle's
    value rounded once (to nearest even) to the output type."""
    gen = torch.Generator().manual_seed(91)
    A = torch.randint(-4, 5, (M, K), generator=gen).to(torch.bfloat16)
    B = torch.randint(-4, 5, (K, N), generator=gen).to(torch.bfloat16)
    got = run_ex(plan, stored(A, op_a), stored(B, op_b), op_a, op_b, M, N, K, out,
                 kernel=g.GEMM_KERNEL_PAIR, expect=g.GEMM_KERNEL_PAIR)
    assert np.all(got[M:] == SENTINEL)
    ref = torch.from_numpy(oracle.gemm(A, B)).float().to(TORCH_OUT[out]).double().numpy()
    assert np.array_equal(got[:M, :N], ref)


def test_matmul_accepts_transposed_views(plan):
    """Plan.matmul on torch views: x @ w.t() with w stored [out, in] (a linear layer)."""
    M, K, N = 256, 512, 384
    X, Wt = workloads.custom(M, K, N, "bf16", seed=8, dist="normal")   # Wt is K x N
    W = Wt.t().contiguous()                                             # stored N x K
    dev = torch.device("cuda:0")
    x, w = X.to(dev), W.to(dev)
    c = plan.matmul(x, w.t())
    torch.cuda.synchronize()
    ref = oracle.gemm(X, Wt)
    bnd = oracle.absbound(X, Wt)
    assert np.all(np.abs(c.cpu().double().numpy() - ref) <= REL * bnd + ABS)
    c16 = plan.matmul(x, w.t(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    err = np.abs(c16.float().cpu().double().numpy() - ref)
    assert np.all(err <= REL * bnd + ABS + 2.0 ** -8 * (np.abs(ref) + REL * bnd))


def test_layout_argument_errors(plan):
    dev = torch.device("cuda:0")
    a = torch.ones(64, 64, dtype=torch.bfloat16, device=dev)
    c = torch.empty(64, 64, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    h = plan.handle
    E, U = g.GEMM_ERR_INVALID_ARG, g.GEMM_ERR_UNSUPPORTED
    # op T for A needs lda >= M
    assert g.gemm_run_ex(h, T_, N_, a.data_ptr(), 63, a.data_ptr(), 64, c.data_ptr(), 64,
                         g.GEMM_OUT_F32, 64, 64, 32, g.GEMM_BF16, s) == E
    # op T for B needs ldb >= K
    assert g.gemm_run_ex(h, N_, T_, a.data_ptr(), 64, a.data_ptr(), 31, c.data_ptr(), 64,
                         g.GEMM_OUT_F32, 64, 64, 32, g.GEMM_BF16, s) == E
    assert g.gemm_run_ex(h, 2, N_, a.data_ptr(), 64, a.data_ptr(), 64, c.data_ptr(), 64,
                         g.GEMM_OUT_F32, 64, 64, 64, g.GEMM_BF16, s) == E
    assert g.gemm_run_ex(h, N_, N_, a.data_ptr(), 64, a.data_ptr(), 64, c.data_ptr(), 64,
                         9, 64, 64, 64, g.GEMM_BF16, s) == U
    # a 16-bit C must be 2-byte aligned
    assert g.gemm_run_ex(h, N_, N_, a.data_ptr(), 64, a.data_ptr(), 64, c.data_ptr() + 1, 64,
                         g.GEMM_OUT_F16, 64, 64, 64, g.GEMM_BF16, s) == E
    torch.cuda.synchronize()


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("out", [g.GEMM_OUT_F32, g.GEMM_OUT_F16, g.GEMM_OUT_BF16])
@pytest.mark.parametrize("M,K,N,ldc_pad", [(256, 256, 256, 0), (200, 136, 72, 8), (96, 128, 136, 8),
                                           (184, 64, 248, 0)])
def test_64_row_tiles_every_layout_and_output(plan, op_a, op_b, out, M, K, N, ldc_pad):
    """Small problems run on 64 x 64 tiles with M = 64 MMAs (16 accumulator rows
    per epilogue warp): integer inputs, exact in every output type, ragged edges
    and guard cells, every operand layout.  The planner must pick those tiles."""
    gen = torch.Generator().manual_seed(M + N + 3 * op_a + op_b + 7 * out)
    A = torch.randint(-1, 2, (M, K), generator=gen).to(torch.float16)   # |C| <= K <= 256: exact
    B = torch.randint(-1, 2, (K, N), generator=gen).to(torch.float16)   # in fp16 and bf16 too
    dev = torch.device("cuda:0")
    a, b = stored(A, op_a).to(dev), stored(B, op_b).to(dev)
    ldc = N + ldc_pad
    cbuf = torch.full((M + 2, ldc), SENTINEL, dtype=TORCH_OUT[out], device=dev)
    cfg = g.gemm_query_ex(plan.handle, op_a, op_b, a.data_ptr(), a.stride(0), b.data_ptr(),
                          b.stride(0), cbuf.data_ptr(), ldc, out, M, N, K, g.GEMM_F16)
    assert (cfg["kernel"], cfg["block_m"], cfg["block_n"]) == (g.GEMM_KERNEL_TMA, 64, 64), cfg
    got = run_ex(plan, stored(A, op_a), stored(B, op_b), op_a, op_b, M, N, K, out, ldc=ldc)
    assert np.all(got[:M, N:] == SENTINEL) and np.all(got[M:] == SENTINEL), "guard cells"
    ref = oracle.gemm(A, B)
    assert np.array_equal(got[:M, :N], ref), f"max diff {np.abs(got[:M, :N] - ref).max()}"
