"""GPU parity at the sizes where 32-bit offsets would break (through the C ABI).

The boundary accepts M, N and K up to 2^31 - 1025 each, so C, A and B may hold
more than 2^31 elements and their byte offsets may pass 2^32.  These cases put
entries there and compare them with the fp64 oracle:

* C of 65600 x 33000 (2.16e9 elements, 8.7 GB) with the automatic kernel, with
  the one-CTA kernel forced, and with a pitch that rules out TMA stores;
* a tall problem (10^8 + 3 rows of A and C) and a wide one (N = 5e7 + 8, B of
  6.4 GB), whose operand offsets pass 2^32 bytes;
* K = 2^20 with the automatic kernel and K = 2^18 with the pair kernel's
  whole-problem stream-K, on integer-valued inputs that must match exactly.

Large operands repeat a block whose period (65537 rows or columns) is prime, so
an offset that wrapped at any power of two would land on a different row or
column of the block and change the value.  Entries are compared on a sample
(random, corners, tile edges, and the part of C past 2^31 elements) by the
oracle's entry-wise routine; every entry of C is checked to be written, and
the cells right of column N (padded pitch) to be untouched.
"""
import numpy as np
import pytest
import torch

import dense_gemm_05_gb300 as g
import oracle

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-5
PERIOD = 65537          # prime: no power of two is a multiple of it


@pytest.fixture(scope="module")
def plan():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    p = g.Plan(0)
    yield p
    p.close()


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def uniform(rows, cols, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    return (torch.rand(rows, cols, generator=gen) * 2.0 - 1.0).to(dtype)


def ternary(rows, cols, dtype, seed):
    """Entries in {-1, 0, 1}: every partial sum up to K = 2^24 is exact in fp32."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(-1, 2, (rows, cols), generator=gen).to(dtype)


def sample(M, N, ld, n, seed, tile_m=256, tile_n=256):
    """Row and column indices: random, the four corners, entries on tile edges,
    and (when C has more than 2^31 elements) entries past element 2^31."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n)) + [0, 0, M - 1, M - 1]
    cols = list(rng.integers(0, N, n)) + [0, N - 1, 0, N - 1]
    for _ in range(n // 4):
        r = int(rng.integers(0, M))
        c = int(rng.integers(0, N))
        rows += [min(M - 1, (r // tile_m) * tile_m + tile_m - 1), r]
        cols += [c, min(N - 1, (c // tile_n) * tile_n + tile_n - 1)]
    first = -(-(1 << 31) // ld)
    if first < M:
        rows += list(rng.integers(first, M, n // 2))
        cols += list(rng.integers(0, N, n // 2))
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


def gather(c, rows, cols):
    dev = c.device
    return c[torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)].cpu().double().numpy()


def check_close(got, ref, bnd, what):
    ok = np.abs(got - ref) <= REL * bnd + ABS
    assert ok.all(), (f"{what}: {int((~ok).sum())} of {ok.size} sampled entries outside tolerance; "
                      f"first bad index {int(np.argmax(~ok))}")


@pytest.mark.parametrize("kernel,pad", [(0, 0), (0, 1), (g.GEMM_KERNEL_TMA, 0)],
                         ids=["auto", "auto-unaligned-ldc", "one-cta"])
def test_c_beyond_2_31_elements(plan, kernel, pad):
    M, N, K = 65600, 33000, 64
    A, B = uniform(M, K, torch.float16, 21), uniform(K, N, torch.float16, 22)
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    buf = torch.full((M, N + pad), float("nan"), dtype=torch.float32, device=dev)
    c = buf[:, :N]
    assert M * c.stride(0) > (1 << 31)
    plan.force(kernel, 0, 0)
    try:
        cfg = plan.query(a, b, c)
        if kernel:
            assert cfg["kernel"] == kernel, cfg
        plan.run(a, b, c)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
    assert not torch.isnan(c).any().item(), "some C entries were never written"
    if pad:
        assert torch.isnan(buf[:, N:]).all().item(), "a store landed right of column N"
    rows, cols = sample(M, N, c.stride(0), 4096, 23, cfg["block_m"], cfg["block_n"])
    ref, bnd = oracle.gemm_entries(A, B, rows, cols)
    check_close(gather(c, rows, cols), ref, bnd, f"65600x33000 C, kernel {cfg['kernel']}")


def test_tall_operand_offsets_past_2_32_bytes(plan):
    """A and C of 10^8 + 3 rows: A's byte offsets reach 6.4e9, C's 9.6e9."""
    M, N, K = 100_000_003, 24, 32
    blk = uniform(PERIOD, K, torch.bfloat16, 31)
    B = uniform(K, N, torch.bfloat16, 32)
    dev = torch.device("cuda:0")
    a = blk.to(dev).repeat(-(-M // PERIOD), 1)[:M].contiguous()
    b = B.to(dev)
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    plan.run(a, b, c)
    torch.cuda.synchronize()
    assert not torch.isnan(c).any().item(), "some C entries were never written"
    rows, cols = sample(M, N, N, 4096, 33)
    ref, bnd = oracle.gemm_entries(blk, B, rows % PERIOD, cols)
    check_close(gather(c, rows, cols), ref, bnd, "tall 1e8 x 24 x 32")


def test_wide_operand_offsets_past_2_32_bytes(plan):
    """M = 16 and N = 5e7 + 8: B's byte offsets reach 6.4e9 (the small-M kernels)."""
    M, N, K = 16, 50_000_008, 64
    A = uniform(M, K, torch.bfloat16, 41)
    blk = uniform(K, PERIOD, torch.bfloat16, 42)
    dev = torch.device("cuda:0")
    a = A.to(dev)
    b = blk.to(dev).repeat(1, -(-N // PERIOD))[:, :N].contiguous()
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    cfg = plan.query(a, b, c)
    plan.run(a, b, c)
    torch.cuda.synchronize()
    assert not torch.isnan(c).any().item(), "some C entries were never written"
    rows, cols = sample(M, N, N, 4096, 43, M, cfg["block_n"])
    ref, bnd = oracle.gemm_entries(A, blk, rows, cols % PERIOD)
    check_close(gather(c, rows, cols), ref, bnd, f"wide 16 x 5e7 x 64, kernel {cfg['kernel']}")


@pytest.mark.parametrize("M,N,K,kernel,split,block_n",
                         [(256, 256, 1 << 20, 0, 0, 0),
                          (512, 512, 1 << 18, g.GEMM_KERNEL_PAIR, 2, 256)],
                         ids=["auto-k2^20", "pair-stream-k-k2^18"])
def test_long_k_integer_exact(plan, M, N, K, kernel, split, block_n):
    """Deep K loops (16384 and 4096 K blocks): sampled entries equal the exact sums."""
    A, B = ternary(M, K, torch.bfloat16, 51), ternary(K, N, torch.bfloat16, 52)
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    plan.force(kernel, split, block_n)
    try:
        cfg = plan.query(a, b, c)
        if kernel:
            assert cfg["kernel"] == kernel, cfg
        plan.run(a, b, c)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
    assert not torch.isnan(c).any().item(), "some C entries were never written"
    rows, cols = sample(M, N, N, 256, 53, cfg["block_m"], cfg["block_n"])
    ref, _ = oracle.gemm_entries(A, B, rows, cols)
    got = gather(c, rows, cols)
    assert np.array_equal(got, ref), f"K = {K}, kernel {cfg['kernel']}: max diff {np.abs(got - ref).max()}"
