"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerance (the problem's stated bar): |C_gpu - C_ref| <= 1e-3 * sum_k |A_ik||B_kj| + 1e-5
element-wise.  Integer-valued inputs (entries in [-4, 4], |sums| < 2^24) must
match bit for bit.  Every C buffer carries guard cells (extra rows and a padded
leading dimension filled with a sentinel) that must survive unchanged.
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


def run(plan, A, B, M, N, K, *, ldc=None, kernel=0, split=0, block_n=0, group=None,
        expect=None):
    """Copy A, B (CPU, possibly padded) to the GPU, run the C ABI, return the C buffer."""
    ldc = N if ldc is None else ldc
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    cbuf = torch.full((M + 2, max(ldc, 1)), SENTINEL, dtype=torch.float32, device=dev)
    plan.force(kernel, split, block_n)
    if group is not None:
        plan.set_group(group)
    try:
        if expect is not None:
            cfg = plan.query(a, b, cbuf, M, N, K)
            assert cfg["kernel"] == expect, cfg
        plan.run(a, b, cbuf, M, N, K)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
        if group is not None:
            plan.set_group(8)
    return cbuf.cpu().double().numpy()


def assert_guards(cbuf, M, N):
    assert np.all(cbuf[:M, N:] == SENTINEL), "a store landed right of column N"
    assert np.all(cbuf[M:, :] == SENTINEL), "a store landed below row M"


def assert_close(got, A, B, M, N, K, what=""):
    ref = oracle.gemm(A, B, K=K, N=N)
    bnd = oracle.absbound(A, B, K=K, N=N)
    ok = np.abs(got - ref) <= REL * bnd + ABS
    if not ok.all():
        idx = np.argwhere(~ok)
        i, j = idx[0]
        raise AssertionError(
            f"{what}: {len(idx)} of {ok.size} entries outside tolerance; first at ({i}, {j}): "
            f"gpu {got[i, j]!r} oracle {ref[i, j]!r} bound {bnd[i, j]!r}")
    return ref


# ---------------------------------------------------------------- bounded waits

def test_wait_selftest_gives_up_and_context_survives(plan):
    st = g.gemm_wait_selftest(2000, torch.cuda.current_stream().cuda_stream)
    assert st == g.GEMM_ERR_TIMEOUT
    A, B = workloads.custom(64, 64, 64, "f16", seed=0)
    got = run(plan, A, B, 64, 64, 64)
    assert_close(got[:64, :64], A, B, 64, 64, 64, "after self-test")


# ---------------------------------------------------------------- the five workloads

def test_workload_256_f16_full(plan):
    w = workloads.WORKLOADS["gemm256_f16"]
    A, B = workloads.make_inputs(w)
    got = run(plan, A, B, w.M, w.N, w.K, expect=g.GEMM_KERNEL_TMA)
    assert_guards(got, w.M, w.N)
    assert_close(got[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name)


def test_workload_ragged_f16_full(plan):
    """M=1023 K=1000 N=1029: ldb = 1029 halves is not a 16-byte pitch -> B is staged
    into 16-byte rows and the TMA-fed kernels read the copy: automatically the
    split-K cluster kernel (72 tiles of 128 x 128 on 144 SMs), and the one-CTA
    kernel when forced; with staging off the cluster kernel reads B in place."""
    w = workloads.WORKLOADS["ragged1023x1000x1029_f16"]
    A, B = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    cfg = plan.query(A.to(dev), B.to(dev), torch.empty(w.M, w.N, device=dev))
    assert cfg["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR and cfg["staged"] == 2, cfg
    assert cfg["block_m"] == 128 and cfg["block_n"] == 128 and cfg["grid"] == 144, cfg
    got = run(plan, A, B, w.M, w.N, w.K, expect=g.GEMM_KERNEL_SPLIT_PAIR)
    assert_guards(got, w.M, w.N)
    assert_close(got[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name)
    got = run(plan, A, B, w.M, w.N, w.K, kernel=g.GEMM_KERNEL_TMA, expect=g.GEMM_KERNEL_TMA)
    assert_guards(got, w.M, w.N)
    assert_close(got[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name + " one-CTA tiles")
    plan.set_staging(False)
    try:
        got = run(plan, A, B, w.M, w.N, w.K, expect=g.GEMM_KERNEL_SPLIT_PAIR)
    finally:
        plan.set_staging(True)
    assert_guards(got, w.M, w.N)
    assert_close(got[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name + " B in place")


def test_workload_ragged_f16_generic_in_place(plan):
    """The same workload with the generic kernel forced: B read in place."""
    w = workloads.WORKLOADS["ragged1023x1000x1029_f16"]
    A, B = workloads.make_inputs(w)
    got = run(plan, A, B, w.M, w.N, w.K, kernel=g.GEMM_KERNEL_GENERIC,
              expect=g.GEMM_KERNEL_GENERIC)
    assert_guards(got, w.M, w.N)
    assert_close(got[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name + " generic")


def test_workload_ragged_f16_padded_pitch_uses_tma(plan):
    """Same logical shape with 16-byte pitches (NaN padding): TMA path, ragged edges."""
    w = workloads.WORKLOADS["ragged1023x1000x1029_f16"]
    A, B = workloads.make_inputs(w, lda=1008, ldb=1032)
    got = run(plan, A, B, w.M, w.N, w.K, ldc=1032, kernel=g.GEMM_KERNEL_TMA,
              expect=g.GEMM_KERNEL_TMA)
    assert_guards(got, w.M, w.N)
    assert_close(got[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name + " padded")
    got = run(plan, A, B, w.M, w.N, w.K, ldc=1032, expect=g.GEMM_KERNEL_SPLIT_PAIR)
    assert_guards(got, w.M, w.N)
    assert_close(got[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name + " padded, split pair")


def test_workload_skinny_full_and_deterministic(plan):
    w = workloads.WORKLOADS["skinny16x4096x14336_bf16"]
    A, B = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    cfg = plan.query(A.to(dev), B.to(dev), torch.empty(w.M, w.N, device=dev))
    # 56 strips of 256 columns on 56 two-CTA clusters.
    assert cfg["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR, cfg
    assert cfg["block_n"] == 256 and cfg["grid"] == 112 and cfg["cluster"] == 2, cfg
    got1 = run(plan, A, B, w.M, w.N, w.K)
    got2 = run(plan, A, B, w.M, w.N, w.K)
    assert_guards(got1, w.M, w.N)
    assert np.array_equal(got1, got2), "split-K result changed between runs"
    assert_close(got1[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name)
    # the stream-K kernel on the same problem agrees within the tolerance too
    got3 = run(plan, A, B, w.M, w.N, w.K, kernel=g.GEMM_KERNEL_SKINNY, expect=g.GEMM_KERNEL_SKINNY)
    assert_close(got3[:w.M, :w.N], A, B, w.M, w.N, w.K, w.name + " stream-K")


@pytest.mark.parametrize("M,K,N,dtype,shares", [
    (8, 1024, 65600, "bf16", 152),   # 513 tiles in 152 shares: shares span several tiles
    (8, 1024, 65600, "bf16", 0),     # automatic choice
    (33, 2048, 640, "f16", 0),       # 5 tiles, MMA N = 64, tiles split across many shares
    (1, 8192, 136, "bf16", 0),       # 2 tiles, 128 K blocks, ragged last tile
    (16, 4096, 14336, "bf16", 152),  # the M=16 workload's shape, one share per SM
    (16, 4096, 14336, "bf16", 448),  # four shares per tile
])
def test_skinny_stream_k_shapes(plan, M, K, N, dtype, shares):
    A, B = workloads.custom(M, K, N, dtype, seed=M + K + N, dist="normal")
    got1 = run(plan, A, B, M, N, K, kernel=g.GEMM_KERNEL_SKINNY, split=shares,
               expect=g.GEMM_KERNEL_SKINNY)
    got2 = run(plan, A, B, M, N, K, kernel=g.GEMM_KERNEL_SKINNY, split=shares,
               expect=g.GEMM_KERNEL_SKINNY)
    assert_guards(got1, M, N)
    assert np.array_equal(got1, got2), "stream-K result changed between runs"
    assert_close(got1[:M, :N], A, B, M, N, K, f"skinny {M}x{N}x{K} shares={shares}")


@pytest.mark.parametrize("M,K,N,dtype,block_n", [
    (16, 4096, 14336, "bf16", 0),    # the M=16 workload: automatic 256-column strips
    (1, 256, 1000, "f16", 128),      # M = 1, 4 K blocks, ragged last strip
    (1023, 1000, 1029, "f16", 0),    # 128-row tiles, 8 x 9 of them, ragged M, K and N
    (129, 520, 300, "bf16", 128),    # 128-row tiles: 2 rows of tiles, the second holds one row
    (600, 2048, 1100, "bf16", 128),  # 5 x 9 tiles
    (256, 130, 4000, "f16", 128),    # 3 K blocks, 64 tiles
    (640, 1024, 2048, "bf16", 128),  # 80 tiles: more clusters than fit at once
    (33, 1000, 700, "bf16", 192),    # M padded to 64 (two TMEM lane quadrants), ragged K and N
    (64, 130, 513, "f16", 256),      # 3 K blocks: halves of 1 and 2, ragged everywhere
    (17, 2048, 9728, "bf16", 128),   # M padded to 32, 76 strips
    (16, 128, 256, "bf16", 256),     # 2 K blocks: one per CTA, a single strip
    (8, 512, 40000, "bf16", 128),    # 313 strips: more clusters than fit at once
])
def test_split_pair_shapes(plan, M, K, N, dtype, block_n):
    """Small M on 2-CTA clusters (K halves exchanged through distributed shared memory)."""
    A, B = workloads.custom(M, K, N, dtype, seed=M + K + N + 1, dist="normal")
    kernel = 0 if block_n == 0 else g.GEMM_KERNEL_SPLIT_PAIR
    got1 = run(plan, A, B, M, N, K, kernel=kernel, block_n=block_n,
               expect=g.GEMM_KERNEL_SPLIT_PAIR)
    got2 = run(plan, A, B, M, N, K, kernel=kernel, block_n=block_n)
    assert_guards(got1, M, N)
    assert np.array_equal(got1, got2), "result changed between runs"
    assert_close(got1[:M, :N], A, B, M, N, K, f"split pair {M}x{N}x{K} bn={block_n}")


def test_split_pair_query(plan):
    dev = torch.device("cuda:0")
    a = torch.empty(64, 4096, dtype=torch.bfloat16, device=dev)
    b = torch.empty(4096, 40000, dtype=torch.bfloat16, device=dev)
    c = torch.empty(64, 40000, device=dev)
    plan.force(g.GEMM_KERNEL_SPLIT_PAIR, 0, 192)
    try:
        cfg = plan.query(a, b, c, 20, 1000, 4096)
        assert cfg["block_m"] == 32 and cfg["block_n"] == 192 and cfg["split_k"] == 2, cfg
        assert cfg["tiles"] == 6 and cfg["grid"] == 12 and cfg["cluster"] == 2, cfg
        plan.force(g.GEMM_KERNEL_SPLIT_PAIR, 0, 0)
        assert plan.query(a, b, c, 20, 1000, 4096)["block_n"] == 128
        assert plan.query(a, b, c, 20, 14336, 4096)["block_n"] == 256
        assert plan.query(a, b, c, 40, 14336, 4096)["block_n"] == 192
        r = plan.query(a, b, c, 65, 1000, 4096)          # M > 64: tiles of 128 x 128
        assert r["block_m"] == 128 and r["block_n"] == 128 and r["tiles"] == 8, r
        plan.force(g.GEMM_KERNEL_SPLIT_PAIR, 0, 192)
        with pytest.raises(RuntimeError):
            plan.query(a, b, c, 65, 1000, 4096)          # M > 64 takes 128 columns only
        plan.force(g.GEMM_KERNEL_SPLIT_PAIR, 0, 0)
        with pytest.raises(RuntimeError):
            plan.query(a, b, c, 16, 1000, 64)            # one K block
        plan.force(g.GEMM_KERNEL_TMA, 0, 192)            # 192 columns: this kernel only
        with pytest.raises(RuntimeError):
            plan.query(a, b, c, 16, 1000, 4096)
    finally:
        plan.force(0, 0, 0)
    # automatic: few strips leave SMs idle, so the stream-K kernel is chosen
    assert plan.query(a, b, c, 16, 4096, 4096)["kernel"] == g.GEMM_KERNEL_SKINNY
    assert plan.query(a, b, c, 16, 8192, 4096)["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR
    assert plan.query(a, b, c, 16, 14336, 512)["kernel"] == g.GEMM_KERNEL_SKINNY   # 8 K blocks


def test_dependent_launches_read_the_previous_output(plan):
    """Kernels are launched as programmatic dependents: each may start while the
    previous one drains and must wait before reading its output.  A chain on one
    stream, each GEMM reading the C of the one before (exact integer values, so
    any stale or partial read shows): C1 = A B1 (bf16 out, pair tiles), then
    C1 I (pair tiles), C1[:16] I (stream-K swap-AB, M = 16), C1[:300] I[:, :1024]
    (split pair with 128-row tiles), each into a NaN-filled buffer."""
    dev = torch.device("cuda:0")
    gen = torch.Generator().manual_seed(17)
    M, K, N = 4096, 256, 4096
    A = torch.randint(-1, 2, (M, K), generator=gen).to(torch.bfloat16)
    B1 = torch.randint(-1, 2, (K, N), generator=gen).to(torch.bfloat16)
    a, b1 = A.to(dev), B1.to(dev)
    eye = torch.eye(N, dtype=torch.bfloat16, device=dev)
    c1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    c2 = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    c3 = torch.full((16, N), float("nan"), dtype=torch.float32, device=dev)
    c4 = torch.full((300, N), float("nan"), dtype=torch.float32, device=dev)
    assert plan.query_ex(a, b1, c1)["kernel"] == g.GEMM_KERNEL_PAIR
    assert plan.query_ex(c1, eye, c2)["kernel"] == g.GEMM_KERNEL_PAIR
    assert plan.query_ex(c1[:16], eye, c3)["kernel"] == g.GEMM_KERNEL_SKINNY
    assert plan.query_ex(c1[:300], eye[:, :1024], c4[:, :1024])["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR
    for _ in range(3):
        for t in (c1, c2, c3, c4):
            t.fill_(float("nan"))
        plan.run_ex(a, b1, c1)
        plan.run_ex(c1, eye, c2)
        plan.run_ex(c1[:16], eye, c3)
        plan.run_ex(c1[:300], eye[:, :1024], c4[:, :1024])
        torch.cuda.synchronize()
        ref = torch.from_numpy(oracle.gemm(A, B1))          # |entries| <= 256: exact in bf16
        assert torch.equal(c1.cpu().double(), ref)
        assert torch.equal(c2.cpu(), c1.float().cpu())
        assert torch.equal(c3.cpu(), c1[:16].float().cpu())
        assert torch.equal(c4[:, :1024].cpu(), c1[:300, :1024].float().cpu())


def _sample_entries(M, N, bm, bn, n_random, seed):
    """n_random uniform entries plus, for every tile on the border of C, its four
    corners and 16 random entries."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n_random))
    cols = list(rng.integers(0, N, n_random))
    tm, tn = -(-M // bm), -(-N // bn)
    for ti in range(tm):
        for tj in range(tn):
            if ti not in (0, tm - 1) and tj not in (0, tn - 1):
                continue
            r0, c0 = ti * bm, tj * bn
            r1, c1 = min(M, r0 + bm) - 1, min(N, c0 + bn) - 1
            rows += [r0, r0, r1, r1] + list(rng.integers(r0, r1 + 1, 16))
            cols += [c0, c1, c0, c1] + list(rng.integers(c0, c1 + 1, 16))
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


@pytest.mark.parametrize("name,kernel", [("square4096_bf16", 0), ("square8192_bf16", 0),
                                         ("square4096_bf16", g.GEMM_KERNEL_TMA),
                                         ("square8192_bf16", g.GEMM_KERNEL_TMA)])
def test_workload_square_sampled(plan, name, kernel):
    """The square workloads with the automatic choice (pair tiles) and the one-CTA kernel."""
    w = workloads.WORKLOADS[name]
    A, B = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    c = torch.full((w.M, w.N), float("nan"), dtype=torch.float32, device=dev)
    plan.force(kernel, 0, 0)
    try:
        cfg = plan.query(a, b, c)
        assert cfg["kernel"] == (kernel or g.GEMM_KERNEL_PAIR), cfg
        plan.run(a, b, c)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
    assert not torch.isnan(c).any().item(), "some C entries were never written"
    rows, cols = _sample_entries(w.M, w.N, cfg["block_m"], cfg["block_n"], 4096, w.seed)
    got = c[torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)].cpu().double().numpy()
    ref, bnd = oracle.gemm_entries(A, B, rows, cols)
    ok = np.abs(got - ref) <= REL * bnd + ABS
    assert ok.all(), f"{name}: {int((~ok).sum())} of {ok.size} sampled entries outside tolerance"


@pytest.mark.parametrize("name,block_n", [("square4096_bf16", 128), ("square4096_bf16", 256),
                                          ("square8192_bf16", 256)])
def test_workload_square_sampled_pair(plan, name, block_n):
    """The 2-SM pair-tile kernel on the square workloads."""
    w = workloads.WORKLOADS[name]
    A, B = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    c = torch.full((w.M, w.N), float("nan"), dtype=torch.float32, device=dev)
    plan.force(g.GEMM_KERNEL_PAIR, 0, block_n)
    try:
        cfg = plan.query(a, b, c)
        assert cfg["kernel"] == g.GEMM_KERNEL_PAIR and cfg["cluster"] == 2, cfg
        plan.run(a, b, c)
        torch.cuda.synchronize()
    finally:
        plan.force(0, 0, 0)
    assert not torch.isnan(c).any().item(), "some C entries were never written"
    rows, cols = _sample_entries(w.M, w.N, cfg["block_m"], cfg["block_n"], 4096, w.seed)
    got = c[torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)].cpu().double().numpy()
    ref, bnd = oracle.gemm_entries(A, B, rows, cols)
    ok = np.abs(got - ref) <= REL * bnd + ABS
    assert ok.all(), f"{name} pair: {int((~ok).sum())} of {ok.size} sampled entries outside tolerance"


@pytest.mark.parametrize("M,N,K,block_n", [(257, 130, 70, 128), (1, 64, 64, 128),
                                           (129, 520, 1000, 256), (1023, 1029, 1000, 256)])
def test_pair_ragged_padded(plan, M, N, K, block_n):
    lda, ldb = -(-K // 8) * 8, -(-N // 8) * 8
    A, B = workloads.custom(M, K, N, "f16", seed=M + N, lda=lda, ldb=ldb)
    got = run(plan, A, B, M, N, K, ldc=N + 5, kernel=g.GEMM_KERNEL_PAIR, block_n=block_n,
              expect=g.GEMM_KERNEL_PAIR)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, f"pair {M}x{N}x{K}")


@pytest.mark.parametrize("group", [0, 3, 8])
def test_pair_tile_order_does_not_change_bits(plan, group):
    A, B = workloads.custom(1000, 512, 1300, "bf16", seed=22, dist="normal", ldb=1304)
    base = run(plan, A, B, 1000, 1300, 512, kernel=g.GEMM_KERNEL_PAIR, group=8)
    got = run(plan, A, B, 1000, 1300, 512, kernel=g.GEMM_KERNEL_PAIR, group=group)
    assert np.array_equal(base, got)


# ---------------------------------------------------------------- pair stream-K phase

def pair_sk_expected(cfg, M, N, K):
    """Stream-K shares the pair kernel should use, from the grid the plan reports:
    one per cluster when the last wave of tiles is at most half full, at least
    two full waves precede it and tiles have at least 32 K blocks; the split
    covers that partial wave, plus one full wave when the shares would otherwise
    be shorter than 16 K blocks."""
    ncl = cfg["grid"] // 2
    units = -(-M // 256) * -(-N // cfg["block_n"])
    num_kb = -(-K // 64)
    rem = units % ncl
    if rem == 0 or 2 * rem > ncl or units // ncl < 2 or num_kb < 32:
        return 0
    sk = rem if rem * num_kb // ncl >= 16 else rem + ncl
    return ncl if sk * num_kb // ncl >= 16 else 0


def query_pair(plan, A, B, M, N, K, block_n, split=0):
    dev = torch.device("cuda:0")
    c = torch.empty(M, N, dtype=torch.float32, device=dev)
    plan.force(g.GEMM_KERNEL_PAIR, split, block_n)
    try:
        return plan.query(A.to(dev), B.to(dev), c, M, N, K)
    finally:
        plan.force(0, 0, 0)


# (M, K, N, dtype, block_n), with 76 clusters: 160 tiles of 256 columns over
# K = 3072 (8 + 76 split tiles, two shares per split tile); 176 tiles of 128
# columns over K = 4096 (the 24 tiles of the partial wave, each split over 4-5
# shares); 190 tiles of 256 columns over K = 2048 (38 split tiles, 2-3 shares
# each).
SK_EXACT = [(2048, 3072, 5120, "bf16", 256), (2048, 4096, 2816, "f16", 128),
            (2560, 2048, 4864, "bf16", 256)]


@pytest.mark.parametrize("M,K,N,dtype,block_n", SK_EXACT)
def test_pair_stream_k_integer_exact(plan, M, K, N, dtype, block_n):
    A, B = int_inputs(M, K, N, dtype, seed=M + K + N + 1)
    cfg = query_pair(plan, A, B, M, N, K, block_n)
    expected = pair_sk_expected(cfg, M, N, K)
    assert cfg["shares"] == expected, cfg
    if expected == 0:
        pytest.skip(f"{cfg['grid'] // 2} clusters leave no partial wave for this shape")
    assert cfg["split_k"] >= 2, cfg
    got = run(plan, A, B, M, N, K, ldc=N + 8, kernel=g.GEMM_KERNEL_PAIR, block_n=block_n)
    assert_guards(got, M, N)
    ref = oracle.gemm(A, B)
    assert np.array_equal(got[:M, :N], ref), f"max diff {np.abs(got[:M, :N] - ref).max()}"


@pytest.mark.parametrize("block_n", [128, 256])
def test_pair_whole_problem_stream_k(plan, block_n):
    """split_k = 2: every tile's 128 K blocks split over all clusters (76 shares of
    27 or 54 K blocks: 3-6 shares per tile); integer inputs stay exact."""
    M, K, N = 1024, 8192, 1024
    A, B = int_inputs(M, K, N, "bf16", seed=77)
    cfg = query_pair(plan, A, B, M, N, K, block_n, split=2)
    assert cfg["shares"] == cfg["grid"] // 2 and cfg["split_k"] >= 3, cfg
    got = run(plan, A, B, M, N, K, ldc=N + 4, kernel=g.GEMM_KERNEL_PAIR, split=2, block_n=block_n)
    assert_guards(got, M, N)
    assert np.array_equal(got[:M, :N], oracle.gemm(A, B))


@pytest.mark.parametrize("block_n", [128, 256])
def test_pair_stream_k_ragged(plan, block_n):
    """Ragged M, N and K in the split tiles: 10 x 17 (or 33) tiles, K = 2100."""
    M, K, N = 2500, 2100, 4100
    lda, ldb = 2104, 4104
    A, B = workloads.custom(M, K, N, "bf16", seed=31 + block_n, dist="normal", lda=lda, ldb=ldb)
    cfg = query_pair(plan, A, B, M, N, K, block_n)
    assert cfg["shares"] == pair_sk_expected(cfg, M, N, K), cfg
    got = run(plan, A, B, M, N, K, ldc=N + 5, kernel=g.GEMM_KERNEL_PAIR, block_n=block_n)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, f"pair stream-K {M}x{N}x{K} bn={block_n}")


def test_pair_stream_k_deterministic_and_ablation(plan):
    """Fixed-order fix-up: repeated runs agree bit for bit; split_k = 1 turns the
    phase off and still matches the oracle."""
    M, K, N = 2048, 2048, 5120
    A, B = workloads.custom(M, K, N, "bf16", seed=44, dist="normal")
    assert query_pair(plan, A, B, M, N, K, 256)["shares"] > 0
    assert query_pair(plan, A, B, M, N, K, 256, split=1)["shares"] == 0
    got1 = run(plan, A, B, M, N, K, kernel=g.GEMM_KERNEL_PAIR, block_n=256)
    got2 = run(plan, A, B, M, N, K, kernel=g.GEMM_KERNEL_PAIR, block_n=256)
    assert np.array_equal(got1, got2), "stream-K result changed between runs"
    off = run(plan, A, B, M, N, K, kernel=g.GEMM_KERNEL_PAIR, split=1, block_n=256)
    assert_close(got1[:M, :N], A, B, M, N, K, "pair stream-K on")
    assert_close(off[:M, :N], A, B, M, N, K, "pair stream-K off")


# ---------------------------------------------------------------- exactness

def int_inputs(M, K, N, dtype, seed, lda=None, ldb=None):
    gen = torch.Generator().manual_seed(seed)
    td = torch.float16 if dtype == "f16" else torch.bfloat16
    A = torch.randint(-4, 5, (M, K), generator=gen).to(td)
    B = torch.randint(-4, 5, (K, N), generator=gen).to(td)
    if lda is not None:
        Ap = torch.full((M, lda), float("nan"), dtype=td)
        Ap[:, :K] = A
        A = Ap
    if ldb is not None:
        Bp = torch.full((K, ldb), float("nan"), dtype=td)
        Bp[:, :N] = B
        B = Bp
    return A, B


@pytest.mark.parametrize("kernel,split,shape,dtype", [
    (g.GEMM_KERNEL_TMA, 0, (300, 1000, 520), "bf16"),
    (g.GEMM_KERNEL_TMA, 0, (1024, 2048, 1024), "f16"),
    (g.GEMM_KERNEL_GENERIC, 0, (300, 1000, 520), "f16"),
    (g.GEMM_KERNEL_SKINNY, 1, (16, 4096, 1024), "bf16"),
    (g.GEMM_KERNEL_SKINNY, 12, (16, 4096, 1024), "bf16"),
    (g.GEMM_KERNEL_SKINNY, 0, (33, 2048, 640), "f16"),
    (g.GEMM_KERNEL_SKINNY, 3, (64, 1000, 256), "bf16"),
    (g.GEMM_KERNEL_SPLIT_PAIR, 192, (16, 4096, 1024), "bf16"),
    (g.GEMM_KERNEL_SPLIT_PAIR, 128, (40, 1000, 520), "f16"),
    (g.GEMM_KERNEL_SPLIT_PAIR, 128, (300, 1000, 520), "bf16"),
    (g.GEMM_KERNEL_PAIR, 128, (600, 1024, 1104), "bf16"),
    (g.GEMM_KERNEL_PAIR, 256, (600, 1024, 1104), "f16"),
    (g.GEMM_KERNEL_PAIR, 256, (1024, 4096, 1024), "bf16"),
])
def test_small_integer_inputs_are_bit_exact(plan, kernel, split, shape, dtype):
    """For the pair kernels the second parameter is the tile width (block_n)."""
    M, K, N = shape
    A, B = int_inputs(M, K, N, dtype, seed=M + K + N)
    if kernel in (g.GEMM_KERNEL_PAIR, g.GEMM_KERNEL_SPLIT_PAIR):
        got = run(plan, A, B, M, N, K, kernel=kernel, block_n=split, expect=kernel)
    else:
        got = run(plan, A, B, M, N, K, kernel=kernel, split=split, expect=kernel)
    assert_guards(got, M, N)
    ref = oracle.gemm(A, B)
    assert np.array_equal(got[:M, :N], ref), f"max diff {np.abs(got[:M, :N] - ref).max()}"


def test_mn_major_layout_pin(plan):
    """A = I, B with distinct entries: C must equal B exactly (a transposed or
    mis-swizzled B tile shows up as a permutation)."""
    M = K = 192
    N = 320
    A = torch.eye(M, K, dtype=torch.bfloat16)
    B = (torch.arange(K * N, dtype=torch.float32).reshape(K, N) % 251).to(torch.bfloat16)
    for kernel in (g.GEMM_KERNEL_TMA, g.GEMM_KERNEL_GENERIC, g.GEMM_KERNEL_PAIR):
        got = run(plan, A, B, M, N, K, kernel=kernel)
        assert np.array_equal(got[:M, :N], B.double().numpy()), kernel
    # skinny: first 16 rows of the identity
    A16 = torch.eye(16, K, dtype=torch.bfloat16)
    got = run(plan, A16, B, 16, N, K, kernel=g.GEMM_KERNEL_SKINNY, split=2)
    assert np.array_equal(got[:16, :N], B[:16].double().numpy())
    for bn in (128, 192, 256):
        got = run(plan, A16, B, 16, N, K, kernel=g.GEMM_KERNEL_SPLIT_PAIR, block_n=bn)
        assert np.array_equal(got[:16, :N], B[:16].double().numpy()), bn


# ---------------------------------------------------------------- ragged sweep

SWEEP = [(m, n, k) for m in (1, 17, 128, 129, 255) for n in (1, 15, 128, 257)
         for k in (1, 16, 63, 130)] + [(1000, 1023, 127), (127, 255, 1000), (65, 4096, 96)]


@pytest.mark.parametrize("M,N,K", SWEEP)
def test_ragged_sweep(plan, M, N, K):
    A, B = workloads.custom(M, K, N, "f16", seed=M * 7 + N * 3 + K)
    got = run(plan, A, B, M, N, K)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 130), (17, 15, 63), (255, 128, 1000)])
def test_ragged_sweep_generic_in_place(plan, M, N, K):
    A, B = workloads.custom(M, K, N, "f16", seed=M + N + K)
    got = run(plan, A, B, M, N, K, kernel=g.GEMM_KERNEL_GENERIC, expect=g.GEMM_KERNEL_GENERIC)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, f"generic {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,lda,ldb,staged", [
    (300, 520, 1001, 1001, 520, 1),      # A rows of 1001 halves
    (300, 517, 640, 640, 517, 2),        # B rows of 517 halves (10 K blocks: one-CTA tiles)
    (1000, 1300, 777, 779, 1301, 3),     # both, with padding beyond K and N
    (40, 3000, 1003, 1003, 3000, 1),     # skinny M with A staged
])
def test_staged_operands(plan, M, N, K, lda, ldb, staged):
    A, B = workloads.custom(M, K, N, "bf16", seed=lda + ldb, dist="normal", lda=lda, ldb=ldb)
    dev = torch.device("cuda:0")
    cfg = plan.query(A.to(dev), B.to(dev), torch.empty(M, N, device=dev), M, N, K)
    assert cfg["staged"] == staged and cfg["kernel"] != g.GEMM_KERNEL_GENERIC, cfg
    got = run(plan, A, B, M, N, K, ldc=N + 1)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, f"staged {M}x{N}x{K}")


def test_staged_misaligned_base_and_integer_exact(plan):
    """A starting one element past a 16-byte boundary is staged; small integers stay exact."""
    M, K, N = 500, 640, 384
    A, B = int_inputs(M, K, N, "f16", seed=5)
    dev = torch.device("cuda:0")
    abuf = torch.zeros(M * K + 8, dtype=torch.float16, device=dev)
    a = abuf[1:1 + M * K].view(M, K)
    a.copy_(A.to(dev))
    b = B.to(dev)
    c = torch.full((M, N), SENTINEL, dtype=torch.float32, device=dev)
    cfg = plan.query(a, b, c)
    assert cfg["staged"] == 1, cfg
    plan.run(a, b, c)
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().double().numpy(), oracle.gemm(A, B))


def test_too_large_to_stage_uses_generic(plan):
    # B of 33.6 MB (more than the staging buffer) and 528 tiles (too many for the
    # split-pair kernel): the generic kernel reads both operands in place.
    M, K, N = 1100, 4096, 4100
    A, B = workloads.custom(M, K, N, "bf16", seed=3, dist="normal", ldb=4101)
    got = run(plan, A, B, M, N, K, expect=g.GEMM_KERNEL_GENERIC)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, "unstaged generic")


# ---------------------------------------------------------------- B read in place
# A K x N B whose base or pitch is not a multiple of 16 bytes, with an aligned
# A, in a problem the split-pair kernel takes with 128 x 128 tiles, read in
# place (staging off, or a B too large for the staging buffer): the kernel's
# four epilogue warps copy each row's 16-byte-aligned span during the K loop
# and shift it into the swizzled stage.  Pitches with various 2-byte residues
# modulo 16, bases 1-3 elements past a 16-byte boundary (row 0's aligned span
# then starts before B: read element by element), K and N not multiples of
# the tile.

@pytest.mark.parametrize("M,N,K,ldb,b_off", [
    (1023, 1029, 1000, 1029, 0),         # the ragged workload's shape
    (300, 517, 1000, 517, 0),
    (129, 250, 776, 251, 1),             # K = 776, 2000: ragged, with A's pitch aligned
    (200, 1000, 2000, 1003, 2),
    (513, 381, 768, 390, 3),
    (1000, 1000, 4096, 1001, 0),
    (65, 130, 768, 133, 1),              # one tile row, ragged N
])
def test_b_in_place_integer_exact(plan, M, N, K, ldb, b_off):
    A, B = int_inputs(M, K, N, "f16" if (M + N) % 2 else "bf16", seed=M + N + K + ldb)
    dev = torch.device("cuda:0")
    td = A.dtype
    a = A.to(dev)
    bbuf = torch.full((K * ldb + b_off + 8,), float("nan"), dtype=td, device=dev)
    b = bbuf[b_off:b_off + K * ldb].view(K, ldb)
    b[:, :N].copy_(B.to(dev))
    cbuf = torch.full((M + 2, N + 3), SENTINEL, dtype=torch.float32, device=dev)
    plan.set_staging(False)
    try:
        cfg = plan.query(a, b, cbuf, M, N, K)
        assert cfg["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR and cfg["staged"] == 4, cfg
        plan.run(a, b, cbuf, M, N, K)
        torch.cuda.synchronize()
    finally:
        plan.set_staging(True)
    got = cbuf.cpu().double().numpy()
    assert_guards(got, M, N)
    ref = oracle.gemm(A, B)
    assert np.array_equal(got[:M, :N], ref), f"max diff {np.abs(got[:M, :N] - ref).max()}"


def test_b_in_place_large_b_within_tolerance(plan):
    # B of 35 MB (larger than the staging buffer): read in place, N(0,1) inputs
    M, K, N = 130, 16000, 1100
    A, B = workloads.custom(M, K, N, "bf16", seed=7, dist="normal", ldb=1103)
    got = run(plan, A, B, M, N, K, expect=g.GEMM_KERNEL_SPLIT_PAIR)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, "split pair, B in place")


def test_b_in_place_16bit_output(plan):
    M, K, N = 700, 1000, 517
    A, B = int_inputs(M, K, N, "bf16", seed=11, ldb=521)
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)[:, :N]
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    plan.set_staging(False)
    try:
        cfg = plan.query_ex(a, b, c)
        assert cfg["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR and cfg["staged"] == 4, cfg
        plan.run_ex(a, b, c)
        torch.cuda.synchronize()
    finally:
        plan.set_staging(True)
    ref = oracle.gemm(A[:, :K], B[:, :N])
    want = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert np.array_equal(c.cpu().double().numpy(), want)


@pytest.mark.parametrize("M,N,K", [(129, 257, 130), (17, 128, 63), (255, 15, 1000)])
def test_ragged_sweep_padded_pitches_tma(plan, M, N, K):
    lda, ldb = -(-K // 8) * 8 + 8, -(-N // 8) * 8 + 8
    A, B = workloads.custom(M, K, N, "bf16", seed=K, lda=lda, ldb=ldb)
    got = run(plan, A, B, M, N, K, ldc=N + 3)
    assert_guards(got, M, N)
    assert_close(got[:M, :N], A, B, M, N, K, f"padded {M}x{N}x{K}")


# ---------------------------------------------------------------- degenerate sizes

def test_k_zero_writes_zeros(plan):
    A = torch.zeros(5, 0, dtype=torch.float16)
    B = torch.zeros(0, 7, dtype=torch.float16)
    dev = torch.device("cuda:0")
    cbuf = torch.full((7, 9), SENTINEL, dtype=torch.float32, device=dev)
    st = g.gemm_run(plan.handle, 0, 0, 0, 7, cbuf.data_ptr(), 9, 5, 7, 0, g.GEMM_F16,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == g.GEMM_OK
    c = cbuf.cpu().numpy()
    assert np.all(c[:5, :7] == 0.0)
    assert np.all(c[:5, 7:] == SENTINEL) and np.all(c[5:] == SENTINEL)
    del A, B


@pytest.mark.parametrize("M,N", [(0, 7), (5, 0), (0, 0)])
def test_empty_output_is_a_no_op(plan, M, N):
    dev = torch.device("cuda:0")
    cbuf = torch.full((4, 8), SENTINEL, dtype=torch.float32, device=dev)
    a = torch.ones(8, 8, dtype=torch.float16, device=dev)
    st = g.gemm_run(plan.handle, a.data_ptr(), 8, a.data_ptr(), 8, cbuf.data_ptr(), 8, M, N, 8,
                    g.GEMM_F16, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == g.GEMM_OK
    assert torch.all(cbuf == SENTINEL).item()


# ---------------------------------------------------------------- scheduler order

@pytest.mark.parametrize("group", [0, 1, 3, 8, 16])
def test_tile_order_does_not_change_bits(plan, group):
    A, B = workloads.custom(1000, 512, 1300, "bf16", seed=21, dist="normal")
    base = run(plan, A, B, 1000, 1300, 512, group=8)
    got = run(plan, A, B, 1000, 1300, 512, group=group)
    assert np.array_equal(base, got)


# ---------------------------------------------------------------- argument checks

def test_argument_errors(plan):
    dev = torch.device("cuda:0")
    a = torch.ones(64, 64, dtype=torch.bfloat16, device=dev)
    c = torch.empty(64, 64, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    h = plan.handle
    A, C = a.data_ptr(), c.data_ptr()
    E = g.GEMM_ERR_INVALID_ARG
    U = g.GEMM_ERR_UNSUPPORTED
    assert g.gemm_run(h, A, 63, A, 64, C, 64, 64, 64, 64, g.GEMM_BF16, s) == E      # lda < K
    assert g.gemm_run(h, A, 64, A, 63, C, 64, 64, 64, 64, g.GEMM_BF16, s) == E      # ldb < N
    assert g.gemm_run(h, A, 64, A, 64, C, 63, 64, 64, 64, g.GEMM_BF16, s) == E      # ldc < N
    assert g.gemm_run(h, A, 64, A, 64, C, 64, -1, 64, 64, g.GEMM_BF16, s) == E      # M < 0
    assert g.gemm_run(h, 0, 64, A, 64, C, 64, 64, 64, 64, g.GEMM_BF16, s) == E      # A null
    assert g.gemm_run(h, A, 64, A, 64, 0, 64, 64, 64, 64, g.GEMM_BF16, s) == E      # C null
    assert g.gemm_run(h, A + 1, 64, A, 64, C, 64, 64, 64, 64, g.GEMM_BF16, s) == E  # odd address
    assert g.gemm_run(h, A, 64, A, 64, C + 2, 64, 64, 64, 64, g.GEMM_BF16, s) == E  # C misaligned
    assert g.gemm_run(h, A, 64, A, 64, A, 64, 32, 32, 64, g.GEMM_BF16, s) == E      # C overlaps A
    assert g.gemm_run(h, A, 64, A, 64, C, 64, 64, 64, 64, 7, s) == U                # dtype
    assert g.gemm_run(h, A, 64, A, 64, C, 64, 1 << 31, 64, 64, g.GEMM_BF16, s) == U
    a2 = torch.ones(128, 64, dtype=torch.bfloat16, device=dev)
    c2 = torch.empty(128, 64, dtype=torch.float32, device=dev)
    plan.force(g.GEMM_KERNEL_SKINNY, 0)
    try:
        assert g.gemm_run(h, a2.data_ptr(), 64, a2.data_ptr(), 64, c2.data_ptr(), 64, 65, 64, 64,
                          g.GEMM_BF16, s) == U                                      # skinny M > 64
    finally:
        plan.force(0, 0)
    torch.cuda.synchronize()


def test_kernel_selection(plan):
    dev = torch.device("cuda:0")
    def q(M, K, N, lda=None, ldb=None):
        a = torch.empty(M, lda or K, dtype=torch.bfloat16, device=dev)
        b = torch.empty(K, ldb or N, dtype=torch.bfloat16, device=dev)
        c = torch.empty(M, N, dtype=torch.float32, device=dev)
        return plan.query(a, b, c, M, N, K)
    assert q(8192, 8192, 8192)["kernel"] == g.GEMM_KERNEL_PAIR
    assert q(8192, 8192, 8192)["block_n"] == 256
    r = q(1023, 1000, 1029)                     # odd ldb: B staged, then TMA-fed split pairs
    assert r["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR and r["staged"] == 2, r
    r = q(1100, 4096, 4100, ldb=4101)           # a 33.6 MB B does not fit the staging buffer
    assert r["kernel"] == g.GEMM_KERNEL_GENERIC and r["staged"] == 0, r
    s = q(16, 4096, 14336)
    # 56 strips of 256 columns, K halved over the two CTAs of each cluster.
    assert s["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR and s["block_m"] == 16, s
    assert s["block_n"] == 256 and s["split_k"] == 2 and s["tiles"] == 56, s
    s = q(16, 4096, 4096)
    # 32 tiles of 128 columns: stream-K shares put every SM on the stream.
    assert s["kernel"] == g.GEMM_KERNEL_SKINNY and s["block_m"] == 16, s
    # Tile shape by estimated time: pair tiles once their waves are cheaper than
    # one-CTA tiles' (few K-long tiles), 128 x 128 one-CTA tiles for small ones.
    for shape, kern, bn in [((2048, 8192, 2048), g.GEMM_KERNEL_PAIR, 256),
                            ((512, 8192, 8192), g.GEMM_KERNEL_PAIR, 256),
                            ((1536, 1536, 1536), g.GEMM_KERNEL_TMA, 128),
                            ((128, 8192, 8192), g.GEMM_KERNEL_SPLIT_PAIR, 128),
                            ((1024, 8192, 1024), g.GEMM_KERNEL_SPLIT_PAIR, 128),
                            ((1024, 512, 1024), g.GEMM_KERNEL_TMA, 64)]:
        r = q(*shape)
        assert r["kernel"] == kern and r["block_n"] == bn, (shape, r)
    assert q(4096, 1024, 4096)["shares"] == 0       # 16 K blocks: no stream-K phase
    t = q(16, 4096, 4864)    # 38 tiles: stream-K spreads them over the SMs
    assert t["shares"] > 38 and t["split_k"] > 1, t
    assert q(64, 512, 512)["kernel"] == g.GEMM_KERNEL_SKINNY
    assert q(65, 512, 512)["kernel"] == g.GEMM_KERNEL_TMA
