"""GPU parity of the row-wise softmax (through the C ABI) against the binary64 oracle.

Tolerance, derived from the fp32 arithmetic of the kernels (u = 2^-24):
  * exp(x - m) is evaluated as exp2f((x - m) * log2(e)): the two roundings of
    the argument give a relative error <= 2u |x - m| in the result, exp2f is
    within 2 ulp (relative 4u), and y = e * (1 / s) rounds twice (2u);
  * the row sum is a chain of at most k fp32 additions (each thread's own
    elements in order -- at most ceil(N / threads) + 3 of them are not zero --
    then a butterfly over the threads of the row) and, on the
    two-pass path, one rescale (an expf and a multiply, <= 5u) per 16-element
    slab; its relative error is at most k u plus the weighted mean of the
    summands' own errors, sum_j y_j (2u |x_j - m| + 4u).
So |y - y*| <= u y* (2 |x - m| + 2 sum_j y*_j |x_j - m| + k + 12) + 2^-126 (the
last term covers results below fp32's normal range).
"""
import math

import numpy as np
import pytest
import torch

import dense_gemm_05_gb300 as g
import workloads
from oracle import softmax as osm

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
SENTINEL = -7.25


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()


def chain_bound(cfg, N):
    tpr = cfg["threads_per_row"]
    k = math.ceil(N / tpr) + 4 + math.ceil(math.log2(tpr))
    if cfg["path"] == g.SOFTMAX_PATH_STREAM:
        k += 5 * math.ceil(N / (tpr * 16))
    return k


def assert_softmax_close(got, X, N, cfg, what):
    x = np.asarray(X, dtype=np.float64)[:, :N]
    ref = osm.softmax_rows(X, N)
    finite_rows = np.all(np.isfinite(ref), axis=1)
    with np.errstate(invalid="ignore"):
        m = np.max(x, axis=1, keepdims=True)
        dist = np.where(np.isfinite(x), np.abs(x - m), 0.0)
    wmean = np.sum(np.where(np.isfinite(ref), ref, 0.0) * dist, axis=1, keepdims=True)
    tol = U * ref * (2 * dist + 2 * wmean + chain_bound(cfg, N) + 12) + 2.0 ** -126
    ok = np.where(finite_rows[:, None], np.abs(got - ref) <= tol, np.isnan(got))
    if not ok.all():
        i, j = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} entries off; first ({i}, {j}): "
                             f"gpu {got[i, j]!r} oracle {ref[i, j]!r} tol {tol[i, j]!r}")


def run(X, N, ldy=None, extra_rows=2):
    """X: CPU float32 (M, ldx).  Returns (Y buffer as float64 numpy, config)."""
    dev = torch.device("cuda:0")
    M, ldx = X.shape
    ldy = N if ldy is None else ldy
    x = X.to(dev)
    ybuf = torch.full((M + extra_rows, max(ldy, 1)), SENTINEL, dtype=torch.float32, device=dev)
    cfg = g.softmax_rows_query(x.data_ptr(), ldx, ybuf.data_ptr(), ldy, M, N)
    st = g.softmax_rows(x.data_ptr(), ldx, ybuf.data_ptr(), ldy, M, N,
                        torch.cuda.current_stream().cuda_stream)
    assert st == g.GEMM_OK, g.status_string(st)
    torch.cuda.synchronize()
    return ybuf.cpu().double().numpy(), cfg


def assert_guards(ybuf, M, N):
    assert np.all(ybuf[:M, N:] == SENTINEL), "a store landed right of column N"
    assert np.all(ybuf[M:] == SENTINEL), "a store landed below row M"


def test_demo_shape_full():
    """The chapter's demo input shape (128 x 1000, N(0,1))."""
    X = workloads.make_rows("softmax128x1000_f32")
    y, cfg = run(X, 1000)
    assert cfg["path"] == g.SOFTMAX_PATH_WARP and cfg["vec"] == 4, cfg
    assert_guards(y, 128, 1000)
    assert_softmax_close(y[:128, :1000], X, 1000, cfg, "128x1000")


SWEEP_N = [1, 2, 3, 5, 31, 32, 33, 127, 128, 129, 255, 1000, 1023, 1024, 1025, 2047, 2048,
           2049, 4095, 4097, 8191, 9000, 16385, 24576, 24577, 32768, 32769, 40000, 70001]


@pytest.mark.parametrize("N", SWEEP_N)
@pytest.mark.parametrize("layout", ["contiguous", "padded16", "unaligned"])
def test_lengths_and_layouts(N, layout):
    """Every path (warp / CTA / two-pass), 16-byte and 4-byte accesses, ragged tails."""
    M = 37 if N <= 4096 else 5
    if layout == "contiguous":
        ldx, ldy = N, N
    elif layout == "padded16":
        ldx, ldy = -(-N // 4) * 4 + 4, -(-N // 4) * 4 + 8
    else:
        ldx, ldy = N + 3, N + 1
    X = workloads.custom_rows(M, N, seed=N + 11 * len(layout), scale=3.0, ld=ldx)
    y, cfg = run(X, N, ldy=ldy)
    want_vec = 4 if (ldx % 4 == 0 and ldy % 4 == 0) else 1
    assert cfg["vec"] == want_vec, cfg
    want_path = (g.SOFTMAX_PATH_WARP if N <= 2048 else
                 g.SOFTMAX_PATH_CTA if N <= 32768 else g.SOFTMAX_PATH_STREAM)
    assert cfg["path"] == want_path, cfg
    assert cfg["staged"] == int(ldx % 4 == 0 and 8192 < N <= 24576), cfg
    assert_guards(y, M, N)
    assert_softmax_close(y[:M, :N], X, N, cfg, f"N={N} {layout}")


@pytest.mark.parametrize("N", [1000, 4096, 50000])
def test_in_place(N):
    M = 9
    X = workloads.custom_rows(M, N, seed=5, scale=2.0)
    x = X.cuda()
    cfg = g.softmax_rows_query(x.data_ptr(), N, x.data_ptr(), N, M, N)
    g.softmax(x, out=x)
    torch.cuda.synchronize()
    assert_softmax_close(x.cpu().double().numpy(), X, N, cfg, f"in place N={N}")


@pytest.mark.parametrize("N", [7, 1000, 5000, 40000])
def test_special_values(N):
    """-inf entries weigh nothing; a row of -inf, a row with +inf and a row with a
    NaN come out NaN; huge and constant rows."""
    X = workloads.custom_rows(6, N, seed=17, scale=1.0)
    X[0, ::3] = -math.inf                 # masked positions (a causal-mask pattern)
    X[1, :] = -math.inf                   # fully masked row
    X[2, N // 2] = math.inf
    X[3, N - 1] = math.nan
    X[4, :] = 3.5                         # constant row
    X[5, N // 3] = 1e30                   # one-hot limit
    y, cfg = run(X, N)
    assert_softmax_close(y[:6, :N], X, N, cfg, f"special N={N}")
    assert np.all(y[0, ::3] == 0.0)
    assert np.all(np.isnan(y[1, :N])) and np.all(np.isnan(y[2, :N])) and np.all(np.isnan(y[3, :N]))
    assert y[5, N // 3] == 1.0


def test_repeatable_bits():
    X = workloads.custom_rows(64, 3000, seed=2)
    a, _ = run(X, 3000)
    b, _ = run(X, 3000)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("name", ["softmax65536x1000_f32", "softmax4096x32768_f32"])
def test_full_size_sampled(name):
    """The measured workloads, launched exactly as bench.py launches them: sampled
    rows (first, last and random) against the oracle, every row's sum near 1."""
    w = workloads.SOFTMAX_WORKLOADS[name]
    X = workloads.make_rows(w)
    x = X.cuda()
    y = g.softmax(x)
    torch.cuda.synchronize()
    cfg = g.softmax_rows_query(x.data_ptr(), w.N, y.data_ptr(), w.N, w.M, w.N)
    rng = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([[0, 1, w.M - 1], rng.integers(0, w.M, 96)]))
    got = y[torch.from_numpy(rows).cuda()].cpu().double().numpy()
    assert_softmax_close(got, X[torch.from_numpy(rows)], w.N, cfg, name)
    # Every row: sum_j y_j = 1 + sum_j y*_j d_j with |d_j| <= u (2|x_j - m| + 2 wmean + k + 12),
    # and |x - m| < 14 for N(0,1) rows of these lengths (so wmean < 14 too).
    sums = y.double().sum(dim=1).cpu().numpy()
    bound = (56 + chain_bound(cfg, w.N) + 12) * U
    assert np.all(np.abs(sums - 1.0) <= bound), np.abs(sums - 1).max()


def test_device_errors():
    dev = torch.device("cuda:0")
    x = torch.randn(4, 64, device=dev)
    y = torch.empty(4, 64, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    assert g.softmax_rows(x.data_ptr() + 2, 64, y.data_ptr(), 64, 4, 63, s) == g.GEMM_ERR_INVALID_ARG
    assert g.softmax_rows(x.data_ptr(), 64, x.data_ptr() + 4, 64, 4, 63, s) == g.GEMM_ERR_INVALID_ARG
    assert g.softmax_rows(x.data_ptr(), 64, y.data_ptr(), 64, 4, 64, s) == g.GEMM_OK
    with pytest.raises(TypeError):
        g.softmax(x.double())
    torch.cuda.synchronize()


# ---------------------------------------------------------------- maximum sizes

PERIOD = 65537   # prime: an offset that wrapped at a power of two reads a different element


def _periodic_rows(M, N, seed):
    """X (on the GPU, M x N contiguous) whose flat element i is blk[i mod PERIOD],
    blk drawn N(0, 1) in float32; returns (blk as numpy, X)."""
    gen = torch.Generator().manual_seed(seed)
    blk = torch.randn(PERIOD, generator=gen)
    x = blk.cuda().repeat(-(-(M * N) // PERIOD))[: M * N].view(M, N)
    return blk.numpy(), x


def _row_of(blk, N, r):
    start = (r * N) % PERIOD
    return np.tile(np.roll(blk, -start), -(-N // PERIOD) + 1)[:N]


@pytest.mark.parametrize("M,N", [(2_200_007, 1000), (65_600, 32_768), (17, (1 << 27) + 5)],
                         ids=["warp-path", "cta-path", "two-pass-path"])
def test_inputs_beyond_2_31_elements(M, N):
    """More than 2^31 elements in X and Y (8.6-9.1 GB each), one case per path:
    sampled rows (first, last, the first row past element 2^31, random) against
    the oracle, and every row's sum near 1."""
    blk, x = _periodic_rows(M, N, seed=61)
    y = g.softmax(x)
    torch.cuda.synchronize()
    cfg = g.softmax_rows_query(x.data_ptr(), N, y.data_ptr(), N, M, N)
    rng = np.random.default_rng(62)
    first = -(-(1 << 31) // N)
    assert first < M
    extra = rng.integers(0, M, 12 if N < (1 << 20) else 0)
    rows = np.unique(np.concatenate([[0, M - 1, first], extra])).astype(np.int64)
    for r in rows:
        got = y[int(r)].double().cpu().numpy()[None, :]
        assert_softmax_close(got, _row_of(blk, N, int(r))[None, :], N, cfg, f"{M} x {N} row {r}")
    spread = float(blk.max() - blk.min())         # bounds |x - m| and its weighted mean
    bound = (4 * spread + chain_bound(cfg, N) + 12) * U
    sums = y.sum(dim=1, dtype=torch.float64).cpu().numpy()
    assert np.all(np.abs(sums - 1.0) <= bound), np.abs(sums - 1.0).max()
    del x, y
    torch.cuda.empty_cache()
