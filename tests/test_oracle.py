"""Pins of the CPU oracle against what the pages and the mathematics fix (CPU only).

Every pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a swapped index, a transposed operand, a bad 16-bit decode) fails
at least one of them.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads


def f16(rows):
    return torch.tensor(rows, dtype=torch.float32).to(torch.float16)


def bf16(rows):
    return torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)


# ---------------------------------------------------------------- 16-bit decoding

def test_f16_decode_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode(int(b), oracle.F16) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_every_pattern_matches_torch():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode(b, oracle.BF16) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- worked examples

@pytest.mark.parametrize("mk", [f16, bf16])
def test_worked_2x2(golden, mk):
    g = golden("matmul_2x2.txt")
    C = oracle.gemm(mk(g["A"]), mk(g["B"]))
    assert np.array_equal(C, np.array(g["C"], dtype=np.float64))


@pytest.mark.parametrize("mk", [f16, bf16])
def test_worked_4x4(golden, mk):
    g = golden("matmul_4x4.txt")
    C = oracle.gemm(mk(g["A"]), mk(g["B"]))
    assert np.array_equal(C, np.array(g["C"], dtype=np.float64))
    # B is not symmetric: a transposed operand gives a different product.
    Ct = oracle.gemm(mk(g["A"]), mk(np.array(g["B"]).T.tolist()))
    assert not np.array_equal(Ct, C)


def test_k_split_rounds(golden):
    """Section 3.3: the two K rounds of program (0, 0) and their sum."""
    g4 = golden("matmul_4x4.txt")
    gk = golden("ksplit_program00.txt")
    A = np.array(g4["A"])
    B = np.array(g4["B"])
    r1 = oracle.gemm(f16(A[0:2, 0:2].tolist()), f16(B[0:2, 0:2].tolist()))
    r2 = oracle.gemm(f16(A[0:2, 2:4].tolist()), f16(B[2:4, 0:2].tolist()))
    assert np.array_equal(r1, np.array(gk["ROUND1"], dtype=np.float64))
    assert np.array_equal(r2, np.array(gk["ROUND2"], dtype=np.float64))
    assert np.array_equal(r1 + r2, np.array(gk["ACC"], dtype=np.float64))
    full = oracle.gemm(f16(g4["A"]), f16(g4["B"]))
    assert np.array_equal(full[0:2, 0:2], np.array(gk["ACC"], dtype=np.float64))


def test_offsets_select_rows_and_ks(golden):
    """Section 4.3: offset = row * K + k picks A[2:4, 0:2] = [[9, 10], [13, 14]].

    The oracle is driven with B = columns of the identity that pick k = 0, 1, so
    C = A[:, ks]; its rows 2 and 3 must be the printed values (a transposed index
    would give [[3, 7], [4, 8]] instead)."""
    g4 = golden("matmul_4x4.txt")
    go = golden("offsets_program10.txt")
    rows, ks = go["ROWS"][0], go["KS"][0]
    K = 4
    offs = np.array(rows)[:, None] * K + np.array(ks)[None, :]
    assert np.array_equal(offs, np.array(go["OFFSETS"]))
    flat = np.array(g4["A"]).reshape(-1)
    assert np.array_equal(flat[offs], np.array(go["VALUES"]))
    sel = np.zeros((K, len(ks)))
    for j, k in enumerate(ks):
        sel[k, j] = 1.0
    C = oracle.gemm(f16(g4["A"]), f16(sel.tolist()))
    assert np.array_equal(C[rows, :], np.array(go["VALUES"], dtype=np.float64))


def test_load_tiles_program00(golden):
    """Section 4.4: program (0, 0), in its first K step, loads A[0:2, 0:2] and B[0:2, 0:2]."""
    g4 = golden("matmul_4x4.txt")
    gl = golden("load_program00.txt")
    A = np.array(g4["A"]).reshape(-1)
    B = np.array(g4["B"]).reshape(-1)
    rows = cols = np.array([0, 1])
    ks = np.array([0, 1])
    a_off = rows[:, None] * 4 + ks[None, :]
    b_off = ks[:, None] * 4 + cols[None, :]
    assert np.array_equal(a_off, np.array(gl["A_OFFSETS"]))
    assert np.array_equal(b_off, np.array(gl["B_OFFSETS"]))
    assert np.array_equal(A[a_off], np.array(gl["A_TILE"]))
    assert np.array_equal(B[b_off], np.array(gl["B_TILE"]))
    r1 = oracle.gemm(f16(A[a_off].tolist()), f16(B[b_off].tolist()))
    assert np.array_equal(r1, np.array(golden("ksplit_program00.txt")["ROUND1"], dtype=float))


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_and_zero(dtype):
    A, B = workloads.custom(37, 41, 29, dtype, seed=11)
    eyeK = torch.eye(41, dtype=A.dtype)
    assert np.array_equal(oracle.gemm(A, eyeK), A.to(torch.float64).numpy())
    eyeM = torch.eye(37, dtype=A.dtype)
    assert np.array_equal(oracle.gemm(eyeM, A), A.to(torch.float64).numpy())
    Z = torch.zeros(41, 29, dtype=A.dtype)
    assert np.array_equal(oracle.gemm(A, Z), np.zeros((37, 29)))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (17, 33, 9), (64, 129, 65)])
def test_small_integer_product_is_exact(dtype, shape):
    M, K, N = shape
    g = torch.Generator().manual_seed(M * 1000 + K * 10 + N)
    Ai = torch.randint(-4, 5, (M, K), generator=g)
    Bi = torch.randint(-4, 5, (K, N), generator=g)
    td = torch.float16 if dtype == "f16" else torch.bfloat16
    exact = Ai.numpy().astype(np.int64) @ Bi.numpy().astype(np.int64)
    C = oracle.gemm(Ai.to(td), Bi.to(td))
    assert np.array_equal(C, exact.astype(np.float64))


def test_sign_pin():
    """A negative entry must subtract: [[1, -2]] @ [[3], [4]] = -5."""
    assert oracle.gemm(f16([[1, -2]]), f16([[3], [4]]))[0, 0] == -5.0


@pytest.mark.parametrize("bs", [1, 2, 3, 4, 7, 16, 100])
def test_blockwise_equals_naive_on_integers(bs):
    g = torch.Generator().manual_seed(bs)
    Ai = torch.randint(-4, 5, (23, 31), generator=g).to(torch.float16)
    Bi = torch.randint(-4, 5, (31, 19), generator=g).to(torch.float16)
    assert np.array_equal(oracle.gemm_blockwise(Ai, Bi, bs), oracle.gemm(Ai, Bi))


def test_blockwise_4x4_by_hand(golden):
    """Step 2 of the first page: the blockwise loop on the 4x4 example with 2x2 tiles."""
    g = golden("matmul_4x4.txt")
    C = oracle.gemm_blockwise(f16(g["A"]), f16(g["B"]), 2)
    assert np.array_equal(C, np.array(g["C"], dtype=np.float64))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_matches_torch_float64_matmul(dtype):
    """Library cross-check: torch.matmul in float64 on the same rounded inputs."""
    A, B = workloads.custom(70, 45, 50, dtype, seed=5, dist="normal")
    ref = (A.to(torch.float64) @ B.to(torch.float64)).numpy()
    C = oracle.gemm(A, B)
    bnd = oracle.absbound(A, B)
    assert np.all(np.abs(C - ref) <= 1e-12 * bnd + 1e-300)


def test_absbound_is_product_of_absolute_values():
    A, B = workloads.custom(33, 65, 17, "bf16", seed=7, dist="normal")
    bnd = oracle.absbound(A, B)
    assert np.array_equal(bnd, oracle.gemm(A.abs(), B.abs()))
    assert np.all(np.abs(oracle.gemm(A, B)) <= bnd)


def test_entries_match_full_product():
    A, B = workloads.custom(40, 77, 53, "f16", seed=3)
    C = oracle.gemm(A, B)
    bnd = oracle.absbound(A, B)
    rng = np.random.default_rng(0)
    r = rng.integers(0, 40, 200)
    c = rng.integers(0, 53, 200)
    v, b = oracle.gemm_entries(A, B, r, c)
    assert np.array_equal(v, C[r, c])
    assert np.allclose(b, bnd[r, c], rtol=1e-15, atol=0)


def test_padded_leading_dimensions():
    """Row-major storage with lda > K, ldb > N: padding (NaN) is never read."""
    w = workloads.WORKLOADS["ragged1023x1000x1029_f16"]
    A, B = workloads.custom(45, 37, 29, "f16", seed=9)
    Ap, Bp = workloads.custom(45, 37, 29, "f16", seed=9, lda=48, ldb=40)
    assert torch.isnan(Ap[:, 37:].float()).all() and torch.isnan(Bp[:, 29:].float()).all()
    C = oracle.gemm(A, B)
    Cp = oracle.gemm(Ap, Bp, K=37, N=29)
    assert np.array_equal(C, Cp)
    assert w.K == 1000


def test_empty_sizes():
    A = torch.zeros(5, 0, dtype=torch.float16)
    B = torch.zeros(0, 7, dtype=torch.float16)
    assert np.array_equal(oracle.gemm(A, B), np.zeros((5, 7)))
    assert oracle.gemm(torch.zeros(0, 4, dtype=torch.float16),
                       torch.zeros(4, 3, dtype=torch.float16)).shape == (0, 3)
    assert oracle.gemm(torch.zeros(2, 4, dtype=torch.float16),
                       torch.zeros(4, 0, dtype=torch.float16)).shape == (2, 0)


def test_thread_count_does_not_change_bits():
    A, B = workloads.custom(64, 300, 48, "bf16", seed=1, dist="normal")
    c1 = oracle.gemm(A, B, nthreads=1)
    c4 = oracle.gemm(A, B, nthreads=4)
    assert np.array_equal(c1, c4)


def test_k_order_is_ascending():
    """Summation-order pin: terms 1, 2^60, -2^60 (exact in bf16).  With k ascending
    (the naive loop's order) binary64 gives (1 + 2^60) - 2^60 = 0; k descending
    would give (-2^60 + 2^60) + 1 = 1."""
    A = bf16([[1.0, 2.0 ** 60, -(2.0 ** 60)]])
    B = bf16([[1.0], [1.0], [1.0]])
    assert oracle.gemm(A, B)[0, 0] == 0.0
    v, _ = oracle.gemm_entries(A, B, [0], [0])
    assert v[0] == 0.0


def test_tolerance_mask():
    ok = oracle.within_tolerance([1.0 + 5e-4, 1.0 + 2e-3], [1.0, 1.0], [1.0, 1.0])
    assert ok.tolist() == [True, False]
