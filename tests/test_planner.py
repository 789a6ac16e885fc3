"""The planner (argument checks, staging decision, kernel and configuration
choice) on a modelled GB300, without a GPU: gemm_plan_create_model gives a plan
with the device facts a GB300 reports (152 SMs, 76 co-resident 2-CTA clusters)
and the capacities of a device plan, and gemm_query / gemm_query_ex answer on it
exactly as on a device plan.  Pointers are fake addresses (only alignment and
overlap are checked)."""
import pytest

import dense_gemm_05_gb300 as g

A_ADDR, B_ADDR, C_ADDR = 1 << 40, 2 << 40, 3 << 40


@pytest.fixture(scope="module")
def model():
    g.build()
    h = g.gemm_plan_create_model()
    yield h
    g.gemm_plan_destroy(h)


def q(h, M, N, K, lda=None, ldb=None, ldc=None, dtype=g.GEMM_BF16, a_off=0, b_off=0):
    return g.gemm_query(h, A_ADDR + a_off, K if lda is None else lda, B_ADDR + b_off,
                        N if ldb is None else ldb, C_ADDR, N if ldc is None else ldc,
                        M, N, K, dtype)


def qx(h, op_a, op_b, M, N, K, c_type=g.GEMM_OUT_F32):
    lda = K if op_a == g.GEMM_OP_N else M
    ldb = N if op_b == g.GEMM_OP_N else K
    return g.gemm_query_ex(h, op_a, op_b, A_ADDR, lda, B_ADDR, ldb, C_ADDR, N, c_type, M, N, K,
                           g.GEMM_BF16)


def test_the_five_workloads(model):
    """The choices measured in the bench, pinned."""
    r = q(model, 8192, 8192, 8192)
    assert (r["kernel"], r["block_m"], r["block_n"], r["grid"], r["cluster"]) == \
        (g.GEMM_KERNEL_PAIR, 256, 256, 152, 2), r
    assert r["shares"] == 76 and r["split_k"] >= 2, r      # stream-K phase for the partial wave
    r = q(model, 4096, 4096, 4096)
    assert r["kernel"] == g.GEMM_KERNEL_PAIR and r["block_n"] == 256 and r["shares"] == 76, r
    # the stream-K phase by last-wave fill and full waves (576, 196, 441 tiles on 76 pairs)
    assert q(model, 6144, 6144, 6144)["shares"] == 76        # 58% full behind 7 waves
    assert q(model, 3584, 3584, 3584)["shares"] == 0         # 58% behind 2
    assert q(model, 5376, 5376, 5376)["shares"] == 0         # 80% behind 5
    r = q(model, 16, 14336, 4096)
    assert (r["kernel"], r["block_m"], r["block_n"], r["grid"], r["split_k"], r["tiles"]) == \
        (g.GEMM_KERNEL_SPLIT_PAIR, 16, 256, 112, 2, 56), r
    r = q(model, 256, 256, 256, dtype=g.GEMM_F16)       # 64 x 64 tiles (M = 64 MMAs): 16 CTAs
    assert (r["kernel"], r["block_m"], r["block_n"], r["grid"], r["tiles"]) == \
        (g.GEMM_KERNEL_TMA, 64, 64, 16, 16), r
    r = q(model, 1023, 1029, 1000, dtype=g.GEMM_F16)      # tight pitches: ldb = 1029 halves
    assert (r["kernel"], r["block_m"], r["block_n"], r["grid"], r["staged"]) == \
        (g.GEMM_KERNEL_SPLIT_PAIR, 128, 128, 144, 2), r


def test_degenerate_sizes(model):
    assert q(model, 0, 100, 100)["kernel"] == g.GEMM_KERNEL_NONE
    assert q(model, 100, 0, 100)["kernel"] == g.GEMM_KERNEL_NONE
    r = q(model, 100, 100, 0)
    assert r["kernel"] == g.GEMM_KERNEL_ZERO_FILL and r["block_k"] == 0, r


SHAPES = [(m, n, k) for m in (1, 16, 17, 33, 64, 65, 128, 300, 1023, 2048, 4096)
          for n in (1, 100, 1000, 4096, 14336) for k in (1, 64, 500, 1024, 4096)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_every_choice_is_consistent(model, M, N, K):
    r = q(model, M, N, K, lda=(K + 7) // 8 * 8, ldb=(N + 7) // 8 * 8, ldc=N)
    k = r["kernel"]
    assert k in (g.GEMM_KERNEL_TMA, g.GEMM_KERNEL_PAIR, g.GEMM_KERNEL_SKINNY,
                 g.GEMM_KERNEL_SPLIT_PAIR), r          # aligned operands: never GENERIC
    assert r["block_k"] == 64 and r["stages"] >= 2 and r["grid"] >= 1, r
    assert r["cluster"] == (2 if k in (g.GEMM_KERNEL_PAIR, g.GEMM_KERNEL_SPLIT_PAIR) else 1), r
    if k == g.GEMM_KERNEL_SPLIT_PAIR:
        assert r["grid"] == 2 * r["tiles"] and r["split_k"] == 2, r
        if M <= 64:
            assert r["block_m"] in (16, 32, 64) and r["block_m"] >= M, r
            assert r["tiles"] == -(-N // r["block_n"]), r
        else:
            assert r["block_m"] == 128 and r["block_n"] == 128, r
            assert r["tiles"] == -(-M // 128) * -(-N // 128) and r["tiles"] <= 76, r
        assert K >= 128, r                              # both halves of K non-empty
    elif k == g.GEMM_KERNEL_SKINNY:
        assert M <= 64 and r["block_n"] == 128 and r["grid"] <= 152, r
    elif k == g.GEMM_KERNEL_PAIR:
        assert M > 64 and r["block_m"] == 256 and r["grid"] <= 152 and r["grid"] % 2 == 0, r
    else:
        assert r["grid"] <= 152 and r["block_m"] in (64, 128), r
        if r["block_m"] == 64:                         # 64 x 64 tiles, one wave, small problems
            assert r["block_n"] == 64 and r["tiles"] == -(-M // 64) * -(-N // 64) <= 152, r
            assert 2 * -(-M // 128) * -(-N // 64) <= 152, r
    if M <= 64:
        assert k in (g.GEMM_KERNEL_SKINNY, g.GEMM_KERNEL_SPLIT_PAIR), r


def test_operand_layouts(model):
    # a transposed A with M <= 64 cannot use the small-M kernels (they read A K-major)
    assert qx(model, g.GEMM_OP_T, g.GEMM_OP_N, 16, 14336, 4096)["kernel"] == g.GEMM_KERNEL_TMA
    # the weight layout for B is fine for both
    assert qx(model, g.GEMM_OP_N, g.GEMM_OP_T, 16, 14336, 4096)["kernel"] == \
        g.GEMM_KERNEL_SPLIT_PAIR
    assert qx(model, g.GEMM_OP_N, g.GEMM_OP_T, 16, 4096, 4096)["kernel"] == g.GEMM_KERNEL_SKINNY
    r = qx(model, g.GEMM_OP_T, g.GEMM_OP_T, 8192, 8192, 8192, g.GEMM_OUT_BF16)
    assert r["kernel"] == g.GEMM_KERNEL_PAIR, r


def test_staging_decisions(model):
    # odd pitches that fit the 32 MiB staging buffer are staged for the TMA kernels
    r = q(model, 1000, 1000, 1000, lda=1001, ldb=1003, dtype=g.GEMM_F16)
    assert r["staged"] == 3 and r["kernel"] != g.GEMM_KERNEL_GENERIC, r
    # a misaligned base pointer is staged too
    assert q(model, 1000, 1000, 1000, a_off=2)["staged"] == 1
    # a 33.6 MB B does not fit, and 528 tiles are too many for the split-pair
    # kernel: the generic kernel reads both in place
    r = q(model, 2000, 4100, 4096, ldb=4101)
    assert r["kernel"] == g.GEMM_KERNEL_GENERIC and r["staged"] == 0, r
    # with 66 tiles the split-pair kernel takes it and reads B in place
    r = q(model, 200, 4100, 4096, ldb=4101)
    assert (r["kernel"], r["staged"]) == (g.GEMM_KERNEL_SPLIT_PAIR, 4), r
    # split-pair-sized problems (M > 64, one wave of 128 x 128 tiles, K >= 768) with
    # an aligned A: a misaligned B that fits the buffer is staged ...
    r = q(model, 1000, 1000, 4096, ldb=1001, dtype=g.GEMM_F16)
    assert (r["kernel"], r["staged"]) == (g.GEMM_KERNEL_SPLIT_PAIR, 2), r
    # ... one that does not is read in place
    r = q(model, 300, 1100, 20000, ldb=1103)           # B of 44 MB
    assert (r["kernel"], r["staged"]) == (g.GEMM_KERNEL_SPLIT_PAIR, 4), r
    # never with a misaligned A, small M or a transposed B
    r = q(model, 300, 1100, 20000, lda=20001, ldb=1103)
    assert r["staged"] & 4 == 0, r
    assert q(model, 64, 4100, 4096, ldb=4101)["staged"] & 4 == 0
    r = g.gemm_query_ex(model, g.GEMM_OP_N, g.GEMM_OP_T, A_ADDR, 4096, B_ADDR, 4097, C_ADDR,
                        1000, g.GEMM_OUT_F32, 1000, 1000, 4096, g.GEMM_BF16)
    assert r["staged"] & 4 == 0, r


def test_staging_off(model):
    # with staging off nothing is copied: the split-pair kernel reads B in place
    # where it can, the generic kernel takes the rest
    assert g.gemm_plan_set_staging(model, 0) == g.GEMM_OK
    try:
        r = q(model, 1023, 1029, 1000, dtype=g.GEMM_F16)
        assert (r["kernel"], r["staged"]) == (g.GEMM_KERNEL_SPLIT_PAIR, 4), r
        r = q(model, 1000, 1000, 1000, lda=1001, ldb=1003, dtype=g.GEMM_F16)
        assert (r["kernel"], r["staged"]) == (g.GEMM_KERNEL_GENERIC, 0), r
    finally:
        assert g.gemm_plan_set_staging(model, 1) == g.GEMM_OK
    assert q(model, 1023, 1029, 1000, dtype=g.GEMM_F16)["staged"] == 2
    assert g.gemm_plan_set_staging(model, 2) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_plan_set_staging(None, 1) == g.GEMM_ERR_INVALID_ARG


def test_forcing(model):
    h = model
    try:
        assert g.gemm_plan_force(h, g.GEMM_KERNEL_SKINNY, 0, 0) == g.GEMM_OK
        with pytest.raises(g.GemmError):
            q(h, 65, 512, 512)                           # skinny needs M <= 64
        assert g.gemm_plan_force(h, g.GEMM_KERNEL_SPLIT_PAIR, 0, 192) == g.GEMM_OK
        assert q(h, 16, 14336, 4096)["block_n"] == 192
        with pytest.raises(g.GemmError):
            q(h, 65, 512, 4096)                          # 128-row tiles take 128 columns only
        assert g.gemm_plan_force(h, g.GEMM_KERNEL_TMA, 0, 192) == g.GEMM_OK
        with pytest.raises(g.GemmError):
            q(h, 1024, 1024, 1024)                       # 192 columns: split pair only
        assert g.gemm_plan_force(h, g.GEMM_KERNEL_PAIR, 1, 256) == g.GEMM_OK
        assert q(h, 4096, 4096, 4096)["shares"] == 0     # stream-K phase off
        assert g.gemm_plan_force(h, g.GEMM_KERNEL_SKINNY, 152, 0) == g.GEMM_OK
        r = q(h, 16, 14336, 4096)
        assert r["kernel"] == g.GEMM_KERNEL_SKINNY and r["shares"] == 152 and r["grid"] == 152, r
        assert g.gemm_plan_force(h, 99, 0, 0) == g.GEMM_ERR_INVALID_ARG
        assert g.gemm_plan_force(h, 0, 0, 96) == g.GEMM_ERR_INVALID_ARG
    finally:
        g.gemm_plan_force(h, 0, 0, 0)


def test_smaller_device_model():
    """Fewer SMs move the boundaries: 132 SMs and 66 clusters."""
    g.build()
    h = g.gemm_plan_create_model(132, 66, 66, 66)
    try:
        r = q(h, 16, 14336, 4096)
        assert r["kernel"] == g.GEMM_KERNEL_SPLIT_PAIR and r["grid"] == 112, r
        r = q(h, 8192, 8192, 8192)
        assert r["kernel"] == g.GEMM_KERNEL_PAIR and r["grid"] == 132, r
        r = q(h, 1023, 1029, 1000, dtype=g.GEMM_F16)     # 72 tiles > 66 clusters
        assert r["kernel"] != g.GEMM_KERNEL_SPLIT_PAIR, r
    finally:
        g.gemm_plan_destroy(h)


def test_model_plan_runs_nothing_and_rejects_bad_facts():
    g.build()
    h = g.gemm_plan_create_model()
    try:
        assert g.gemm_run(h, A_ADDR, 64, B_ADDR, 64, C_ADDR, 64, 64, 64, 64, g.GEMM_BF16, 0) == \
            g.GEMM_ERR_INVALID_ARG
    finally:
        assert g.gemm_plan_destroy(h) == g.GEMM_OK
    for facts in [(0, 0, 0, 0), (152, 77, 76, 76), (152, 76, -1, 76), (5000, 0, 0, 0)]:
        with pytest.raises(g.GemmError):
            g.gemm_plan_create_model(*facts)


@pytest.mark.parametrize("N,K", [(4096 * 128 + 128, 64), (50_000_008, 64), (600_000, 512)])
def test_small_m_many_tiles_short_k(model, N, K):
    """M <= 64 with more 128-column tiles than the stream-K share limit and K too
    short for the cluster kernel: one share per tile, which needs no workspace,
    so any number of tiles is accepted."""
    r = q(model, 16, N, K)
    tiles = -(-N // 128)
    assert (r["kernel"], r["tiles"], r["shares"], r["split_k"], r["grid"]) == \
        (g.GEMM_KERNEL_SKINNY, tiles, tiles, 1, 152), r
