"""Failure paths of the real kernels, without a GPU fault (GPU).

Every spin-wait in the kernels is bounded.  A plan's wait limit can be set far
below a kernel's run time (gemm_plan_set_debug), which makes a real launch give
up part-way: its CTAs stop only after the copies and MMAs they have in flight
have landed, the status word is set, and in debug-sync mode gemm_run returns
GEMM_ERR_TIMEOUT.  The next GEMM on the same context, with the default limit,
must then match the oracle -- the context stays usable and no state (tile
counters, partial tiles) leaks into it.  Kernels covered: the 2-SM pair kernel
with its stream-K phase, the one-CTA kernel, the swap-AB stream-K kernel with
split tiles, and the split-K cluster kernel; and the attention kernel (both head dimensions).

The allocation path is tested on the host: GEMM_TEST_FAIL_ALLOC=k makes the
k-th device allocation of gemm_plan_create fail, which must return
GEMM_ERR_OOM and leave the device's free memory as it was.
"""
import os

import numpy as np
import pytest
import torch

import dense_gemm_05_gb300 as g
import oracle
import workloads

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-5
# 2 us: far below the longest wait of each of these launches (tens to hundreds
# of microseconds).  A wait gives up somewhat after its limit (a suspended poll
# resumes on the hardware's schedule), so a launch whose waits are all short
# (about 20 us at M = 16, N = 14336) may finish first; measured: 5 of 12.
SHORT_NS = 2000


@pytest.fixture(scope="module")
def plan():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()
    p = g.Plan(0)
    yield p
    p.close()


def check_sampled(c, A, B, M, N, K, seed):
    rng = np.random.default_rng(seed)
    rows = np.concatenate([rng.integers(0, M, 2048), [0, M - 1, 0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 2048), [0, 0, N - 1, N - 1]])
    ref, bound = oracle.gemm_entries(A, B, rows, cols)
    got = c.cpu().double().numpy()[rows, cols]
    ok = np.abs(got - ref) <= REL * bound + ABS
    assert ok.all(), f"{int((~ok).sum())} sampled entries outside tolerance"


@pytest.mark.parametrize("M,K,N,kernel,block_n", [
    (4096, 4096, 4096, g.GEMM_KERNEL_PAIR, 256),       # pair tiles + stream-K phase
    (1024, 8192, 1024, g.GEMM_KERNEL_TMA, 128),        # one-CTA tiles, 128 K blocks each
    (16, 32768, 4864, g.GEMM_KERNEL_SKINNY, 0),        # swap-AB stream-K, split tiles
    (16, 65536, 2048, g.GEMM_KERNEL_SPLIT_PAIR, 256),  # split-K clusters, 256-column strips
    (1000, 16384, 1000, g.GEMM_KERNEL_SPLIT_PAIR, 128),  # split-K clusters, 128-row tiles
])
def test_a_wait_that_runs_out_is_reported_and_the_context_survives(plan, M, K, N, kernel, block_n):
    A, B = workloads.custom(M, K, N, "bf16", seed=M + K + N, dist="normal")
    dev = torch.device("cuda:0")
    a, b = A.to(dev), B.to(dev)
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    plan.force(kernel, 0, block_n)
    try:
        assert plan.query(a, b, c)["kernel"] == kernel
        plan.set_debug(True, SHORT_NS)
        st = g.gemm_run(plan.handle, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, M, N, K,
                        g.GEMM_BF16, torch.cuda.current_stream().cuda_stream)
        assert st == g.GEMM_ERR_TIMEOUT, g.status_string(st)
        # default limit again (debug-sync kept, so a give-up would show): correct result
        plan.set_debug(True, 0)
        c.fill_(float("nan"))
        plan.run(a, b, c)
        torch.cuda.synchronize()
    finally:
        plan.set_debug(False, 0)
        plan.force(0, 0, 0)
    assert not torch.isnan(c).any(), "an entry of C was not written"
    check_sampled(c, A, B, M, N, K, seed=M + N)
    # and once more without debug-sync, through the normal asynchronous path
    c.fill_(float("nan"))
    plan.run(a, b, c)
    torch.cuda.synchronize()
    check_sampled(c, A, B, M, N, K, seed=M + N + 1)


@pytest.mark.parametrize("name", ["attn_bh16_s8192_d64_bf16_causal", "attn_bh16_s8192_d128_bf16_causal"])
def test_attention_wait_that_runs_out_is_reported_and_the_context_survives(plan, name):
    """The attention kernel's roles (the K and V producer lanes, the S and P V
    issuers, the softmax warpgroups): a 2 us limit makes a full-size launch give
    up; the next launch with the default limit must match the oracle."""
    from oracle import attention as oa
    w = workloads.ATTN_WORKLOADS[name]
    Q, K, V = workloads.make_qkv(w)
    dev = torch.device("cuda:0")
    q, k, v = Q.to(dev), K.to(dev), V.to(dev)
    o = torch.full((w.BH, w.seq, w.d), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    BH, seq, d = w.BH, w.seq, w.d
    try:
        assert g.attention_set_debug(1, SHORT_NS) == g.GEMM_OK
        st = g.attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), BH, seq, d, d,
                             seq * d, d, seq * d, int(w.causal), g.GEMM_BF16, 0, stream)
        assert st == g.GEMM_ERR_TIMEOUT, g.status_string(st)
        assert g.attention_set_debug(1, 0) == g.GEMM_OK      # default limit, still synchronous
        o.fill_(float("nan"))
        st = g.attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), BH, seq, d, d,
                             seq * d, d, seq * d, int(w.causal), g.GEMM_BF16, 0, stream)
        assert st == g.GEMM_OK, g.status_string(st)
    finally:
        g.attention_set_debug(-1, 0)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any(), "an entry of O was not written"
    for head in (0, BH - 1):
        rows = np.linspace(0, seq - 1, 48).astype(np.int64)
        ref = oa.attention_rows(Q, K, V, w.causal, head, rows)
        got = o[head].cpu().double().numpy()[rows]
        scale = np.abs(ref).max()
        assert np.abs(got - ref).max() <= 1e-2 * scale, f"head {head}"


def test_attention_debug_settings_are_checked():
    assert g.attention_set_debug(2, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.attention_set_debug(-2, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.attention_set_debug(-1, 0) == g.GEMM_OK


def test_debug_settings_are_checked(plan):
    assert g.gemm_plan_set_debug(plan.handle, 2, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_plan_set_debug(None, 1, 0) == g.GEMM_ERR_INVALID_ARG


def test_failed_allocation_returns_oom_and_leaks_nothing(plan):
    torch.cuda.synchronize()
    g.Plan(0).close()                      # warm: kernels loaded, context settled
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    try:
        for k in (1, 2, 3, 4):
            os.environ["GEMM_TEST_FAIL_ALLOC"] = str(k)
            with pytest.raises(g.GemmError) as e:
                g.Plan(0)
            assert e.value.status == g.GEMM_ERR_OOM, k
            torch.cuda.synchronize()
            free, _ = torch.cuda.mem_get_info()
            assert free == free0, f"allocation {k}: {free0 - free} bytes not returned"
    finally:
        del os.environ["GEMM_TEST_FAIL_ALLOC"]
    p = g.Plan(0)                          # and a plan can be made again
    p.close()
