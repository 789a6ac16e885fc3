"""GPU parity of the attention forward pass (through the C ABI) against the binary64 oracle.

Tolerance, derived from the kernel's arithmetic (u_t = 2^-8 for bf16 inputs,
2^-11 for fp16; u = 2^-24):
  * the weights P are rounded to the input type before P V while the row sum
    l adds the unrounded fp32 values: each weight p/l is off by at most u_t
    relatively;
  * a score s = q.k is an fp32 sum of d exact products: |ds| <= d u sum|q||k|;
    scaled by 1/sqrt(d) it moves every weight of its row by a factor
    exp(+-|ds|/sqrt(d)), i.e. 2 eps relatively with eps = max_j d u sum|q||k_j| / sqrt(d);
  * ex2.approx (relative 2^-22 per value), the fp32 row sum, the fp32 MMA
    sums of P V and the rescales add far less than 2^-12 relatively;
so |O - O*| <= (2 u_t + 2 eps + 2^-12) sum_j P*_j |V_j| (+ u_out |O*| for a
16-bit O, the one output rounding) + 1e-7.
"""
import math

import numpy as np
import pytest
import torch

import dense_gemm_05_gb300 as g
import workloads
from oracle import attention as oa

pytestmark = pytest.mark.gpu

U_IN = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
U_OUT = {torch.float32: 0.0, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build()


def dtype_name(t):
    return "bf16" if t.dtype == torch.bfloat16 else "f16"


def assert_attn_close(got, Q, K, V, causal, head, rows, out_dtype, what):
    """got: float64 numpy [len(rows), d] for head `head`."""
    rows = np.asarray(rows, dtype=np.int64)
    ref = oa.attention_rows(Q, K, V, causal, head, rows)
    wabs = oa.weight_abs_v(Q, K, V, causal, head, rows)
    q = Q[head].double().numpy()[rows]
    k = K[head].double().numpy()
    d = q.shape[1]
    qk = np.abs(q) @ np.abs(k).T
    if causal:
        qk = np.where(rows[:, None] >= np.arange(k.shape[0])[None, :], qk, 0.0)
    eps = d * 2.0 ** -24 * qk.max(axis=1, keepdims=True) / math.sqrt(d)
    tol = (2 * U_IN[dtype_name(Q)] + 2 * eps + 2.0 ** -12) * wabs + U_OUT[out_dtype] * np.abs(ref) + 1e-7
    err = np.abs(got - ref)
    ok = err <= tol
    if not ok.all():
        i, c = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} off; first row {rows[i]} col {c}: "
                             f"gpu {got[i, c]!r} oracle {ref[i, c]!r} tol {tol[i, c]!r}")


def run(Q, K, V, causal, out_dtype=torch.float32, layout="heads"):
    """Q, K, V: CPU [BH, seq, d].  layout 'heads' = contiguous [BH, seq, d];
    'interleaved' = stored [seq, BH, d]; 'padded' = rows padded to d + 8 elements."""
    dev = torch.device("cuda:0")
    BH, seq, d = Q.shape
    if layout == "heads":
        q, k, v = (t.to(dev) for t in (Q, K, V))
    elif layout == "interleaved":
        q, k, v = (t.transpose(0, 1).contiguous().to(dev).transpose(0, 1) for t in (Q, K, V))
    else:
        def pad(t):
            buf = torch.full((BH, seq, d + 8), float("nan"), dtype=t.dtype)
            buf[:, :, :d] = t
            return buf.to(dev)[:, :, :d]
        q, k, v = pad(Q), pad(K), pad(V)
    out = torch.full((BH, seq, d), float("nan"), dtype=out_dtype, device=dev)
    g.attention(q, k, v, causal=causal, out=out)
    torch.cuda.synchronize()
    return out.float().cpu().double().numpy()


@pytest.mark.parametrize("name", ["attn_bh2_s256_d64_f16_causal", "attn_bh2_s1000_d64_bf16"])
def test_small_workloads_full(name):
    w = workloads.ATTN_WORKLOADS[name]
    Q, K, V = workloads.make_qkv(w)
    got = run(Q, K, V, w.causal)
    for h in range(w.BH):
        assert_attn_close(got[h], Q, K, V, w.causal, h, np.arange(w.seq), torch.float32, f"{name} head {h}")


SEQS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 300, 513]


@pytest.mark.parametrize("seq", SEQS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_lengths(seq, causal, d):
    dt = "bf16" if seq % 2 else "f16"
    Q, K, V = workloads.custom_qkv(3, seq, d, dt, seed=seq * 3 + causal + d)
    got = run(Q, K, V, causal)
    assert np.all(np.isfinite(got))
    for h in range(3):
        assert_attn_close(got[h], Q, K, V, causal, h, np.arange(seq), torch.float32,
                          f"d {d} seq {seq} causal {causal} head {h}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_several_items_per_cta_with_ragged_tiles(d, causal):
    """More work items than SMs, so CTAs walk several items whose last query
    tile is ragged (seq 1100 = 8 tiles + 76 rows) and, for d = 64, whose
    second tile of the last pair lies beyond the sequence; every head against
    the oracle on a row sample that covers both edges."""
    BH, seq = 40, 1100
    Q, K, V = workloads.custom_qkv(BH, seq, d, "bf16" if causal else "f16", seed=77 + d + causal)
    items = BH * ((seq + 127) // 128 + (1 if d == 64 else 0)) // (2 if d == 64 else 1)
    assert items > torch.cuda.get_device_properties(0).multi_processor_count
    got = run(Q, K, V, causal)
    assert np.all(np.isfinite(got))
    rows = np.unique(np.concatenate([np.arange(0, 4), np.arange(1020, seq), np.arange(5, 1020, 97)]))
    for h in range(0, BH, 3):
        assert_attn_close(got[h][rows], Q, K, V, causal, h, rows, torch.float32,
                          f"d {d} causal {causal} head {h}")


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("layout", ["heads", "interleaved", "padded"])
@pytest.mark.parametrize("d", [64, 128])
def test_layouts_and_output_types(out_dtype, layout, d):
    Q, K, V = workloads.custom_qkv(4, 333, d, "bf16", seed=7 + d)
    got = run(Q, K, V, True, out_dtype=out_dtype, layout=layout)
    for h in range(4):
        assert_attn_close(got[h], Q, K, V, True, h, np.arange(333), out_dtype, f"{layout} {out_dtype} head {h}")


def test_fp32_output_layouts():
    Q, K, V = workloads.custom_qkv(3, 200, 64, "f16", seed=8)
    for layout in ("interleaved", "padded"):
        got = run(Q, K, V, False, layout=layout)
        for h in range(3):
            assert_attn_close(got[h], Q, K, V, False, h, np.arange(200), torch.float32, f"{layout} head {h}")


def test_closed_forms_on_gpu():
    """Constant V rows give O = that row; identical keys give (prefix) means of V."""
    Q, K, V = workloads.custom_qkv(2, 300, 64, "bf16", seed=9)
    Vc = torch.ones_like(V) * torch.linspace(-2, 2, 64).to(torch.bfloat16)
    got = run(Q, K, Vc, True)
    assert np.allclose(got, Vc.double().numpy(), rtol=2 ** -7, atol=1e-6)
    Ks = K[:, :1].expand(-1, 300, -1).contiguous()
    got = run(Q, Ks, V, True)
    prefix = np.cumsum(V.double().numpy(), axis=1) / np.arange(1, 301)[None, :, None]
    wabs = np.cumsum(np.abs(V.double().numpy()), axis=1) / np.arange(1, 301)[None, :, None]
    assert np.all(np.abs(got - prefix) <= (2 * 2 ** -8 + 2 ** -12) * wabs + 1e-6)


def test_repeatable_bits():
    Q, K, V = workloads.custom_qkv(2, 700, 64, "bf16", seed=10)
    a = run(Q, K, V, True)
    b = run(Q, K, V, True)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bits_do_not_depend_on_the_schedule(d, causal):
    """The launch is persistent (at most one CTA per SM, each walking several
    work items): a head computed alone and the same heads inside a 20-head
    batch (several items per CTA, other CTAs and places in their sequences) give
    identical bits."""
    BH, seq = 20, 4096
    Q, K, V = workloads.custom_qkv(BH, seq, d, "bf16", seed=31 + d + causal)
    items = BH * (seq // 128 // (2 if d == 64 else 1))
    assert items > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    batch = run(Q, K, V, causal)
    for h in (0, 7, BH - 1):
        alone = run(Q[h:h + 1], K[h:h + 1], V[h:h + 1], causal)
        assert np.array_equal(alone[0], batch[h]), h


@pytest.mark.parametrize("name", ["attn_bh16_s8192_d64_bf16_causal", "attn_bh16_s8192_d64_bf16",
                                  "attn_bh16_s8192_d128_bf16_causal"])
def test_full_size_sampled(name):
    """The measured workloads, launched as bench.py launches them: sampled rows of
    three heads (first and last rows of the sequence included) against the oracle;
    every output finite."""
    w = workloads.ATTN_WORKLOADS[name]
    Q, K, V = workloads.make_qkv(w)
    dev = torch.device("cuda:0")
    q, k, v = Q.to(dev), K.to(dev), V.to(dev)
    out = g.attention(q, k, v, causal=w.causal)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(w.seed)
    for h in (0, w.BH // 2, w.BH - 1):
        rows = np.unique(np.concatenate([[0, 1, 127, 128, w.seq - 1], rng.integers(0, w.seq, 48)]))
        got = out[h, torch.from_numpy(rows).to(dev)].double().cpu().numpy()
        assert_attn_close(got, Q, K, V, w.causal, h, rows, torch.float32, f"{name} head {h}")


def test_device_errors():
    dev = torch.device("cuda:0")
    q = torch.randn(2, 64, 64, device=dev).to(torch.bfloat16)
    o = torch.empty(2, 64, 64, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    st = g.attention_fwd(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 2, 64, 64, 64,
                         4096, 64, 4096, 0, g.GEMM_BF16, g.GEMM_OUT_BF16, s)
    assert st == g.GEMM_ERR_INVALID_ARG                       # O overlaps Q
    st = g.attention_fwd(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 2, 64, 64, 64,
                         4096, 64, 4096, 0, g.GEMM_BF16, g.GEMM_OUT_F32, s)
    assert st == g.GEMM_OK                                    # Q = K = V is fine
    with pytest.raises(TypeError):
        g.attention(q, q.half(), q)
    torch.cuda.synchronize()


# ---------------------------------------------------------------- maximum sizes

PERIOD = 65537   # prime: an offset that wrapped at a power of two reads a different element


@pytest.mark.parametrize("BH,seq,d,causal", [(65535, 512, 128, True), (65535, 640, 64, False)],
                         ids=["d128-causal", "d64"])
def test_most_heads_past_2_31_elements(BH, seq, d, causal):
    """BH at its limit (65535 heads, the grid's y extent), Q, K and V of 2.7e9-4.3e9
    elements each: flat element i of each is a block value at i mod PERIOD, so every
    head differs; sampled rows of the first, middle and last heads against the oracle."""
    gen = torch.Generator().manual_seed(71)
    blks = [torch.randn(PERIOD, generator=gen).to(torch.bfloat16) for _ in range(3)]
    dev = torch.device("cuda:0")
    n = BH * seq * d
    q, k, v = (b.to(dev).repeat(-(-n // PERIOD))[:n].view(BH, seq, d) for b in blks)
    out = g.attention(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(out).all())
    rng = np.random.default_rng(72)
    idx = np.arange(seq * d)
    for h in (0, BH // 2, BH - 1):
        head = [b[torch.from_numpy((h * seq * d + idx) % PERIOD)].view(1, seq, d) for b in blks]
        rows = np.unique(np.concatenate([[0, 1, 127, 128, seq - 1], rng.integers(0, seq, 8)]))
        got = out[h, torch.from_numpy(rows).to(dev)].double().cpu().numpy()
        assert_attn_close(got, *head, causal, 0, rows, torch.float32, f"{BH} heads, head {h}")
    del q, k, v, out
    torch.cuda.empty_cache()


def test_longest_sequence_sampled():
    """seq = 2^20 + 3 (ragged), causal, d = 64: 8193 key blocks for the last queries."""
    Q, K, V = workloads.custom_qkv(1, (1 << 20) + 3, 64, "bf16", seed=81)
    dev = torch.device("cuda:0")
    out = g.attention(Q.to(dev), K.to(dev), V.to(dev), causal=True)
    torch.cuda.synchronize()
    seq = Q.shape[1]
    rng = np.random.default_rng(82)
    rows = np.unique(np.concatenate([[0, 1, 1 << 20, seq - 2, seq - 1], rng.integers(0, seq, 8)]))
    got = out[0, torch.from_numpy(rows).to(dev)].double().cpu().numpy()
    assert_attn_close(got, Q, K, V, True, 0, rows, torch.float32, "seq 2^20 + 3")
    del out
    torch.cuda.empty_cache()
