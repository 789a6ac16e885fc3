"""Pins of the attention oracle (CPU only).

Each pin checks the oracle against something other than itself: closed forms,
torch's scaled_dot_product_attention in float64 (an independent library
routine), and the blockwise online-softmax loop of "How to hand-write Triton
kernels for matmul and Flash Attention" (section "Flash Attention in Triton and
online softmax") evaluated in binary64.  The same pins are run on copies of
the oracle with one plausible mistake planted in each; every copy must fail at
least one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oa


def _rng_qkv(bh, seq, d, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    mk = lambda: (torch.randn(bh, seq, d, generator=g) * scale).to(torch.bfloat16)  # noqa: E731
    return mk(), mk(), mk()


def online_blockwise(Q, K, V, causal, block_q=16, block_kv=16):
    """The section's loop in binary64: per query block, running maximum m (from
    -1e9), running sum l and accumulator acc, rescaled by alpha = exp(m - m_new)
    for every key block; causal positions kept where query >= key (else -1e9)."""
    q, k, v = (np.asarray(t.float().numpy(), dtype=np.float64) for t in (Q, K, V))
    seq, d = q.shape
    out = np.zeros_like(q)
    for q0 in range(0, seq, block_q):
        qi = np.arange(q0, min(seq, q0 + block_q))
        m = np.full(len(qi), -1e9)
        l = np.zeros(len(qi))
        acc = np.zeros((len(qi), d))
        for k0 in range(0, seq, block_kv):
            kj = np.arange(k0, min(seq, k0 + block_kv))
            s = q[qi] @ k[kj].T / math.sqrt(d)
            if causal:
                s = np.where(qi[:, None] >= kj[None, :], s, -1e9)
            m_new = np.maximum(m, s.max(axis=1))
            p = np.exp(s - m_new[:, None])
            alpha = np.exp(m - m_new)
            acc = acc * alpha[:, None] + p @ v[kj]
            l = l * alpha + p.sum(axis=1)
            m = m_new
        out[qi] = acc / l[:, None]
    return out


def _pins(fn):
    out = []
    # Closed forms.
    Q, K, V = _rng_qkv(2, 24, 16, seed=1)
    Vc = torch.ones_like(V) * torch.tensor([1.5, -2.0] * 8, dtype=torch.bfloat16)
    for causal in (False, True):
        o = fn(Q, K, Vc, causal)
        out.append((f"constant V rows -> O = that row (causal={causal})",
                    bool(np.allclose(o, np.broadcast_to(Vc[0, 0].double().numpy(), o.shape),
                                     rtol=0, atol=1e-13))))
    Ksame = K[:, :1].expand(-1, 24, -1).contiguous()
    vv = V.double().numpy()
    o = fn(Q, Ksame, V, False)
    out.append(("identical keys -> mean of V", bool(np.allclose(o, vv.mean(axis=1, keepdims=True).repeat(24, axis=1),
                                                                 rtol=0, atol=1e-13))))
    o = fn(Q, Ksame, V, True)
    prefix = np.cumsum(vv, axis=1) / np.arange(1, 25)[None, :, None]
    out.append(("identical keys, causal -> prefix means of V", bool(np.allclose(o, prefix, rtol=0, atol=1e-13))))
    o = fn(Q, K, V, True)
    out.append(("causal first row = V[0]", bool(np.allclose(o[:, 0], vv[:, 0], rtol=0, atol=0))))
    o1 = fn(Q[:, :1], K[:, :1], V[:, :1], False)
    out.append(("one key -> O = V", bool(np.allclose(o1, vv[:, :1], rtol=0, atol=0))))
    # Two keys, the 1/sqrt(d) scale written out.
    d = 4
    q2 = torch.tensor([[[1.0, 2.0, 0.0, -1.0]]]).to(torch.bfloat16)
    k2 = torch.tensor([[[0.5, 1.0, 2.0, 0.0], [-1.0, 0.5, 1.0, 3.0]]]).to(torch.bfloat16)
    v2 = torch.tensor([[[1.0, 0.0, 2.0, -1.0], [0.0, 3.0, -2.0, 1.0]]]).to(torch.bfloat16)
    a = (1.0 * 0.5 + 2.0 * 1.0) / math.sqrt(d)          # q . k0 / sqrt(d)
    b = (-1.0 + 1.0 - 3.0) / math.sqrt(d)               # q . k1 / sqrt(d)
    wa, wb = 1.0 / (1.0 + math.exp(b - a)), 1.0 / (1.0 + math.exp(a - b))
    want = wa * np.array([1.0, 0.0, 2.0, -1.0]) + wb * np.array([0.0, 3.0, -2.0, 1.0])
    q2full = torch.cat([q2, q2], dim=1)
    o = fn(q2full, k2, v2, False)
    out.append(("two keys, scale 1/sqrt(d)", bool(np.allclose(o[0, 0], want, rtol=0, atol=1e-14))))
    o = fn(q2full, k2, v2, True)
    out.append(("two keys, causal row 0 sees key 0 only",
                bool(np.allclose(o[0, 0], [1.0, 0.0, 2.0, -1.0], rtol=0, atol=0)
                     and np.allclose(o[0, 1], want, rtol=0, atol=1e-14))))
    # Library routine.
    Q, K, V = _rng_qkv(3, 40, 32, seed=2, scale=2.0)
    for causal in (False, True):
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q.double(), K.double(), V.double(), is_causal=causal).numpy()
        out.append((f"torch sdpa float64 (causal={causal})",
                    bool(np.allclose(fn(Q, K, V, causal), ref, rtol=1e-12, atol=1e-13))))
    # The section's online loop.
    for causal in (False, True):
        want = online_blockwise(Q[1], K[1], V[1], causal)
        out.append((f"online blockwise loop (causal={causal})",
                    bool(np.allclose(fn(Q, K, V, causal)[1], want, rtol=1e-12, atol=1e-13))))
    # Permuting keys and values together changes nothing (no mask).
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(5))
    out.append(("key permutation invariance",
                bool(np.allclose(fn(Q, K[:, perm], V[:, perm], False), fn(Q, K, V, False),
                                 rtol=1e-12, atol=1e-13))))
    return out


def test_oracle_passes_every_pin():
    bad = [name for name, ok in _pins(oa.attention) if not ok]
    assert not bad, bad


def test_rows_and_weight_helpers_match_whole():
    Q, K, V = _rng_qkv(2, 33, 16, seed=9)
    full = oa.attention(Q, K, V, True)
    rows = [0, 5, 32, 5]
    assert np.array_equal(oa.attention_rows(Q, K, V, True, 1, rows), full[1, rows])
    w = oa.weight_abs_v(Q, K, V, True, 0, rows)
    assert w.shape == (4, 16) and np.all(w >= np.abs(full[0, rows]) - 1e-12)
    assert np.allclose(oa.weight_abs_v(Q, K, V, True, 0, [0]), np.abs(V[0, :1].double().numpy()), atol=0)


# ------------------------------------------------------------ planted mistakes

def _mut(scale_fn=None, causal_fn=None, axis=1, v_t=False):
    def f(Q, K, V, causal):
        q, k, v = (np.asarray(t.float().numpy(), dtype=np.float64) for t in (Q, K, V))
        outs = []
        for h in range(q.shape[0]):
            d = q.shape[2]
            s = q[h] @ k[h].T * (scale_fn(d) if scale_fn else 1.0 / math.sqrt(d))
            if causal:
                n = q.shape[1]
                keep = (causal_fn or (lambda i, j: i >= j))(np.arange(n)[:, None], np.arange(k.shape[1])[None, :])
                s = np.where(keep, s, -np.inf)
            e = np.exp(s - np.max(s, axis=axis, keepdims=True))
            p = e / np.sum(e, axis=axis, keepdims=True)
            vh = v[h]
            if v_t and vh.shape[0] == vh.shape[1]:
                vh = vh.T
            outs.append(p @ vh if not v_t else p @ vh[::-1])
        return np.stack(outs)
    return f


MUTANTS = {
    "no_scale": _mut(scale_fn=lambda d: 1.0),
    "scale_1_over_d": _mut(scale_fn=lambda d: 1.0 / d),
    "strict_mask": _mut(causal_fn=lambda i, j: i > j),
    "mask_transposed": _mut(causal_fn=lambda i, j: j >= i),
    "softmax_over_queries": _mut(axis=0),
    "values_reversed": _mut(v_t=True),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_reject_planted_mistake(name):
    with np.errstate(all="ignore"):
        failed = [n for n, ok in _pins(MUTANTS[name]) if not ok]
    assert failed, f"{name} passed every pin"
