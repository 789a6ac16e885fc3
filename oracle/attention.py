"""CPU oracle for attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module; the product library never does, and nothing here
imports the product package.

What it computes ("How to hand-write Triton kernels for matmul and Flash
Attention", section "Flash Attention in Triton and online softmax"): for each
of BH independent heads, with Q, K, V of shape [seq, d],

    S = Q K^T / sqrt(d)
    S[i, j] = -inf where the causal mask removes it (key j after query i:
              the section keeps S[i, j] only where i >= j)
    O = softmax_rows(S) V

The section's kernel reaches this result blockwise with an online softmax
(running maximum, rescaled running sum and accumulator); that is exact in
exact arithmetic, so the oracle is the definition itself, evaluated directly:
the 16-bit inputs are widened exactly to binary64 and every step runs in
binary64 (numpy matmul for the two products, the max-subtracted softmax of
"Writing GPU kernels in Triton: Vector Add, Softmax, MatMul", section 2.3).
The section masks with -1e9 instead of -inf; after the maximum is subtracted
both give a weight of exactly 0, and -inf is used here.

Pinned by ``tests/test_attention_oracle.py``: closed forms (constant values,
identical keys, one-key rows, a two-key case with the 1/sqrt(d) scale written
out), torch's scaled_dot_product_attention in float64 as an independent
library routine, the section's blockwise online-softmax loop evaluated in
binary64, permutation invariance, and planted mistakes.
"""
from __future__ import annotations

import numpy as np


def _f64(t) -> np.ndarray:
    if hasattr(t, "detach"):
        t = t.detach().float().numpy()
    return np.asarray(t, dtype=np.float64)


def _one_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool, rows=None) -> np.ndarray:
    d = q.shape[1]
    qi = q if rows is None else q[rows]
    s = (qi @ k.T) / np.sqrt(d)
    if causal:
        qidx = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
        s = np.where(qidx[:, None] >= np.arange(k.shape[0])[None, :], s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    p = e / np.sum(e, axis=1, keepdims=True)
    return p @ v


def attention(Q, K, V, causal: bool) -> np.ndarray:
    """O for Q, K, V of shape [BH, seq, d] (or [seq, d]); binary64."""
    q, k, v = _f64(Q), _f64(K), _f64(V)
    if q.ndim == 2:
        return _one_head(q, k, v, causal)
    return np.stack([_one_head(q[h], k[h], v[h], causal) for h in range(q.shape[0])])


def attention_rows(Q, K, V, causal: bool, head: int, rows) -> np.ndarray:
    """Rows `rows` of O for head `head` only (for inputs too large to do whole)."""
    q, k, v = _f64(Q[head]), _f64(K[head]), _f64(V[head])
    return _one_head(q, k, v, causal, rows=np.asarray(rows, dtype=np.int64))


def weight_abs_v(Q, K, V, causal: bool, head: int, rows) -> np.ndarray:
    """sum_j P[i, j] |V[j, :]| for the listed rows: the scale of a rounding error
    made on the weights P (a tolerance helper)."""
    q, k, v = _f64(Q[head]), _f64(K[head]), _f64(V[head])
    rows = np.asarray(rows, dtype=np.int64)
    d = q.shape[1]
    s = (q[rows] @ k.T) / np.sqrt(d)
    if causal:
        s = np.where(rows[:, None] >= np.arange(k.shape[0])[None, :], s, -np.inf)
    e = np.exp(s - np.max(s, axis=1, keepdims=True))
    p = e / np.sum(e, axis=1, keepdims=True)
    return p @ np.abs(v)
