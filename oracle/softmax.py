"""CPU oracle for row-wise softmax -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module; the product library never does, and nothing here
imports the product package.

What it computes ("Writing GPU kernels in Triton: Vector Add, Softmax, MatMul",
chapter 2): for an M x N matrix X, every row on its own (section 2.4,
Y[i, :] = Softmax(X[i, :])), with Softmax(x)_j = e^{x_j} / sum_k e^{x_k} (the
chapter's opening definition), evaluated by the five steps of section 2.3:
Max -> Subtract -> Exp -> Sum -> Divide.  Subtracting the row maximum leaves
the exact result unchanged (the identity printed in section 2.3) and keeps
every exponent <= 0, so binary64 cannot overflow.

Arithmetic: the float32 inputs are widened exactly to binary64 and every step
runs in binary64 with numpy (``np.max``, ``np.exp``, ``np.sum``, one division).
Special values follow the formula: an entry of -inf contributes e^{-inf} = 0
(the padding argument of section 2.6), a row whose entries are all -inf gives
-inf - (-inf) = NaN everywhere, and a NaN entry makes its row NaN.

Pinned by ``tests/test_softmax_oracle.py``: the page's worked example
(section 2.3), closed forms (constant rows, two-element rows = the logistic
function, one-hot limits of wide rows), invariants (row sums, shift and
permutation invariance, log-ratios), a library routine (scipy) and planted
mistakes that each pin must reject.
"""
from __future__ import annotations

import numpy as np


def _rows64(X, N: int | None) -> np.ndarray:
    x = np.asarray(X.numpy() if hasattr(X, "numpy") else X)
    if x.ndim != 2:
        raise ValueError("X must be 2-D (rows x columns)")
    if N is None:
        N = x.shape[1]
    if N > x.shape[1]:
        raise ValueError("N exceeds the stored columns")
    return x[:, :N].astype(np.float64)


def softmax_rows(X, N: int | None = None) -> np.ndarray:
    """Y[i, :] = softmax(X[i, :N]) in binary64 (rows x N).  Columns of a padded
    row beyond N are never read."""
    x = _rows64(X, N)
    if x.shape[1] == 0:
        return x.copy()
    with np.errstate(invalid="ignore", over="ignore"):
        m = np.max(x, axis=1, keepdims=True)      # Max
        z = x - m                                 # Subtract
        e = np.exp(z)                             # Exp
        s = np.sum(e, axis=1, keepdims=True)      # Sum
        return e / s                              # Divide


def softmax_rows_sampled(X, rows, N: int | None = None) -> np.ndarray:
    """softmax_rows on the listed rows only (for matrices too large to do whole)."""
    rows = np.asarray(rows, dtype=np.int64)
    x = np.asarray(X.numpy() if hasattr(X, "numpy") else X)
    return softmax_rows(x[rows], N)
