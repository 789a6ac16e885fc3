"""Pins of the row-wise softmax oracle (CPU only).

Every pin checks the oracle against something other than itself: the worked
example of "Writing GPU kernels in Triton: Vector Add, Softmax, MatMul",
section 2.3 (tests/golden/softmax_page4.txt), closed forms, invariants that the
mathematics fixes, and scipy's softmax as an independent library routine.  The
same pins are run on copies of the oracle with one plausible mistake planted
in each; every copy must fail at least one pin.
"""
import math

import numpy as np
import pytest
import scipy.special

from oracle import softmax as sm


def _pins(fn, golden):
    """(name, ok) for every pin, evaluated on the softmax function ``fn``."""
    out = []
    g = golden("softmax_page4.txt")
    X, Y = np.array(g["X"], dtype=np.float32), np.array(g["Y"])
    with np.errstate(all="ignore"):
        got = fn(X)
    out.append(("page example, 4 decimals", bool(np.all(np.abs(got - Y) <= 0.5e-4))))

    # Closed forms.
    with np.errstate(all="ignore"):
        c = fn(np.full((3, 7), 2.5, dtype=np.float32))
    out.append(("constant row = 1/N", bool(np.allclose(c, 1.0 / 7, rtol=0, atol=1e-15))))
    a, b = 0.75, -1.25
    with np.errstate(all="ignore"):
        two = fn(np.array([[a, b]], dtype=np.float32))
    logistic = 1.0 / (1.0 + math.exp(b - a))
    out.append(("two entries = logistic",
                bool(abs(two[0, 0] - logistic) <= 1e-15 and abs(two[0, 1] - (1 - logistic)) <= 1e-15)))
    with np.errstate(all="ignore"):
        wide = fn(np.array([[0.0, 800.0], [-800.0, 0.0]], dtype=np.float32))
    out.append(("wide rows are one-hot (no overflow)",
                bool(np.array_equal(wide, np.array([[0.0, 1.0], [0.0, 1.0]])))))
    with np.errstate(all="ignore"):
        one = fn(np.array([[-3.0], [1e30]], dtype=np.float32))
    out.append(("one column = 1", bool(np.array_equal(one, np.ones((2, 1))))))

    # Invariants on random rows of several lengths.
    rng = np.random.default_rng(7)
    # Multiples of 1/64 below 2^10 in magnitude: adding 37.5 is exact in float32.
    R = (np.round(rng.standard_normal((6, 37)) * 3 * 64) / 64).astype(np.float32)
    with np.errstate(all="ignore"):
        y = fn(R)
        y_shift = fn((R.astype(np.float64) + 37.5).astype(np.float32))
        perm = rng.permutation(37)
        y_perm = fn(R[:, perm])
    out.append(("rows sum to 1", bool(np.all(np.abs(y.sum(axis=1) - 1) <= 1e-14))))
    out.append(("shift invariance", bool(np.allclose(y, y_shift, rtol=1e-13, atol=0))))
    out.append(("permutation equivariance", bool(np.allclose(y[:, perm], y_perm, rtol=1e-14, atol=0))))
    with np.errstate(all="ignore"):
        lr = np.log(y[:, 3]) - np.log(y[:, 11])
    out.append(("log-ratio = difference", bool(np.allclose(lr, R[:, 3].astype(np.float64) - R[:, 11],
                                                           rtol=0, atol=1e-12))))
    ref = scipy.special.softmax(R.astype(np.float64), axis=1)
    out.append(("scipy agrees", bool(np.allclose(y, ref, rtol=1e-14, atol=0))))

    # Padding beyond N is never read; -inf entries weigh nothing (section 2.6).
    P = np.full((2, 9), np.nan, dtype=np.float32)
    P[:, :5] = [[1, 2, 3, 4, 5], [-3, -2, -5, -1, -4]]
    with np.errstate(all="ignore"):
        pad = fn(P, 5) if _takes_n(fn) else fn(P[:, :5])
    out.append(("columns beyond N ignored",
                bool(pad.shape == (2, 5) and np.allclose(pad, scipy.special.softmax(P[:, :5].astype(np.float64), axis=1),
                                                         rtol=1e-14, atol=0))))
    Z = np.array([[-np.inf, 0.0, np.log(3.0), -np.inf]], dtype=np.float32)
    with np.errstate(all="ignore"):
        zi = fn(Z)
    out.append(("-inf weighs nothing",
                bool(zi[0, 0] == 0 and zi[0, 3] == 0 and abs(zi[0, 1] - 0.25) <= 1e-7
                     and abs(zi[0, 2] - 0.75) <= 1e-7)))
    return out


def _takes_n(fn):
    return fn.__code__.co_argcount >= 2


def test_oracle_passes_every_pin(golden):
    bad = [name for name, ok in _pins(sm.softmax_rows, golden) if not ok]
    assert not bad, bad


def test_special_rows_follow_the_formula():
    """A row of -inf gives -inf - (-inf) = NaN; a NaN entry makes its row NaN;
    the other rows are unaffected."""
    X = np.array([[-np.inf, -np.inf, -np.inf], [1.0, np.nan, 2.0], [0.0, 0.0, 0.0]],
                 dtype=np.float32)
    y = sm.softmax_rows(X)
    assert np.all(np.isnan(y[0])) and np.all(np.isnan(y[1]))
    assert np.allclose(y[2], 1.0 / 3, rtol=0, atol=1e-16)


def test_empty_shapes():
    assert sm.softmax_rows(np.zeros((0, 5), np.float32)).shape == (0, 5)
    assert sm.softmax_rows(np.zeros((4, 0), np.float32)).shape == (4, 0)
    assert sm.softmax_rows(np.zeros((4, 6), np.float32), 0).shape == (4, 0)


def test_sampled_rows_match_whole_matrix():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((50, 64)).astype(np.float32)
    rows = [0, 7, 49, 7]
    assert np.array_equal(sm.softmax_rows_sampled(X, rows), sm.softmax_rows(X)[rows])


# ------------------------------------------------------------ planted mistakes

def _no_max(X, N=None):
    x = sm._rows64(X, N)
    e = np.exp(x)
    return e / e.sum(axis=1, keepdims=True)


def _subtract_min(X, N=None):
    x = sm._rows64(X, N)
    e = np.exp(x - x.min(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _sign_flipped(X, N=None):
    x = sm._rows64(X, N)
    m = x.max(axis=1, keepdims=True)
    e = np.exp(m - x)
    return e / e.sum(axis=1, keepdims=True)


def _divide_by_max(X, N=None):
    x = sm._rows64(X, N)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return e / e.max(axis=1, keepdims=True)


def _sum_over_columns(X, N=None):
    x = sm._rows64(X, N)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def _reads_padding(X, N=None):
    x = np.asarray(X, dtype=np.float64)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True))[:, : (N if N is not None else x.shape[1])]


def _drops_last_column(X, N=None):
    x = sm._rows64(X, N)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return e / e[:, :-1].sum(axis=1, keepdims=True) if x.shape[1] > 1 else e / e.sum(axis=1, keepdims=True)


def _float32_exp(X, N=None):
    x = sm._rows64(X, N).astype(np.float32)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float64)


MUTANTS = [_no_max, _subtract_min, _sign_flipped, _divide_by_max, _sum_over_columns,
           _reads_padding, _drops_last_column, _float32_exp]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda f: f.__name__.strip("_"))
def test_pins_reject_planted_mistake(mutant, golden):
    failed = [name for name, ok in _pins(mutant, golden) if not ok]
    assert failed, f"{mutant.__name__} passed every pin"
