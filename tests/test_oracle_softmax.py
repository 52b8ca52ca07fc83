"""Pins for the oracle's row softmax ("06_triton_style.py" demo 3).

  * closed forms: a one-element row is 1, an all-equal row is 1/N, two values a and b give
    the logistic 1 / (1 + exp(b - a)), a row with one value far above the rest is one-hot;
  * invariants: every row sums to 1 within rounding, adding a constant to a row changes
    nothing beyond rounding, the order of values is kept;
  * scipy's softmax on random rows (a library routine), the page's 4096 x 1024 N(0,1) case
    (seed 2, float32) included;
  * rows with huge values do not overflow; -inf entries get 0; a NaN, +inf or all -inf row
    is NaN.
"""
import numpy as np
import pytest

import oracle

scipy_special = pytest.importorskip("scipy.special")


def test_closed_forms():
    assert oracle.softmax_rows_f32(np.array([[3.5]], np.float32))[0, 0] == 1.0
    y = oracle.softmax_rows_f32(np.full((2, 7), -2.25, np.float32))
    assert np.all(y == np.float32(1 / 7))
    a, b = np.float32(0.75), np.float32(-1.5)
    y = oracle.softmax_rows_f32(np.array([[a, b]], np.float32))
    assert y[0, 0] == np.float32(1.0 / (1.0 + np.exp(np.float64(b) - np.float64(a))))
    x = np.zeros((1, 100), np.float32)
    x[0, 17] = 1000.0
    y = oracle.softmax_rows_f32(x)
    assert y[0, 17] == 1.0 and np.all(np.delete(y[0], 17) == 0.0)


def test_invariants():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 513)) * 4).astype(np.float32)
    y = oracle.softmax_rows_f32(x)
    assert np.all(np.abs(y.astype(np.float64).sum(1) - 1) < 1e-6)
    y2 = oracle.softmax_rows_f32(x + np.float32(37.0))
    assert np.max(np.abs(y2 - y)) < 1e-6 * np.max(y)
    order = np.argsort(x, axis=1, kind="stable")
    ys = np.take_along_axis(y, order, 1)
    assert np.all(np.diff(ys, axis=1) >= 0)


@pytest.mark.parametrize("M,N,seed", [(4096, 1024, 2), (100, 3000, 3), (7, 1, 4), (300, 37, 5)])
def test_matches_scipy(M, N, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, N)).astype(np.float32)
    y = oracle.softmax_rows_f32(x)
    ref = scipy_special.softmax(x.astype(np.float64), axis=1)
    assert np.all(np.abs(y - ref) <= 2.0 ** -24 * ref + 1e-45)


def test_extremes():
    x = np.array([[1e30, 1e30 - 1e24, -1e30, 0.0],
                  [-np.inf, 0.0, 1.0, -np.inf],
                  [np.nan, 0.0, 1.0, 2.0],
                  [np.inf, 0.0, 1.0, 2.0],
                  [-np.inf, -np.inf, -np.inf, -np.inf]], np.float32)
    y = oracle.softmax_rows_f32(x)
    assert np.all(np.isfinite(y[0])) and abs(float(y[0].sum()) - 1) < 1e-6
    assert y[1, 0] == 0 and y[1, 3] == 0 and abs(float(y[1].sum()) - 1) < 1e-6
    assert np.all(np.isnan(y[2])) and np.all(np.isnan(y[3])) and np.all(np.isnan(y[4]))


def test_planted_mistakes_are_caught():
    """Forgetting to subtract the maximum overflows; a column-wise softmax fails the sums."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((50, 60)).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        naive = np.exp(x + np.float32(100)) / np.exp(x + np.float32(100)).sum(1, keepdims=True)
    assert not np.all(np.isfinite(naive)) or not np.allclose(naive, oracle.softmax_rows_f32(x + 100))
    colwise = oracle.softmax_rows_f32(np.ascontiguousarray(x.T)).T
    assert not np.all(np.abs(colwise.sum(1) - 1) < 1e-5)
