"""Parity criteria shared by the tests.

Tolerance for N(0,1) FP16 inputs, element by element:
    |C - R| <= 1e-3 * sqrt(K) * max(1, |R|)
where R is the oracle's result.  Integer-valued inputs whose partial sums stay below
2^24 have a unique FP32 result, compared bit for bit (with +0 == -0).
"""
import numpy as np


def tol(R, K):
    return 1e-3 * np.sqrt(max(K, 1)) * np.maximum(1.0, np.abs(R.astype(np.float64)))


def within_tol(C, R, K):
    C = np.asarray(C)
    R = np.asarray(R)
    if C.shape != R.shape:
        return False
    if not np.all(np.isfinite(C)):
        return False
    return bool(np.all(np.abs(C.astype(np.float64) - R.astype(np.float64)) <= tol(R, K)))


def worst_ratio(C, R, K):
    """max over elements of |C - R| / tolerance (<= 1 passes)."""
    if C.size == 0:
        return 0.0
    return float(np.max(np.abs(C.astype(np.float64) - R.astype(np.float64)) / tol(R, K)))


def bit_exact(C, R):
    """Equal FP32 values, treating +0 and -0 as equal."""
    C = np.asarray(C, np.float32)
    R = np.asarray(R, np.float32)
    return C.shape == R.shape and bool(np.all(C == R))
