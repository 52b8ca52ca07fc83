"""Exact reference arithmetic for tiny products, with Python integers only.

Every FP16 value is an integer multiple of 2^-24 (the smallest subnormal), so every
product of two FP16 values is an integer multiple of 2^-48 and a sum of such products
is exact as a Python integer count of 2^-48 units.  ``round_to_f32`` rounds such an
exact value to the nearest FP32 value, ties to even, with integer operations only, so
that nothing here depends on the oracle or on floating-point rounding.
"""
from fractions import Fraction

import numpy as np

UNIT_EXP = -48  # exact sums are counted in units of 2^-48


def f16_units(x16):
    """FP16 array -> nested Python ints in units of 2^-24 (exact)."""
    out = []
    for v in np.asarray(x16, np.float16).ravel().tolist():
        f = Fraction(v) * (1 << 24)
        assert f.denominator == 1
        out.append(int(f))
    return np.array(out, dtype=object).reshape(np.shape(x16))


def exact_gemm_units(A16, B16):
    """Exact C = A.B in units of 2^-48 as an object array of Python ints (tiny sizes)."""
    a = f16_units(A16)
    b = f16_units(B16)
    M, K = a.shape
    _, N = b.shape
    C = np.empty((M, N), dtype=object)
    for i in range(M):
        for j in range(N):
            s = 0
            for k in range(K):
                s += a[i, k] * b[k, j]
            C[i, j] = s
    return C


def abs_sum_units(A16, B16):
    """sum_k |A[i,k]*B[k,j]| in units of 2^-48 (for the FP64 error bound)."""
    a = np.vectorize(abs, otypes=[object])(f16_units(A16))
    b = np.vectorize(abs, otypes=[object])(f16_units(B16))
    M, K = a.shape
    _, N = b.shape
    C = np.empty((M, N), dtype=object)
    for i in range(M):
        for j in range(N):
            C[i, j] = sum(a[i, k] * b[k, j] for k in range(K))
    return C


def round_to_f32(n, unit_exp=UNIT_EXP):
    """Nearest FP32 (ties to even) to the exact value n * 2^unit_exp; n a Python int."""
    if n == 0:
        return np.float32(0.0)
    sign = -1 if n < 0 else 1
    m = abs(n)
    e = m.bit_length() - 1 + unit_exp          # value in [2^e, 2^(e+1))
    q = max(e - 23, -149)                       # quantum: 24-bit significand, subnormals at 2^-149
    shift = q - unit_exp
    if shift <= 0:
        r = m << (-shift)
    else:
        r, rem = divmod(m, 1 << shift)
        half = 1 << (shift - 1)
        if rem > half or (rem == half and (r & 1)):
            r += 1
    val = Fraction(r) * (Fraction(2) ** q)
    assert val < Fraction(2) ** 128, "overflow to inf is not expected in these tests"
    return np.float32(sign * float(val))       # r*2^q is representable in FP32, so exact


def units_to_fraction(n, unit_exp=UNIT_EXP):
    return Fraction(n) * (Fraction(2) ** unit_exp)
