"""Pins for the CPU oracle, each tied to something other than the oracle itself.

The oracle computes R = (float) sum_k (double)A[i,k]*(double)B[k,j] (plain definition of
the product on the lecture pages).  Its pins:
  * its FP16 decoder against numpy's own float16 conversion, all 65536 patterns;
  * exact Python-integer arithmetic on 16x8x16 tiles (the mma.m16n8k16 shape of
    "04_tensor_cores.py" demo 1), random and adversarial, incl. subnormals and +-65504;
  * closed forms: identity, permutation, all-ones, rank-1;
  * integer-valued inputs against numpy's int64 matmul (bit-exact);
  * the error magnitudes the pages print for FP32 accumulation against FP64
    ("04_tensor_cores.py" demos 1-2, "06_triton_style.py" demo 4), reproduced with
    the oracle as the FP64 side;
  * planted mistakes (a transposed operand, a dropped term, a sign flip, the pages'
    missing K mask) that at least one pin must catch.
"""
import numpy as np
import pytest

import oracle
from tensor_core_tiled_gb300 import inputs
from tests import exact
from tests.golden import figures
from tests.parity import within_tol


def test_decoder_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert np.signbit(mine[0x8000]) and not np.signbit(mine[0x0000])
    # spot values from the binary16 definition
    assert oracle.f16_to_f64(0x0001) == 2.0 ** -24
    assert oracle.f16_to_f64(0x03FF) == 1023 * 2.0 ** -24
    assert oracle.f16_to_f64(0x0400) == 2.0 ** -14
    assert oracle.f16_to_f64(0x7BFF) == 65504.0
    assert oracle.f16_to_f64(0x3C00) == 1.0
    assert oracle.f16_to_f64(0xC000) == -2.0
    assert oracle.f16_to_f64(0x7C00) == np.inf


def test_smallest_subnormal_times_one():
    A = np.array([[0x0001]], np.uint16).view(np.float16)
    B = np.array([[1.0]], np.float16)
    C = oracle.gemm_f32(A, B)
    assert C[0, 0] == np.float32(2.0 ** -24)


def _check_tile_exact(A, B):
    """Oracle vs exact integer arithmetic: FP64 error bound, then FP32 rounding."""
    K = A.shape[1]
    R64 = oracle.gemm_f64(A, B)
    R32 = oracle.gemm_f32(A, B)
    ex = exact.exact_gemm_units(A, B)
    absu = exact.abs_sum_units(A, B)
    gamma = K * 2.0 ** -53 / (1 - K * 2.0 ** -53)
    mismatched_near_ties = 0
    for i in range(A.shape[0]):
        for j in range(B.shape[1]):
            e = exact.units_to_fraction(ex[i, j])
            err = abs(e - exact.Fraction(float(R64[i, j])))
            bound = gamma * exact.units_to_fraction(absu[i, j])
            assert err <= bound, (i, j, float(err), float(bound))
            want = exact.round_to_f32(ex[i, j])
            if R32[i, j] != want:
                # only possible when the FP64 sum sits within its error of an FP32 tie
                mismatched_near_ties += 1
                assert err > 0
    return mismatched_near_ties


def test_brute_force_mma_tiles_random():
    rng = np.random.default_rng(0)
    near = 0
    for _ in range(100):
        A = rng.standard_normal((16, 16)).astype(np.float16)
        B = rng.standard_normal((16, 8)).astype(np.float16)
        near += _check_tile_exact(A, B)
    assert near == 0


def test_brute_force_mma_tiles_adversarial():
    rng = np.random.default_rng(11)
    # subnormal-only operands, extremes, and heavy cancellation
    sub = rng.integers(1, 1024, size=(16, 16)).astype(np.uint16).view(np.float16)
    sub = np.where(rng.random((16, 16)) < 0.5, -sub, sub).astype(np.float16)
    big = np.full((16, 8), 65504.0, np.float16)
    big[::2] = -65504.0
    _check_tile_exact(sub, rng.standard_normal((16, 8)).astype(np.float16))
    _check_tile_exact(rng.standard_normal((16, 16)).astype(np.float16), big)
    # cancellation: x_k paired with -x_k plus one tiny term
    A = np.zeros((16, 16), np.float16)
    B = np.zeros((16, 8), np.float16)
    vals = rng.standard_normal(8).astype(np.float16) * np.float16(1000)
    A[:, :8] = vals
    A[:, 8:] = vals
    B[:8, :] = 1.0
    B[8:, :] = -1.0
    A[:, 15] = np.float16(2.0 ** -24)
    B[15, :] = np.float16(2.0 ** -10)
    _check_tile_exact(A, B)
    # mixed magnitudes spanning the whole FP16 range
    bits = rng.integers(0, 0x7BFF, size=(16, 16)).astype(np.uint16)
    bits |= (rng.integers(0, 2, size=(16, 16)).astype(np.uint16) << 15)
    B2 = rng.integers(0, 0x3C00, size=(16, 8)).astype(np.uint16).view(np.float16)
    _check_tile_exact(bits.view(np.float16), B2)


@pytest.mark.parametrize("n", [1, 17, 129])
def test_identity_and_permutation(n):
    rng = np.random.default_rng(5)
    X = rng.standard_normal((n, n + 3)).astype(np.float16)
    eye = np.eye(n, dtype=np.float16)
    assert np.array_equal(oracle.gemm_f32(eye, X), X.astype(np.float32))
    Y = rng.standard_normal((n + 2, n)).astype(np.float16)
    assert np.array_equal(oracle.gemm_f32(Y, eye), Y.astype(np.float32))
    perm = rng.permutation(n)
    P = np.zeros((n, n), np.float16)
    P[np.arange(n), perm] = 1.0
    assert np.array_equal(oracle.gemm_f32(P, X), X[perm].astype(np.float32))
    # right multiplication permutes columns: (Y P)[:, j] = Y[:, i] where P[i, j] = 1
    inv = np.argsort(perm)
    assert np.array_equal(oracle.gemm_f32(Y, P), Y[:, inv].astype(np.float32))


def test_all_ones_and_rank_one():
    for K in (1, 31, 150, 4097):
        A = np.ones((3, K), np.float16)
        B = np.ones((K, 5), np.float16)
        assert np.all(oracle.gemm_f32(A, B) == np.float32(K))
    rng = np.random.default_rng(7)
    a = rng.integers(-4, 5, size=9)
    b = rng.integers(-4, 5, size=11)
    K = 333
    A = np.repeat(a[:, None], K, axis=1).astype(np.float16)
    B = np.repeat(b[None, :], K, axis=0).astype(np.float16)
    want = (K * np.outer(a, b)).astype(np.float32)
    assert np.array_equal(oracle.gemm_f32(A, B), want)


@pytest.mark.parametrize("idx", range(len(inputs.RAGGED_SHAPES)))
def test_integer_inputs_bit_exact(idx):
    (M, N, K), A, B = inputs.workload("ragged_int")[idx]
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
    got = oracle.gemm_f32(A, B)
    assert np.array_equal(got, want)


def test_integer_inputs_bit_exact_256():
    rng = np.random.default_rng(0)
    A, B = inputs.integer_pair(rng, 256, 256, 256)
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
    assert np.array_equal(oracle.gemm_f32(A, B), want)


@pytest.mark.parametrize("idx", range(len(inputs.RAGGED_SHAPES)))
def test_ragged_shapes_vs_fp64_matmul(idx):
    (M, N, K), A, B = inputs.workload("ragged")[idx]
    R = oracle.gemm_f64(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    absum = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    # both are FP64 sums of exact products in different orders: each within K*eps*sum|p|
    assert np.all(np.abs(R - ref) <= 2 * K * 2.0 ** -53 * absum)
    assert R.shape == (M, N)


def test_leading_dimensions():
    rng = np.random.default_rng(9)
    M, N, K = 37, 45, 29
    Aw = rng.standard_normal((M, K + 11)).astype(np.float16)
    Bw = rng.standard_normal((K + 3, N + 5)).astype(np.float16)
    got = oracle.gemm_f32(Aw, Bw, M=M, N=N, K=K)
    want = oracle.gemm_f32(np.ascontiguousarray(Aw[:, :K]), np.ascontiguousarray(Bw[:K, :N]))
    assert np.array_equal(got, want)


def test_empty_dimensions():
    A = np.zeros((4, 0), np.float16)
    B = np.zeros((0, 6), np.float16)
    C = oracle.gemm_f32(A, B)
    assert C.shape == (4, 6) and np.all(C == 0)
    assert oracle.gemm_f32(np.zeros((0, 3), np.float16), np.zeros((3, 5), np.float16)).shape == (0, 5)
    assert oracle.gemm_f32(np.zeros((2, 3), np.float16), np.zeros((3, 0), np.float16)).shape == (2, 0)


def test_elems_and_rows_agree_with_full():
    (M, N, K), A, B = inputs.workload("ragged")[0]
    full = oracle.gemm_f32(A, B)
    rows = np.array([0, M - 1, 5, 123])
    cols = np.array([0, N - 1, 7, 99])
    o64, o32 = oracle.gemm_elems(A, B, rows, cols)
    assert np.array_equal(o32, full[rows, cols])
    part = oracle.gemm_rows_f32(A, B, 100, 50)
    assert np.array_equal(part, full[100:150])


# ---- page figures reproduced with the oracle as the FP64 reference -------------------

def _band(value, approx, factor=3.0):
    return approx / factor <= value <= approx * factor


def _rank1_terms(A, B):
    """The K rank-1 terms A[:, k] B[k, :] of A.B as FP32 arrays.  Each is exact in FP32: a
    product of two FP16 values has at most 22 significant bits (asserted)."""
    P = np.einsum("ik,kj->kij", A.astype(np.float64), B.astype(np.float64))
    P32 = P.astype(np.float32)
    assert np.array_equal(P32.astype(np.float64), P)
    return P32


def _running_sum(terms, init, dtype):
    """Recursive summation with the running sum held in `dtype`: each addition s + t is
    rounded to FP32, and then to FP16 when the running sum is FP16."""
    s = np.asarray(init, dtype)
    for t in terms:
        s = (s.astype(np.float32) + t).astype(dtype)
    return s


def test_page_mma_tile_error_magnitude():
    """16x8x16 tiles plus an FP32 C accumulated in FP32 ("04_tensor_cores.py" demo 1): the
    error against FP64 is of the order the page prints (about 2e-6), and every element obeys
    the recursive-summation bound gamma_n * (|c| + sum |p|) with n = 16 additions."""
    fig = figures.load()
    rng = np.random.default_rng(2024)
    u = 2.0 ** -24
    gamma = 16 * u / (1 - 16 * u)
    worst = 0.0
    for _ in range(200):
        A = rng.standard_normal((16, 16)).astype(np.float16)
        B = rng.standard_normal((16, 8)).astype(np.float16)
        Cm = rng.standard_normal((16, 8)).astype(np.float32)
        P = _rank1_terms(A, B)
        err = np.abs(_running_sum(P, Cm, np.float32) - (oracle.gemm_f64(A, B) + Cm))
        assert np.all(err <= gamma * (np.abs(Cm) + np.abs(P.astype(np.float64)).sum(axis=0)))
        worst = max(worst, float(err.max()))
    assert _band(worst, fig["mma_tile_fp32_err_approx"])


def test_page_block_gemm_error_magnitude():
    """128^3, FP32 accumulation of k16 partial products ("04_tensor_cores.py" demo 2: one
    tensor-core step per 16 k): the error against FP64 is of the order printed (about 5e-6)."""
    fig = figures.load()
    rng = np.random.default_rng(2025)
    A = rng.standard_normal((128, 128)).astype(np.float16)
    B = rng.standard_normal((128, 128)).astype(np.float16)
    steps = [(A[:, k:k + 16].astype(np.float64) @ B[k:k + 16].astype(np.float64)).astype(np.float32)
             for k in range(0, 128, 16)]
    err = np.abs(_running_sum(steps, np.zeros((128, 128)), np.float32) - oracle.gemm_f64(A, B)).max()
    assert _band(err, fig["block_gemm_128_fp32_err_approx"])


def test_page_fp16_accumulation_ratio():
    """An FP16 running sum against an FP32 one, 64x64xK ("06_triton_style.py" demo 4).  Both
    errors grow with the unit roundoff of the accumulator, so their ratio sits near
    2^-11 / 2^-24 = 2^13 = 8192, inside the page's 7000-9000x; the build's tolerance accepts
    FP32 accumulation and rejects FP16 accumulation at large K."""
    fig = figures.load()
    rng = np.random.default_rng(2026)
    ratios = []
    for K in (64, 256, 1024, 4096):
        a = rng.standard_normal((64, K)).astype(np.float16)
        b = rng.standard_normal((K, 64)).astype(np.float16)
        P = _rank1_terms(a, b)
        ref = oracle.gemm_f64(a, b)
        s32 = _running_sum(P, np.zeros((64, 64)), np.float32)
        s16 = _running_sum(P, np.zeros((64, 64)), np.float16).astype(np.float32)
        ratios.append(np.abs(s16 - ref).max() / np.abs(s32 - ref).max())
        assert within_tol(s32, ref.astype(np.float32), K)
        if K >= 1024:
            assert not within_tol(s16, ref.astype(np.float32), K)
    med = float(np.median(ratios))
    assert 2.0 ** 13 / 1.5 <= med <= 2.0 ** 13 * 1.5
    lo, hi = fig["fp16_over_fp32_acc_lo"], fig["fp16_over_fp32_acc_hi"]
    assert min(ratios) >= lo / 2 and max(ratios) <= hi * 2
    assert lo * 0.85 <= med <= hi * 1.15


# ---- planted mistakes: the pins above must have the power to catch them -------------

def _pins_pass(gemm):
    """A compact run of the pins on a candidate gemm(A, B) -> FP32."""
    rng = np.random.default_rng(0)
    for _ in range(5):
        A = rng.standard_normal((16, 16)).astype(np.float16)
        B = rng.standard_normal((16, 8)).astype(np.float16)
        ex = exact.exact_gemm_units(A, B)
        want = np.vectorize(exact.round_to_f32, otypes=[np.float32])(ex)
        if not np.array_equal(gemm(A, B), want):
            return False
    n = 17
    X = rng.standard_normal((n, n + 3)).astype(np.float16)
    perm = rng.permutation(n)
    P = np.zeros((n, n), np.float16)
    P[np.arange(n), perm] = 1.0
    if not np.array_equal(gemm(P, X), X[perm].astype(np.float32)):
        return False
    return True


def test_pins_accept_the_oracle():
    assert _pins_pass(oracle.gemm_f32)


@pytest.mark.parametrize("mistake", ["transposed_B", "dropped_last_k", "sign_flip", "off_by_one_row"])
def test_pins_catch_planted_mistakes(mistake):
    def bad(A, B):
        if mistake == "transposed_B":
            Bt = np.ascontiguousarray(B.T) if B.shape[0] == B.shape[1] else np.ascontiguousarray(
                B[::-1])
            return oracle.gemm_f32(A, Bt)
        if mistake == "dropped_last_k":
            return oracle.gemm_f32(np.ascontiguousarray(A[:, :-1]), np.ascontiguousarray(B[:-1]))
        if mistake == "sign_flip":
            C = oracle.gemm_f32(A, B)
            C[0, 0] = -C[0, 0]
            return C
        if mistake == "off_by_one_row":
            C = oracle.gemm_f32(A, B)
            return np.roll(C, 1, axis=0)
        raise AssertionError
    assert not _pins_pass(bad)


def _missing_k_mask_gemm(A, B, block_k=32):
    """The pages' deliberate bug ("06_triton_style.py" demo 4): the last K block is read
    without a K mask, so A's tail reads run into the next row and B's into rows past K
    (indices clamped to the array, as the page's kernel does)."""
    M, K = A.shape
    _, N = B.shape
    Kp = -(-K // block_k) * block_k
    a = A.ravel()
    b = B.ravel()
    ia = np.clip(np.arange(M)[:, None] * K + np.arange(Kp)[None, :], 0, a.size - 1)
    ib = np.clip(np.arange(Kp)[:, None] * N + np.arange(N)[None, :], 0, b.size - 1)
    return oracle.gemm_f32(a[ia], b[ib])


def test_tolerance_catches_missing_k_mask():
    """The K-mask bug passes on block-multiple shapes and fails otherwise (demo 4 table)."""
    rng = np.random.default_rng(3)
    for (M, N, K) in [(64, 64, 64), (128, 64, 96), (1, 1, 1), (17, 33, 65), (100, 70, 50), (64, 64, 40)]:
        A = rng.standard_normal((M, K)).astype(np.float16)
        B = rng.standard_normal((K, N)).astype(np.float16)
        ref = oracle.gemm_f32(A, B)
        buggy = _missing_k_mask_gemm(A, B)
        if K % 32 == 0:
            assert within_tol(buggy, ref, K)
        else:
            assert not within_tol(buggy, ref, K), (M, N, K)


def test_input_chunking_is_stream_stable():
    """Chunked FP16 generation equals one numpy call (the recipe does not depend on it)."""
    rng1 = np.random.default_rng(42)
    rng2 = np.random.default_rng(42)
    old = inputs._CHUNK_ELEMS
    try:
        inputs._CHUNK_ELEMS = 1000
        a = inputs.normal_f16(rng1, 300, 77)
    finally:
        inputs._CHUNK_ELEMS = old
    b = rng2.standard_normal((300, 77)).astype(np.float16)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
