"""Parity of the fused row softmax (softmax_rows_f32) with the oracle.

The workload is the one of "06_triton_style.py" demo 3: N(0,1) rows, softmax along each
row.  Rows whose base and leading dimension are multiples of 16 bytes take the staged
kernels (a team of threads per row up to 8192 columns, a cluster of CTAs per row beyond,
reading long slices twice past 16 x 28672 columns); other rows take the plain kernels
(a warp per row up to 2048 columns, a CTA per row in shared memory up to 51200, two passes
beyond).  Shapes sit on each boundary, with ragged lengths, padded and unaligned rows,
in-place use, special values and empty shapes.

Error bound (per element, relative to the exact softmax r_j, with u = 2^-24):
  the staged kernels take e^d as 2^(d log2 e) on the hardware base-2 exponential (relative
  error about 2^-22 = 4u), and d = x_j - max, the product d log2 e and the constant log2 e
  each round once, so a term carries (4 + 3 |d_j|) u; the plain kernels use expf (2 ulp)
  and carry less.  The row sum adds the terms' errors (at most 4 + 3 |d|max each, in
  relative terms) and n u for a chain of n additions; a cluster rescales each slice sum by
  expf of a slice-maximum difference (4 + |d|max) and the slice scale takes one more such
  factor; the reciprocal or division, the final product and the oracle's rounding add u
  each.  In total |y_j - r_j| <= u (32 + 3 |d_j| + 6 |d|max + 7 n) r_j, where n bounds the
  longest chain of additions: 64 + ceil(N / 4096) on the staged path (at most 32 terms per
  thread in a team, N / 4096 per thread in a 16-CTA cluster, plus the reduction trees and
  the 16 slice sums), 64 + ceil(N / 256) on the plain path.  Rows of 0 and -inf entries
  have an exact softmax (1/k on the k zeros) and are compared bit for bit, so that a
  dropped or repeated piece of a long row cannot hide inside the bound.
"""
import math

import numpy as np
import pytest

import oracle
import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _chain(N, staged):
    return 64 + (math.ceil(N / 4096) if staged else math.ceil(N / 256))


def _check(x, y, staged=None):
    """y (the kernel's output) against the oracle on x, element by element.  `staged`
    says whether the rows took the staged kernels (default: contiguous rows, N % 4 == 0)."""
    if staged is None:
        staged = x.shape[1] % 4 == 0
    ref = oracle.softmax_rows_f32(x)
    assert y.shape == ref.shape
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan_ref), "NaN rows differ"
    valid = ~nan_ref.any(axis=1)
    with np.errstate(invalid="ignore"):
        d = x.astype(np.float64) - x.max(axis=1, keepdims=True).astype(np.float64)
    ad = np.where(np.isfinite(d), np.abs(d), 0)
    n = _chain(x.shape[1], staged)
    tol = U * (32 + 3 * ad + 6 * ad.max(axis=1, keepdims=True) + 7 * n) * ref + 1e-37
    err = np.abs(y.astype(np.float64) - ref.astype(np.float64))
    bad = ~(err <= tol) & valid[:, None]
    assert not bad.any(), (f"{bad.sum()} elements out of tolerance; worst "
                           f"{np.unravel_index(np.argmax(np.where(valid[:, None], err / tol, 0)), err.shape)}")


def _run(x, inplace=False):
    X = torch.from_numpy(x).cuda()
    out = tct.softmax(X, out=X if inplace else None)
    torch.cuda.synchronize()
    return out.cpu().numpy()


# (M, N, seed) for 16-byte-aligned rows.  Up to 8192 columns a team of 8 to 256 threads
# holds a row in registers (several rows staged per ring slot); up to 8 * 8192 columns a
# cluster of ceil(N / 8192) CTAs splits each row the same way; beyond, a cluster of
# ceil(N / 20480) CTAs (7 taken as 8, at most 16) stages each slice in 16 KB shared-memory
# slots, and reads it twice when it exceeds the 7-slot ring (past 16 * 28672 columns).
# The tall shapes wrap every CTA's slot ring several times.
SHAPES = [(1, 1, 10), (7, 1, 11), (33, 5, 12), (300, 37, 13), (129, 128, 14), (64, 129, 15), (257, 256, 16),
          (100, 511, 17), (65, 1000, 18), (40, 1024, 19), (80000, 100, 40), (31, 1025, 20), (17, 2048, 21),
          (9, 2049, 22), (20, 3000, 23), (5, 4096, 24), (5, 4097, 25), (3, 8192, 26), (8000, 2000, 41),
          (3, 8193, 27), (2, 51200, 28), (2, 51201, 29), (1000, 30000, 42), (2, 65536, 45), (2, 65537, 46), (2, 131072, 43),
          (2, 131073, 44), (2, 143360, 47), (3, 163841, 48), (2, 327680, 49), (2, 327681, 50),
          (2, 200003, 30), (2, 393216, 31), (2, 393217, 32), (2, 458752, 35), (2, 458753, 36), (3, 1 << 20, 33),
          (2, 1000003, 34)]


@pytest.mark.parametrize("M,N,seed", SHAPES)
def test_matches_oracle(M, N, seed):
    x = inputs.normal_f32(np.random.default_rng(seed), M, N)
    _check(x, _run(x))


def test_page_workload():
    """The page's 4096 x 1024 case; row sums are 1 to within the summation bound."""
    x = inputs.normal_f32(np.random.default_rng(2), *inputs.SOFTMAX_PAGE)
    y = _run(x)
    _check(x, y)
    assert np.all(np.abs(y.astype(np.float64).sum(axis=1) - 1) < 1e-5)


@pytest.mark.parametrize("N", [100, 5000, 70000])
def test_wide_range_rows(N):
    """Scaled rows (values up to +-80): exp underflows to zero for most entries."""
    x = (inputs.normal_f32(np.random.default_rng(N), 16, N) * np.float32(20)).astype(np.float32)
    _check(x, _run(x))


@pytest.mark.parametrize("N", [1000, 4000, 30000, 60000])
def test_padded_and_unaligned(N):
    """Rows with ld > N: 16-byte-aligned padded rows (staged kernels), and rows whose ld or base
    is not a multiple of 16 bytes (plain kernels)."""
    M = 37
    rng = np.random.default_rng(N + 1)
    x = inputs.normal_f32(rng, M, N)
    for ld, off in [(N + 3, 0), (N + 8, 4), (N + 1, 1), (N + 4, 0)]:
        buf = torch.full((M * ld + 8,), float("nan"), device="cuda")
        src = buf[off:off + M * ld].view(M, ld)
        src[:, :N] = torch.from_numpy(x).cuda()
        ybuf = torch.full((M * ld + 8,), -7.0, device="cuda")
        dst = ybuf[off:off + M * ld].view(M, ld)
        st = tct.softmax_rows_f32(src.data_ptr(), dst.data_ptr(), M, N, ld, ld,
                                  torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
        _check(x, dst[:, :N].cpu().numpy(), staged=(ld % 4 == 0 and off % 4 == 0))
        assert torch.all(dst[:, N:] == -7.0), "padding columns were written"
        assert torch.all(ybuf[:off] == -7.0) and torch.all(ybuf[off + M * ld:] == -7.0)


@pytest.mark.parametrize("N", [300, 3000, 60000])
def test_in_place(N):
    x = inputs.normal_f32(np.random.default_rng(N + 2), 21, N)
    _check(x, _run(x, inplace=True))


@pytest.mark.parametrize("N", [4, 3000, 60000, 300000, 1 << 20])
def test_special_values(N):
    """-inf entries give exactly 0; rows with NaN, +inf or only -inf give NaN everywhere."""
    x = inputs.normal_f32(np.random.default_rng(N + 3), 6, N)
    x[1, 0] = -np.inf
    x[1, N - 1] = -np.inf
    x[2, N // 2] = np.nan
    x[3, N - 1] = np.inf
    x[4, :] = -np.inf
    x[5, :] = 1e30
    y = _run(x)
    _check(x, y)
    assert y[1, 0] == 0 and y[1, N - 1] == 0
    assert np.isnan(y[2:5]).all()
    assert np.all(y[5] == np.float32(1) / np.float32(N))


def test_empty_and_invalid():
    X = torch.zeros(4, 8, device="cuda")
    p = X.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert tct.softmax_rows_f32(p, p, 0, 8, 8, 8, s) == 0
    assert tct.softmax_rows_f32(p, p, 4, 0, 8, 8, s) == 0
    assert tct.softmax_rows_f32(p, p, 4, 8, 7, 8, s) == 1   # ldx < N
    assert tct.softmax_rows_f32(p, p, 4, 8, 8, 12, s) == 1  # in place with ldx != ldy
    assert tct.softmax_rows_f32(p + 2, p + 64, 2, 8, 8, 8, s) == 1  # misaligned
    assert tct.softmax_rows_f32(0, p, 2, 8, 8, 8, s) == 1
    torch.cuda.synchronize()
    assert torch.all(X == 0)


@pytest.mark.parametrize("N", [3, 8, 100, 128, 1000, 1024, 2047, 4096, 8192, 8196, 30000, 65536, 65540,
                               131072, 131076, 143360, 393216, 500000, 1 << 20])
def test_exact_zero_inf_rows(N):
    """Rows of 0 and -inf: exp gives exactly 1 and 0, so the softmax is exactly 1/k on the k
    zeros, in every kernel; compared bit for bit (k = 0 gives a NaN row)."""
    rng = np.random.default_rng(N + 5)
    M = 6
    x = np.where(rng.random((M, N)) < 0.5, np.float32(0), np.float32(-np.inf)).astype(np.float32)
    x[1, :] = 0  # k = N
    x[2, :] = -np.inf
    x[2, N - 1] = 0  # k = 1, in the tail
    x[3, :] = -np.inf  # k = 0
    y = _run(x)
    k = (x == 0).sum(axis=1)
    for i in range(M):
        if k[i] == 0:
            assert np.isnan(y[i]).all()
        else:
            want = np.where(x[i] == 0, np.float32(1) / np.float32(k[i]), np.float32(0))
            assert np.array_equal(y[i], want), f"row {i}: {np.flatnonzero(y[i] != want)[:5]}"
