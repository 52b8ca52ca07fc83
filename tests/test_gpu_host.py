"""The host-buffer entry points (gemm_f16_f32_host, softmax_rows_f32_host) through the C ABI.

Operands and results live in host memory: page-locked (the pipelined path) and pageable.
Results are checked against the oracle with the parity tolerances, integer GEMM inputs bit
for bit, and against the device-buffer entry points; host leading dimensions larger than
the row, ragged shapes (several row blocks with a short last one, K and N off the 16-byte
pitch), K = 0 and calls queued back to back on one stream are covered.
"""
import numpy as np
import pytest

import oracle
import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs
from tests.parity import within_tol

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK


def _host(x, pinned):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.pin_memory() if pinned else t.clone()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _gemm_host(A, B, M, N, K, pinned, lda=None, ldb=None, ldc=None):
    lda, ldb, ldc = lda or K, ldb or N, ldc or N
    hA = np.zeros((M, lda), np.float16)
    hA[:, :K] = A
    hB = np.zeros((K, ldb), np.float16)
    hB[:, :N] = B
    tA = _host(hA.view(np.int16), pinned)
    tB = _host(hB.view(np.int16), pinned)
    tC = _host(np.full((M, ldc), np.nan, np.float32), pinned)
    st = tct.gemm_f16_f32_host(tA.data_ptr(), tB.data_ptr(), tC.data_ptr(), M, N, K, lda, ldb, ldc, _stream())
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    C = tC.numpy()
    assert np.isnan(C[:, N:]).all(), "columns past N were written"
    return C[:, :N].copy()


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 200, 150), (2100, 777, 515), (4097, 1000, 64),
                                   (17, 4097, 31), (1, 1000, 64)])
def test_gemm_host_matches_oracle(M, N, K, pinned):
    A, B = inputs.normal_pair(np.random.default_rng(M + N + K), M, N, K)
    C = _gemm_host(A, B, M, N, K, pinned)
    assert within_tol(C, oracle.gemm_f32(A, B), K)


def test_gemm_host_integer_exact_with_padded_host_rows():
    M, N, K = 2300, 513, 257
    A, B = inputs.integer_pair(np.random.default_rng(5), M, N, K)
    C = _gemm_host(A, B, M, N, K, True, lda=K + 3, ldb=N + 5, ldc=N + 7)
    R = A.astype(np.int64) @ B.astype(np.int64)
    assert np.array_equal(C, R.astype(np.float32))


def test_gemm_host_equals_device_path_on_whole_blocks():
    """Row blocks of whole 256-row tiles: each block's product equals the device call's rows."""
    M, N, K = 2048, 1024, 512
    A, B = inputs.normal_pair(np.random.default_rng(9), M, N, K)
    C = _gemm_host(A, B, M, N, K, True)
    dA = torch.from_numpy(A.view(np.int16)).cuda().view(torch.float16)
    dB = torch.from_numpy(B.view(np.int16)).cuda().view(torch.float16)
    ref = tct.matmul(dA, dB).cpu().numpy()
    assert within_tol(C, oracle.gemm_f32(A, B), K)
    assert np.abs(C - ref).max() <= 1e-3 * np.sqrt(K)


def test_gemm_host_k_zero_and_back_to_back():
    C = _gemm_host(np.zeros((300, 0), np.float16), np.zeros((0, 40), np.float16), 300, 40, 0, True)
    assert np.all(C == 0)
    # three calls queued on one stream without a sync in between
    outs, refs = [], []
    keep = []
    for seed in range(3):
        A, B = inputs.normal_pair(np.random.default_rng(20 + seed), 700, 300, 200)
        tA, tB = _host(A.view(np.int16), True), _host(B.view(np.int16), True)
        tC = _host(np.zeros((700, 300), np.float32), True)
        keep += [tA, tB]
        assert tct.gemm_f16_f32_host(tA.data_ptr(), tB.data_ptr(), tC.data_ptr(), 700, 300, 200, 200, 300, 300,
                                     _stream()) == tct.GEMM_OK
        outs.append(tC)
        refs.append((A, B))
    torch.cuda.synchronize()
    for tC, (A, B) in zip(outs, refs):
        assert within_tol(tC.numpy(), oracle.gemm_f32(A, B), 200)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M,N", [(1, 1), (9, 37), (4096, 1024), (1000, 3000), (33, 20000), (7, 200003)])
def test_softmax_host_matches_oracle(M, N, pinned):
    X = inputs.normal_f32(np.random.default_rng(M * 7 + N), M, N)
    tX = _host(X, pinned)
    tY = _host(np.zeros_like(X), pinned)
    assert tct.softmax_rows_f32_host(tX.data_ptr(), tY.data_ptr(), M, N, N, N, _stream()) == tct.GEMM_OK
    torch.cuda.synchronize()
    Y = tY.numpy()
    R = oracle.softmax_rows_f32(X).astype(np.float64)
    d = np.abs(X.astype(np.float64) - X.max(axis=1, keepdims=True))
    n = 64 + np.ceil(N / 256)
    tol = 2.0 ** -24 * (32 + 3 * d + 6 * d.max(axis=1, keepdims=True) + 7 * n) * R + 1e-37
    assert np.all(np.abs(Y - R) <= tol)
    # the device-buffer entry point on the same rows gives the same bits (same kernels)
    dev = tct.softmax(torch.from_numpy(X).cuda()).cpu().numpy()
    if N % 4 == 0:
        assert np.array_equal(Y, dev)


def test_softmax_host_in_place_and_padded():
    M, N, ld = 600, 1000, 1003
    X = inputs.normal_f32(np.random.default_rng(3), M, N)
    buf = np.full((M, ld), np.float32(-5.0))
    buf[:, :N] = X
    t = _host(buf, True)
    assert tct.softmax_rows_f32_host(t.data_ptr(), t.data_ptr(), M, N, ld, ld, _stream()) == tct.GEMM_OK
    torch.cuda.synchronize()
    Y = t.numpy()
    assert np.all(Y[:, N:] == -5.0)
    assert np.allclose(Y[:, :N], oracle.softmax_rows_f32(X), rtol=1e-5, atol=1e-37)
