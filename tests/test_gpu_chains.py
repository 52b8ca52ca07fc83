"""Dependent launches back to back on one stream, no host synchronisation in between: each
call reads what the previous one wrote.  The GEMM and the staged softmax launch as
programmatic dependent launches (their set-up may overlap the previous kernel, their first
global access waits for it), so these chains check that no call reads its input early."""
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


def _dev16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)


@pytest.mark.parametrize("M,K", [(1024, 1024), (2000, 768)])
def test_gemm_reads_the_previous_gemms_output(M, K):
    """P_i = P_{i-1} . D (FP16 out), eight links queued without a sync; every link is then
    checked against the oracle applied to the previous link's stored bits."""
    rng = np.random.default_rng(91)
    A = inputs.normal_f16(rng, M, K)
    D = (np.random.default_rng(92).standard_normal((K, K)) / np.sqrt(K)).astype(np.float16)
    dD = _dev16(D)
    links = [_dev16(A)]
    for _ in range(8):
        links.append(tct.gemm(links[-1], dD, out_dtype=torch.float16))
    torch.cuda.synchronize()
    host = [x.cpu().numpy() for x in links]
    for i in range(1, len(host)):
        R = oracle.gemm_f32(host[i - 1], D).astype(np.float64)
        got = host[i].astype(np.float64)
        tol = 1e-3 * np.sqrt(K) * np.maximum(1.0, np.abs(R)) + 2.0 ** -10 * np.abs(R)
        assert np.all(np.abs(got - R) <= tol), i
    # and the FP32 product of the last link, also queued right behind it
    C = tct.matmul(links[-1], dD)
    torch.cuda.synchronize()
    assert within_tol(C.cpu().numpy(), oracle.gemm_f32(host[-1], D), K)


def test_softmax_of_a_gemm_and_softmax_of_a_softmax():
    M, N, K = 4096, 1024, 512
    rng = np.random.default_rng(93)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = _dev16(A), _dev16(B)
    for _ in range(4):
        C = tct.matmul(dA, dB)
        S = tct.softmax(C)           # reads the GEMM's output
        S2 = tct.softmax(S)          # reads the first softmax's output
    torch.cuda.synchronize()
    Cg = C.cpu().numpy()
    assert within_tol(Cg, oracle.gemm_f32(A, B), K)
    for x, y in ((Cg, S), (S.cpu().numpy(), S2)):
        ref = oracle.softmax_rows_f32(x).astype(np.float64)
        assert np.all(np.abs(y.cpu().numpy() - ref) <= 1e-5 * ref + 1e-37)
