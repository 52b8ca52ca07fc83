"""The allocation-free entry point, gemm_f16_f32_noalloc.

It serves callers that cannot allocate device memory themselves or through the library:
their GPU memory belongs to another allocator (a framework's caching pool, a server that
reserves the whole device at start-up), or their interface hands over only the input and
output buffers.  Its only scratch, the aligned copy of operands whose rows TMA cannot read
in place, lives in a fixed library-owned device array.

The test drives it through the C ABI on shapes whose leading dimensions force that copy,
two calls in a row, and compares each result with the allocating entry point's result
within the tolerance the parity tests use.  This file sorts last so that a run stopping
at the first failure has run every other test before it.
"""
import numpy as np
import pytest

import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs
from tests.parity import within_tol

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

# (M, N, K, lda, ldb): the first repacks A only, the others both operands.
SHAPES = [(300, 200, 150, 150, 200), (129, 65, 33, 33, 65), (17, 4097, 31, 31, 4097), (1000, 777, 515, 515, 777)]


def _dev16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


@pytest.mark.parametrize("M,N,K,lda,ldb", SHAPES)
def test_noalloc_matches_allocating_entry_point(M, N, K, lda, ldb):
    rng = np.random.default_rng(31)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = _dev16(A), _dev16(B)
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert tct.gemm_f16_f32(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), M, N, K, lda, ldb, N,
                            stream) == tct.GEMM_OK
    torch.cuda.synchronize()
    ref_h = ref.cpu().numpy()
    for _ in range(2):  # two calls in a row share (and reuse) the scratch array
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = tct.gemm_f16_f32_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, N,
                                      stream)
        assert st == tct.GEMM_OK
        torch.cuda.synchronize()
        assert within_tol(out.cpu().numpy(), ref_h, K)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK


def test_noalloc_aligned_operands_need_no_scratch():
    rng = np.random.default_rng(32)
    M, N, K = 256, 512, 192
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = _dev16(A), _dev16(B)
    s = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert tct.gemm_f16_f32(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), M, N, K, K, N, N, s) == tct.GEMM_OK
    assert tct.gemm_f16_f32_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, K, N, N,
                                    s) == tct.GEMM_OK
    torch.cuda.synchronize()
    assert within_tol(out.cpu().numpy(), ref.cpu().numpy(), K)


def test_noalloc_rejects_scratch_beyond_its_limit():
    # A repack of 5000 x roundup(4001, 8) FP16 elements needs 40 MB > the 32 MiB array.
    M, N, K = 5000, 64, 4001
    dA = torch.zeros(M * K, dtype=torch.float16, device="cuda")
    dB = torch.zeros(K * N, dtype=torch.float16, device="cuda")
    out = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    st = tct.gemm_f16_f32_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, K, N, N,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool(torch.all(out == 7.0))  # nothing was enqueued
