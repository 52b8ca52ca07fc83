"""The allocation-free entry point, gemm_f16_f32_noalloc.

It serves callers that cannot allocate device memory themselves or through the library:
their GPU memory belongs to another allocator (a framework's caching pool, a server that
reserves the whole device at start-up), or their interface hands over only the input and
output buffers.  Its only scratch, the aligned copy of operands whose rows TMA cannot read
in place, lives in a fixed library-owned device array.

The tests drive it through the C ABI on shapes whose leading dimensions force that copy,
two calls in a row, and compare each result with the CPU oracle: within the tolerance of
the parity tests for N(0,1) inputs, bit for bit for integer inputs.  A fresh process checks
the defining property: once the first call has loaded the library, further calls leave the
device's free memory exactly as it was (the allocating entry point, on the same shape,
visibly takes memory, which shows the measurement can see an allocation).  This file sorts
last so that a run stopping at the first failure has run every other test before it.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs
from tests.parity import bit_exact, within_tol, worst_ratio

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (M, N, K, lda, ldb): the first repacks A only, the others both operands.
SHAPES = [(300, 200, 150, 150, 200), (129, 65, 33, 33, 65), (17, 4097, 31, 31, 4097), (1000, 777, 515, 515, 777)]


def _dev16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _noalloc_twice(A, B, M, N, K, lda, ldb):
    """Two calls in a row (they share, and reuse, the scratch array); both results."""
    dA, dB = _dev16(A), _dev16(B)
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = tct.gemm_f16_f32_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, N, stream)
        assert st == tct.GEMM_OK
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    return outs


@pytest.mark.parametrize("M,N,K,lda,ldb", SHAPES)
def test_noalloc_matches_oracle(M, N, K, lda, ldb):
    rng = np.random.default_rng(31)
    A, B = inputs.normal_pair(rng, M, N, K)
    R = oracle.gemm_f32(A, B)
    for out in _noalloc_twice(A, B, M, N, K, lda, ldb):
        assert within_tol(out, R, K), f"worst |err|/tol = {worst_ratio(out, R, K):.3g}"


@pytest.mark.parametrize("M,N,K,lda,ldb", SHAPES)
def test_noalloc_integer_bit_exact(M, N, K, lda, ldb):
    rng = np.random.default_rng(37)
    A, B = inputs.integer_pair(rng, M, N, K)
    R = oracle.gemm_f32(A, B)
    for out in _noalloc_twice(A, B, M, N, K, lda, ldb):
        assert bit_exact(out, R)


def test_noalloc_aligned_operands_need_no_scratch():
    rng = np.random.default_rng(32)
    M, N, K = 256, 512, 192
    A, B = inputs.normal_pair(rng, M, N, K)
    R = oracle.gemm_f32(A, B)
    for out in _noalloc_twice(A, B, M, N, K, K, N):
        assert within_tol(out, R, K)


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


def test_noalloc_rejects_sizes_whose_scratch_overflows():
    # Leading dimensions near the largest accepted value: the scratch size of either operand
    # would not fit in 64 bits, and is rejected before any arithmetic can wrap.  Nothing is
    # read from the (tiny) buffers: the call returns before any device work.
    M, N, K = 2 ** 31 - 1, 1, 2 ** 31 - 1
    dA = torch.zeros(8, dtype=torch.float16, device="cuda")
    out = torch.zeros(8, dtype=torch.float32, device="cuda")
    st = tct.gemm_f16_f32_noalloc(dA.data_ptr() + 2, dA.data_ptr() + 2, out.data_ptr(), M, N, K, K, N, N,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_ERR_INVALID_ARG


_FRESH_PROCESS = r"""
import json, sys
import torch
import tensor_core_tiled_gb300 as tct
tct.load()
M, N, K, lda, ldb = 1000, 777, 515, 515, 777   # rows of A and B both need the aligned copy
dA = torch.randn(M * lda, device="cuda").half()
dB = torch.randn(K * ldb, device="cuda").half()
out = torch.empty(M * N, device="cuda")
s = torch.cuda.current_stream().cuda_stream
def noalloc():
    st = tct.gemm_f16_f32_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, N, s)
    assert st == tct.GEMM_OK, st
torch.cuda.synchronize()
noalloc()                      # first call: loads the library's kernels, looks up the scratch
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for _ in range(5):
    noalloc()
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
st = tct.gemm_f16_f32(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, N, s)
assert st == tct.GEMM_OK, st
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
print(json.dumps({"free_after_first": free0, "free_after_more": free1, "free_after_allocating_call": free2}))
"""


def test_noalloc_allocates_no_device_memory():
    """In a fresh process that calls nothing else of the library first: after the first
    call, five more calls leave cudaMemGetInfo's free bytes unchanged; the allocating entry
    point on the same shape then takes memory from its pool."""
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["free_after_more"] == d["free_after_first"], d
    assert d["free_after_allocating_call"] < d["free_after_more"], d
