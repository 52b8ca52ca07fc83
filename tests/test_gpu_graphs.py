"""The library's calls inside CUDA graphs: captured once on a stream and replayed with new
operand contents (the graph keeps the buffers, the values change), each replay checked
against the oracle.  Covers the whole-tile path, split tiles (flags and their clearing are
part of the graph), an epilogue with beta != 0, a repacked (unaligned) operand and the
softmax, all launched as they are outside a graph (programmatic dependent launches
included)."""
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


def _capture(fn):
    """Runs fn once outside a graph (one-time set-up: attributes, pools, queries), then
    captures it on a side stream and returns the graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _h16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.float16)


@pytest.mark.parametrize("M,N,K,opts", [
    (512, 768, 640, {}),
    (2000, 3000, 1000, dict(stream_k=2)),
    (300, 200, 150, {}),  # K = 150: rows of A are not 16-byte multiples, so A is repacked
])
def test_gemm_graph_replays_with_new_operands(M, N, K, opts):
    dA = torch.empty(M, K, dtype=torch.float16, device="cuda")
    dB = torch.empty(K, N, dtype=torch.float16, device="cuda")
    C = torch.empty(M, N, device="cuda")
    rng = np.random.default_rng(81)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA.copy_(_h16(A))
    dB.copy_(_h16(B))
    g = _capture(lambda: tct.matmul(dA, dB, C, **opts))
    for seed in (82, 83):
        A, B = inputs.normal_pair(np.random.default_rng(seed), M, N, K)
        dA.copy_(_h16(A))
        dB.copy_(_h16(B))
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert within_tol(C.cpu().numpy(), oracle.gemm_f32(A, B), K), (M, N, K, seed)


def test_epilogue_graph_replays():
    M, N, K = 640, 1024, 384
    rng = np.random.default_rng(84)
    dA = torch.empty(M, K, dtype=torch.float16, device="cuda")
    dB = torch.empty(K, N, dtype=torch.float16, device="cuda")
    C = torch.empty(M, N, device="cuda")
    bias = torch.from_numpy(rng.standard_normal(N).astype(np.float32)).cuda()
    g = _capture(lambda: tct.gemm(dA, dB, C, alpha=0.5, beta=1.0, bias=bias))
    for seed in (85, 86):
        A, B = inputs.normal_pair(np.random.default_rng(seed), M, N, K)
        C0 = np.random.default_rng(seed + 100).standard_normal((M, N)).astype(np.float32)
        dA.copy_(_h16(A))
        dB.copy_(_h16(B))
        C.copy_(torch.from_numpy(C0))
        g.replay()
        torch.cuda.synchronize()
        want = 0.5 * oracle.gemm_f32(A, B).astype(np.float64) + C0 + bias.cpu().numpy()[None, :]
        S = np.abs(oracle.gemm_f32(A, B))
        tol = 0.5 * 1e-3 * np.sqrt(K) * np.maximum(1.0, S) + 1e-6 * np.abs(want)
        assert np.all(np.abs(C.cpu().numpy() - want) <= tol), seed


def test_softmax_graph_replays():
    M, N = 4096, 1024
    X = torch.empty(M, N, device="cuda")
    Y = torch.empty(M, N, device="cuda")
    g = _capture(lambda: tct.softmax(X, Y))
    for seed in (87, 88):
        x = inputs.normal_f32(np.random.default_rng(seed), M, N)
        X.copy_(torch.from_numpy(x))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.softmax_rows_f32(x).astype(np.float64)
        assert np.all(np.abs(Y.cpu().numpy() - ref) <= 1e-5 * ref + 1e-37), seed
