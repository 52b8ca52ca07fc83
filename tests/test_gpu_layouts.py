"""GPU parity for the other operand layouts and BF16 (gemm_f32acc through the C ABI):
A and/or B stored transposed, FP16 or BF16, against the oracle's generalised definition."""
import itertools

import numpy as np
import pytest

import oracle
import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs
from tests.parity import bit_exact, within_tol, worst_ratio

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

LAYOUTS = [(dt, ta, tb) for dt in ("f16", "bf16") for ta, tb in itertools.product([False, True], repeat=2)]


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK


def _dev(x, dt):
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()
    return t.view(torch.float16 if dt == "f16" else torch.bfloat16)


def run(A, B, dt, ta, tb, M, N, K, **opts):
    """C = op(A) op(B) with A, B as stored (numpy), through the raw C ABI."""
    dA, dB = _dev(A, dt), _dev(B, dt)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = tct.gemm_f32acc(tct.GEMM_DTYPE_F16 if dt == "f16" else tct.GEMM_DTYPE_BF16, int(ta), int(tb),
                         dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, A.shape[1], B.shape[1], N,
                         torch.cuda.current_stream().cuda_stream, **opts)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    return C.cpu().numpy()


def ref(A, B, dt, ta, tb):
    return oracle.gemm_ex_f32(A, B, dtype=oracle.F16 if dt == "f16" else oracle.BF16, trans_a=ta, trans_b=tb)


@pytest.mark.parametrize("dt,ta,tb", LAYOUTS)
def test_ragged_and_multi_tile_shapes(dt, ta, tb):
    rng = np.random.default_rng(61)
    for (M, N, K) in list(inputs.RAGGED_SHAPES) + [(256, 512, 128), (777, 1500, 515), (1, 1, 1)]:
        A, B = inputs.pair_ex(rng, M, N, K, dtype=dt, trans_a=ta, trans_b=tb)
        C = run(A, B, dt, ta, tb, M, N, K)
        R = ref(A, B, dt, ta, tb)
        assert within_tol(C, R, K), (M, N, K, worst_ratio(C, R, K))


@pytest.mark.parametrize("dt,ta,tb", LAYOUTS)
def test_integer_inputs_bit_exact(dt, ta, tb):
    rng = np.random.default_rng(62)
    for (M, N, K) in [(300, 200, 150), (17, 4097, 31), (700, 900, 1100)]:
        A, B = inputs.pair_ex(rng, M, N, K, dtype=dt, integer=True, trans_a=ta, trans_b=tb)
        assert bit_exact(run(A, B, dt, ta, tb, M, N, K), ref(A, B, dt, ta, tb)), (M, N, K)


@pytest.mark.parametrize("dt,ta,tb", LAYOUTS)
@pytest.mark.parametrize("opts", [dict(cta_group=2, tile_n=256), dict(cta_group=1, tile_n=256),
                                  dict(cta_group=1, tile_n=128), dict(cta_group=2, tile_n=128),
                                  dict(cta_group=2, tile_n=192),
                                  dict(stream_k=2, cta_group=2, tile_n=256)])
def test_every_planner_variant(dt, ta, tb, opts):
    rng = np.random.default_rng(63)
    M, N, K = 1000, 1100, 700
    A, B = inputs.pair_ex(rng, M, N, K, dtype=dt, trans_a=ta, trans_b=tb)
    C = run(A, B, dt, ta, tb, M, N, K, **opts)
    assert within_tol(C, ref(A, B, dt, ta, tb), K)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_layouts_agree_bitwise_on_the_same_logical_operands(dt):
    """The same logical A and B in any storage give the same bits (the tensor core sees the
    same tiles; only their shared-memory arrangement differs)."""
    rng = np.random.default_rng(64)
    M, N, K = 640, 768, 576
    A, B = inputs.pair_ex(rng, M, N, K, dtype=dt)
    base = run(A, B, dt, False, False, M, N, K)
    for ta, tb in [(True, False), (False, True), (True, True)]:
        As = np.ascontiguousarray(A.T) if ta else A
        Bs = np.ascontiguousarray(B.T) if tb else B
        got = run(As, Bs, dt, ta, tb, M, N, K)
        assert np.array_equal(got.view(np.int32), base.view(np.int32)), (ta, tb)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_identity_and_permutation_transposed(dt):
    rng = np.random.default_rng(65)
    n = 384
    X = inputs.pair_ex(rng, 300, n, n, dtype=dt)[0]            # 300 x n
    perm = rng.permutation(n)
    P = np.zeros((n, n), np.float32)
    P[np.arange(n), perm] = 1.0
    P16 = P.astype(np.float16) if dt == "f16" else inputs.to_bf16_bits(P)
    xval = X.astype(np.float32) if dt == "f16" else torch.from_numpy(X.view(np.int16)).view(
        torch.bfloat16).float().numpy()
    # X stored transposed times a transposed permutation: (X P) = X[:, inv]
    C = run(np.ascontiguousarray(X.T), np.ascontiguousarray(P16.T), dt, True, True, 300, n, n)
    assert np.array_equal(C, xval[:, np.argsort(perm)])


def test_matmul_maps_views_to_layouts():
    """The binding passes transposed views as transposed storage and bf16 tensors as BF16."""
    rng = np.random.default_rng(66)
    M, N, K = 300, 260, 200
    for dt in ("f16", "bf16"):
        A, B = inputs.pair_ex(rng, M, N, K, dtype=dt)
        R = ref(A, B, dt, False, False)
        dA, dB = _dev(A, dt), _dev(B, dt)
        dAt = _dev(np.ascontiguousarray(A.T), dt).t()   # column-major view of A
        dBt = _dev(np.ascontiguousarray(B.T), dt).t()
        for a, b in [(dA, dB), (dAt, dB), (dA, dBt), (dAt, dBt)]:
            C = tct.matmul(a, b)
            torch.cuda.synchronize()
            assert within_tol(C.cpu().numpy(), R, K)


@pytest.mark.parametrize("dt,ta,tb", [("bf16", False, False), ("f16", True, False), ("bf16", True, True)])
def test_square_4096_sampled(dt, ta, tb):
    rng = np.random.default_rng(2)
    M = N = K = 4096
    A, B = inputs.pair_ex(rng, M, N, K, dtype=dt, trans_a=ta, trans_b=tb)
    dA, dB = _dev(A, dt), _dev(B, dt)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = tct.gemm_f32acc(tct.GEMM_DTYPE_F16 if dt == "f16" else tct.GEMM_DTYPE_BF16, int(ta), int(tb),
                         dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K if not ta else M,
                         N if not tb else K, N, torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    rr = np.random.default_rng(0)
    rows = np.concatenate([[0, M - 1, 255, 256], rr.integers(0, M, 300)])
    cols = np.concatenate([[N - 1, 0, 255, 256], rr.integers(0, N, 300)])
    _, want = oracle.gemm_ex_elems(A, B, rows, cols, dtype=oracle.F16 if dt == "f16" else oracle.BF16,
                                   trans_a=ta, trans_b=tb)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    assert within_tol(got, want, K)
