"""Failure detection without a GPU fault.

Every pipeline and cross-CTA wait in the kernel is bounded by `timeout_ms`; when one runs
out, the kernel records GEMM_ERR_DEVICE_TIMEOUT in a device word, winds down (drains its
own copies and MMAs, frees tensor memory) and returns.  The test injects the failure from
the host: with fault_inject bit 0 a split tile is never published -- with the plain FP32
epilogue its owner never zeroes and flags its rows of C, so both halves' waits to add into
C run out; with an epilogue the second half's unit never publishes its part, so the
owner's wait runs out.  Either way the wait is on a flag nothing sets.  With bit 1 and
beta != 0 the epilogue's TMA loads of C are never issued, so its waits for C's blocks run
out.  The host reads the status, and the same context then computes a correct product.
"""
import time

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


def _dev16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)


@pytest.mark.parametrize("opts", [dict(cta_group=2, tile_n=256, max_ctas=150),
                                  dict(cta_group=1, tile_n=256, max_ctas=140)])
@pytest.mark.parametrize("through_workspace", [False, True])
def test_unpublished_part_times_out_and_context_survives(opts, through_workspace):
    M, N, K = 2000, 3000, 1000
    plan = tct.gemm_f16_f32_plan(M, N, K, stream_k=2, **opts)
    assert 0 < plan["stream_k_tiles"] < plan["tiles"]
    rng = np.random.default_rng(51)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = _dev16(A), _dev16(B)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    C = torch.full((M, N), float("nan"), device="cuda")
    t0 = time.time()
    if through_workspace:  # a bias (of zeros) makes the epilogue non-plain: workspace combination
        tct.gemm(dA, dB, C, bias=torch.zeros(N, device="cuda"), stream_k=2, timeout_ms=50, fault_inject=1, **opts)
    else:
        tct.matmul(dA, dB, C, stream_k=2, timeout_ms=50, fault_inject=1, **opts)
    status = tct.gemm_f16_f32_get_error()  # synchronises
    elapsed = time.time() - t0
    assert status == tct.GEMM_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0
    # the whole tiles are complete and correct; the split tiles' owners stored nothing
    host = C.cpu().numpy()
    R = oracle.gemm_f32(A, B)
    done = np.isfinite(host)
    assert done.any() and not done.all()
    assert within_tol(host[done], R[done], K)
    # the error word was cleared by the read, and the context computes correctly again
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    C2 = tct.matmul(dA, dB, stream_k=2, **opts)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    assert within_tol(C2.cpu().numpy(), oracle.gemm_f32(A, B), K)


@pytest.mark.parametrize("c_dtype", [torch.float32, torch.bfloat16])
def test_missing_c_load_times_out_and_context_survives(c_dtype):
    """beta != 0 with a C that TMA writes: the epilogue TMA-loads each block of C before it
    adds beta * C; with fault_inject bit 1 those loads are never issued, every epilogue's
    first wait runs out, nothing is stored, and the next call is correct."""
    M, N, K = 1000, 1024, 256
    rng = np.random.default_rng(52)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = _dev16(A), _dev16(B)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    C0 = torch.randn(M, N, device="cuda").to(c_dtype)
    C = C0.clone()
    t0 = time.time()
    tct.gemm(dA, dB, C, beta=1.0, timeout_ms=50, fault_inject=2, stream_k=1)  # whole tiles only
    status = tct.gemm_f16_f32_get_error()
    assert status == tct.GEMM_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 5.0
    assert torch.equal(C.view(torch.int16 if c_dtype != torch.float32 else torch.int32),
                       C0.view(torch.int16 if c_dtype != torch.float32 else torch.int32))
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    tct.gemm(dA, dB, C, beta=1.0)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    want = oracle.gemm_f32(A, B).astype(np.float64) + C0.double().cpu().numpy()
    got = C.double().cpu().numpy()
    ulp = 0.0 if c_dtype == torch.float32 else 2.0 ** -7
    tol = 1e-3 * np.sqrt(K) * np.maximum(1.0, np.abs(want)) + 2 * ulp * np.abs(want)
    assert np.all(np.abs(got - want) <= tol)


@pytest.mark.parametrize("M,N,K,chained", [(4096, 4096, 1024, False), (1024, 1024, 16384, True)])
def test_unpublished_stream_k_piece_times_out_and_context_survives(M, N, K, chained):
    """Stream-K with fault_inject bit 0.  Tiles of two pieces: the piece that starts a tile
    never zeroes and flags its rows of C, so both pieces' waits run out.  Longer chains: a
    piece that starts inside a tile never raises its flag, so the unit before it, whose piece
    of that tile waits to add into C, runs out of time.  The status is read on the host, the
    tiles computed whole are correct, and the next call on the same context is correct
    everywhere."""
    opts = dict(stream_k=3)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = tct.gemm_f16_f32_plan(M, N, K, num_sms=sms, **opts)
    assert plan["split_form"] == 2 and 0 < plan["stream_k_tiles"] <= plan["tiles"]
    assert (plan["split_parts_per_unit"] > 2) == chained
    rng = np.random.default_rng(57)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = _dev16(A), _dev16(B)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    C = torch.full((M, N), float("nan"), device="cuda")
    t0 = time.time()
    tct.matmul(dA, dB, C, timeout_ms=50, fault_inject=1, **opts)
    status = tct.gemm_f16_f32_get_error()
    assert status == tct.GEMM_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 5.0
    host = C.cpu().numpy()
    R = oracle.gemm_f32(A, B)
    tm, tn = plan["tile_m"], plan["tile_n"]
    num_m, num_n = -(-M // tm), -(-N // tn)
    # the whole tiles every unit computes before its stream-K range (a unit whose wait ran out
    # stops there, so whole tiles inside the stream-K region may be left unwritten)
    dp_tiles = plan["tiles"] - plan["stream_k_tiles"]
    whole = []
    for u in range(plan["units"]):
        idx = 0
        while True:
            it = tct.gemm_f16_f32_work_item(M, N, K, sms, u, idx, **opts)
            if it is None:
                break
            if it["mode"] == tct.WORK_STORE and it["tile"] < dp_tiles:
                whole.append(it["tile"])
            idx += 1
    for t in whole:
        r, c = tct.gemm_tile_coord(t, num_m, num_n, plan["group_m"])
        blk = (slice(r * tm, min(M, (r + 1) * tm)), slice(c * tn, min(N, (c + 1) * tn)))
        assert within_tol(host[blk], R[blk], K)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    C2 = tct.matmul(dA, dB, **opts)
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    assert within_tol(C2.cpu().numpy(), R, K)


@pytest.mark.parametrize("dt,ta,tb", [("bf16", False, False), ("f16", True, True), ("f16", True, False)])
def test_timeout_in_every_kernel_object_is_reported(dt, ta, tb):
    """The kernels of BF16 and of both-transposed operands are built in a second object with
    its own device error word; a wait that runs out there is reported by the same status call
    and cleared by it, like one in the first object's kernels (A transposed, FP16); the next
    call then gives the oracle's result."""
    M, N, K = 2000, 3000, 1000
    rng = np.random.default_rng(53)
    A, B = inputs.pair_ex(rng, M, N, K, dtype=dt, trans_a=ta, trans_b=tb)
    tdt = torch.float16 if dt == "f16" else torch.bfloat16
    dA = torch.from_numpy(np.ascontiguousarray(A).view(np.int16)).cuda().view(tdt)
    dB = torch.from_numpy(np.ascontiguousarray(B).view(np.int16)).cuda().view(tdt)
    C = torch.full((M, N), float("nan"), device="cuda")
    ab = tct.GEMM_DTYPE_F16 if dt == "f16" else tct.GEMM_DTYPE_BF16
    opts = dict(stream_k=2, cta_group=2, tile_n=256, max_ctas=150)

    def call(**extra):
        return tct.gemm_f32acc(ab, int(ta), int(tb), dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K,
                               A.shape[1], B.shape[1], N, torch.cuda.current_stream().cuda_stream, **opts, **extra)

    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    assert call(timeout_ms=50, fault_inject=1) == tct.GEMM_OK
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_ERR_DEVICE_TIMEOUT
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    assert call() == tct.GEMM_OK
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    R = oracle.gemm_ex_f32(A, B, dtype=oracle.F16 if dt == "f16" else oracle.BF16, trans_a=ta, trans_b=tb)
    assert within_tol(C.cpu().numpy(), R, K)
