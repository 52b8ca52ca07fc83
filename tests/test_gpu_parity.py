"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Criteria (tests/parity.py): element-wise |C - R| <= 1e-3 * sqrt(K) * max(1, |R|) for N(0,1)
FP16 inputs; bit-exact FP32 for integer-valued inputs in [-4, 4] (partial sums < 2^24).
Every shape, the full-size workloads included, is compared element by element over the whole
of C.
"""
import numpy as np
import pytest

import oracle
import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs
from tests.parity import bit_exact, within_tol, worst_ratio

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK


def dev16(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)


def gpu_gemm(A, B, **opts):
    C = tct.matmul(dev16(A), dev16(B), **opts)
    torch.cuda.synchronize()
    return C.cpu().numpy()


def check_tol(A, B, C=None, **opts):
    M, K = A.shape
    if C is None:
        C = gpu_gemm(A, B, **opts)
    R = oracle.gemm_f32(A, B)
    assert within_tol(C, R, K), f"worst |err|/tol = {worst_ratio(C, R, K):.3g}"
    return C, R


def test_square_256_seed0():
    (M, N, K), A, B = inputs.workload("square256")[0]
    C, R = check_tol(A, B)
    err = np.abs(C.astype(np.float64) - oracle.gemm_f64(A, B)).max()
    # FP32 accumulation error of a 256-term sum: small but not the FP64 result
    assert 1e-7 < err < 1e-4


@pytest.mark.parametrize("idx", range(len(inputs.RAGGED_SHAPES)))
def test_ragged_normal(idx):
    (M, N, K), A, B = inputs.workload("ragged")[idx]
    check_tol(A, B)


@pytest.mark.parametrize("idx", range(len(inputs.RAGGED_SHAPES)))
def test_ragged_integer_bit_exact(idx):
    (M, N, K), A, B = inputs.workload("ragged_int")[idx]
    C = gpu_gemm(A, B)
    assert bit_exact(C, oracle.gemm_f32(A, B))


def test_mma_tile_16x8x16():
    rng = np.random.default_rng(0)
    worst = 0.0
    for _ in range(20):
        A = rng.standard_normal((16, 16)).astype(np.float16)
        B = rng.standard_normal((16, 8)).astype(np.float16)
        C, R = check_tol(A, B)
        worst = max(worst, float(np.abs(C.astype(np.float64) - oracle.gemm_f64(A, B)).max()))
    assert worst < 1e-5


@pytest.mark.parametrize("shape", [(64, 64, 64), (128, 64, 96), (1, 1, 1), (17, 33, 65), (100, 70, 50),
                                   (64, 64, 40), (128, 256, 64), (129, 257, 65), (255, 511, 127)])
def test_edge_shapes(shape):
    M, N, K = shape
    rng = np.random.default_rng(3)
    A, B = inputs.normal_pair(rng, M, N, K)
    check_tol(A, B)


def test_identity_and_permutation():
    rng = np.random.default_rng(5)
    n = 384
    X = rng.standard_normal((n, 300)).astype(np.float16)
    eye = np.eye(n, dtype=np.float16)
    assert np.array_equal(gpu_gemm(eye, X), X.astype(np.float32))
    Y = rng.standard_normal((200, n)).astype(np.float16)
    assert np.array_equal(gpu_gemm(Y, eye), Y.astype(np.float32))
    perm = rng.permutation(n)
    P = np.zeros((n, n), np.float16)
    P[np.arange(n), perm] = 1.0
    assert np.array_equal(gpu_gemm(P, X), X[perm].astype(np.float32))
    assert np.array_equal(gpu_gemm(Y, P), Y[:, np.argsort(perm)].astype(np.float32))


def test_integer_bit_exact_multi_tile():
    rng = np.random.default_rng(1)
    A, B = inputs.integer_pair(rng, 1000, 1300, 2048)
    C = gpu_gemm(A, B)
    assert bit_exact(C, oracle.gemm_f32(A, B))


def test_k_zero_and_empty_outputs():
    A = torch.empty((5, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((0, 7), dtype=torch.float16, device="cuda")
    C = torch.full((5, 7), 3.0, device="cuda")
    tct.matmul(A, B, C)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
    C2 = torch.full((0, 7), 3.0, device="cuda")
    tct.matmul(torch.empty((0, 4), dtype=torch.float16, device="cuda"),
               torch.ones((4, 7), dtype=torch.float16, device="cuda"), C2)
    torch.cuda.synchronize()


@pytest.mark.parametrize("cta_group,tile_n", [(1, 128), (1, 256), (2, 128), (2, 192), (2, 256)])
@pytest.mark.parametrize("off", [1, 2, 3])
def test_unaligned_c_every_variant(cta_group, tile_n, off):
    """Every tile shape writing a C whose rows start 4 * off bytes past a 16-byte boundary
    (row pitch 1001 floats, so consecutive rows shift by one more element): the oracle's
    result bit for bit on integer inputs, with units of one and of several tiles, and the NaN
    guard zones around and between the rows untouched."""
    M, N, K, ldc = 1000, 1000, 320, 1001
    rng = np.random.default_rng(62 + off)
    Ai, Bi = inputs.integer_pair(rng, M, N, K)
    guard = 4096
    for max_ctas in (0, 16):
        c_buf = torch.full((guard + off + M * ldc + guard,), float("nan"), dtype=torch.float32, device="cuda")
        c_base = c_buf.data_ptr() + (guard + off) * 4
        dAi, dBi = dev16(Ai), dev16(Bi)  # kept alive until the call has run
        st = tct.gemm_f16_f32_ex(dAi.data_ptr(), dBi.data_ptr(), c_base, M, N, K, K, N, ldc,
                                 torch.cuda.current_stream().cuda_stream, cta_group=cta_group, tile_n=tile_n,
                                 max_ctas=max_ctas)
        assert st == tct.GEMM_OK
        torch.cuda.synchronize()
        host = c_buf.cpu().numpy()
        assert np.all(np.isnan(host[:guard + off])) and np.all(np.isnan(host[guard + off + M * ldc:]))
        body = host[guard + off:guard + off + M * ldc].reshape(M, ldc)
        assert np.all(np.isnan(body[:, N:]))
        assert bit_exact(body[:, :N], oracle.gemm_f32(Ai, Bi))


@pytest.mark.parametrize("M,N,K,pad_a,pad_b,pad_c,off", [
    (300, 200, 150, 7, 5, 3, 0),
    (129, 65, 33, 0, 0, 0, 1),
    (256, 512, 128, 8, 16, 4, 0),
    (17, 4097, 31, 1, 3, 9, 1),
])
def test_leading_dims_offsets_and_guard_zones(M, N, K, pad_a, pad_b, pad_c, off):
    """lda > K, ldb > N, ldc > N, bases offset by one element (repack path), NaN guard zones
    around C and in its gap columns: only the M x N block may change."""
    rng = np.random.default_rng(17)
    A, B = inputs.normal_pair(rng, M, N, K)
    lda, ldb, ldc = K + pad_a, N + pad_b, N + pad_c
    guard = 4096
    a_buf = torch.zeros(off + M * lda + 8, dtype=torch.float16, device="cuda")
    b_buf = torch.zeros(off + K * ldb + 8, dtype=torch.float16, device="cuda")
    c_buf = torch.full((guard + M * ldc + guard,), float("nan"), dtype=torch.float32, device="cuda")
    a_view = a_buf[off:off + M * lda].view(M, lda)
    b_view = b_buf[off:off + K * ldb].view(K, ldb)
    a_view[:, :K] = dev16(A)
    b_view[:, :N] = dev16(B)
    c_base = c_buf.data_ptr() + guard * 4
    st = tct.gemm_f16_f32(a_view.data_ptr(), b_view.data_ptr(), c_base, M, N, K, lda, ldb, ldc,
                          torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    host = c_buf.cpu().numpy()
    assert np.all(np.isnan(host[:guard])) and np.all(np.isnan(host[guard + M * ldc:]))
    body = host[guard:guard + M * ldc].reshape(M, ldc)
    assert np.all(np.isnan(body[:, N:]))
    R = oracle.gemm_f32(A, B)
    assert within_tol(body[:, :N], R, K)


@pytest.mark.parametrize("M,N,K,ldc,opts", [
    (300, 201, 150, 204, dict(stream_k=1)),
    (300, 201, 150, 204, dict(stream_k=2)),
    (5, 7, 154, 8, {}),
    (257, 516, 100, 520, dict(stream_k=1)),
    (257, 516, 100, 520, dict(stream_k=2)),
    (3000, 2050, 700, 2052, dict(stream_k=2)),
    (1000, 1024, 64, 1024, dict(stream_k=2, cta_group=1, tile_n=128)),
])
def test_aligned_c_padding_bits_untouched(M, N, K, ldc, opts):
    """A 16-byte aligned C with ldc % 4 == 0, whole tiles and split tiles: the columns
    between N and ldc and the rows around C keep their bits (-0.0, which an added zero would
    turn into +0.0), also when N is not a multiple of 4 and the last 16 bytes of a row are
    only partly inside the M x N block."""
    rng = np.random.default_rng(19)
    A, B = inputs.normal_pair(rng, M, N, K)
    guard = 1024
    c_buf = torch.full((guard + M * ldc + guard,), -0.0, dtype=torch.float32, device="cuda")
    c_base = c_buf.data_ptr() + guard * 4
    dA, dB = dev16(A), dev16(B)
    st = tct.gemm_f16_f32_ex(dA.data_ptr(), dB.data_ptr(), c_base, M, N, K, K, N, ldc,
                             torch.cuda.current_stream().cuda_stream, **opts)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    bits = c_buf.view(torch.int32).cpu().numpy()
    neg0 = np.int32(-2 ** 31)
    assert np.all(bits[:guard] == neg0) and np.all(bits[guard + M * ldc:] == neg0)
    body = bits[guard:guard + M * ldc].reshape(M, ldc)
    assert np.all(body[:, N:] == neg0)
    assert within_tol(body[:, :N].view(np.float32), oracle.gemm_f32(A, B), K)


@pytest.mark.parametrize("M,N,K", [(70001, 24, 33), (60000, 25, 10001), (1793, 1793, 1793), (5, 3, 70001)])
def test_repack_tall_wide_and_narrow_operands(M, N, K):
    """Operands with unaligned rows are copied by a kernel that gives each row a group of
    lanes sized to it: tall operands with short rows (several rows per warp), long rows (a
    warp per row, several 16-byte units per lane) and both operands in one launch."""
    rng = np.random.default_rng(19)
    A, B = inputs.normal_pair(rng, M, N, K)
    plan = tct.gemm_f16_f32_plan(M, N, K)
    assert plan["pack_a"] == 1
    check_tol(A, B)


def test_repeat_runs_bitwise_identical():
    rng = np.random.default_rng(21)
    A, B = inputs.normal_pair(rng, 1000, 1100, 700)
    dA, dB = dev16(A), dev16(B)
    first = tct.matmul(dA, dB).cpu()
    for _ in range(9):
        again = tct.matmul(dA, dB).cpu()
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))


VARIANT_OPTS = [
    dict(cta_group=1, tile_n=256, stages=2), dict(cta_group=1, tile_n=256, stages=3),
    dict(cta_group=1, tile_n=256, stages=4, group_m=1), dict(cta_group=1, tile_n=128, stages=4),
    dict(cta_group=1, tile_n=128, stages=6, group_m=3), dict(cta_group=1, tile_n=256, max_ctas=7),
    dict(cta_group=2, tile_n=256, stages=3), dict(cta_group=2, tile_n=256, stages=4, group_m=16),
    dict(cta_group=2, tile_n=256, stages=5), dict(cta_group=2, tile_n=256, stages=6, group_m=1),
    dict(cta_group=2, tile_n=128, stages=6), dict(cta_group=2, tile_n=128, stages=8, group_m=4),
    dict(cta_group=2, tile_n=256, max_ctas=6), dict(cta_group=2, tile_n=128, max_ctas=2),
    dict(cta_group=2, tile_n=192), dict(cta_group=2, tile_n=192, group_m=5, max_ctas=10),
]


@pytest.mark.parametrize("opts", VARIANT_OPTS)
def test_variants_and_schedules_agree(opts):
    """For a given CTA grouping and tile width, with whole tiles only, every pipeline depth,
    launch order and grid size gives the same bits (the k order inside a tile never
    changes); every variant passes the oracle."""
    rng = np.random.default_rng(23)
    M, N, K = 777, 1500, 515
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = dev16(A), dev16(B)
    ref = tct.matmul(dA, dB, cta_group=opts["cta_group"], tile_n=opts["tile_n"], stream_k=1)
    C = tct.matmul(dA, dB, stream_k=1, **opts)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int32), ref.view(torch.int32))
    assert within_tol(C.cpu().numpy(), oracle.gemm_f32(A, B), K)


def test_pair_and_single_cta_tiles_agree():
    rng = np.random.default_rng(29)
    M, N, K = 1000, 1024, 1000
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = dev16(A), dev16(B)
    one = tct.matmul(dA, dB, cta_group=1, tile_n=256)
    two = tct.matmul(dA, dB, cta_group=2, tile_n=256)
    torch.cuda.synchronize()
    R = oracle.gemm_f32(A, B)
    assert within_tol(one.cpu().numpy(), R, K) and within_tol(two.cpu().numpy(), R, K)


@pytest.mark.parametrize("cta_group,tile_n", [(1, 128), (1, 256), (2, 128), (2, 192), (2, 256)])
def test_every_variant_on_ragged_and_integer_inputs(cta_group, tile_n):
    for (M, N, K), A, B in inputs.workload("ragged"):
        C = gpu_gemm(A, B, cta_group=cta_group, tile_n=tile_n)
        assert within_tol(C, oracle.gemm_f32(A, B), K), (M, N, K)
    for (M, N, K), A, B in inputs.workload("ragged_int"):
        C = gpu_gemm(A, B, cta_group=cta_group, tile_n=tile_n)
        assert bit_exact(C, oracle.gemm_f32(A, B)), (M, N, K)
    rng = np.random.default_rng(33)
    A, B = inputs.integer_pair(rng, 700, 900, 1100)
    assert bit_exact(gpu_gemm(A, B, cta_group=cta_group, tile_n=tile_n), oracle.gemm_f32(A, B))


STREAM_K_CASES = [
    ((1000, 1100, 700), dict(stream_k=2)),
    ((777, 1500, 515), dict(stream_k=2, cta_group=1, tile_n=256)),
    ((777, 1000, 515), dict(stream_k=2, cta_group=1, tile_n=128)),
    ((300, 200, 150), dict(stream_k=2)),
    ((129, 65, 33 * 64), dict(stream_k=2, cta_group=1)),
    ((2000, 3000, 5000), dict(stream_k=2, max_ctas=150)),
    ((2000, 3000, 5000), dict(stream_k=2, cta_group=1, tile_n=256, max_ctas=140)),
    ((1, 1000, 640), dict(stream_k=2, cta_group=1, tile_n=128)),
    ((4096, 4096, 1000), dict(stream_k=2, cta_group=2, tile_n=256)),
    # tails larger than half the units: helpers take 2, 6 and 9 second parts in turn
    ((6144, 6144, 1000), dict(stream_k=2)),
    ((2048, 2048, 2048), dict(stream_k=2)),
    ((3072, 3072, 1024), dict(stream_k=2)),
    ((1500, 5000, 777), dict(stream_k=2, cta_group=1, tile_n=128)),
    ((3000, 4000, 1000), dict(stream_k=2, cta_group=2, tile_n=192)),
]


@pytest.mark.parametrize("shape,opts", STREAM_K_CASES)
def test_stream_k_split(shape, opts):
    """Tiles whose k-loop is split in two parts on two units (both parts added into C by TMA
    reduce-add; a helper may take several tiles' second parts in turn) give the oracle's
    result, bit-exact on integer inputs, and the same bits on every run."""
    M, N, K = shape
    plan = tct.gemm_f16_f32_plan(M, N, K, **opts)
    assert plan["stream_k_tiles"] > 0
    rng = np.random.default_rng(41)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = dev16(A), dev16(B)
    C = tct.matmul(dA, dB, **opts)
    again = tct.matmul(dA, dB, **opts)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int32), again.view(torch.int32))
    assert within_tol(C.cpu().numpy(), oracle.gemm_f32(A, B), K)
    Ai, Bi = inputs.integer_pair(rng, M, N, K)
    assert bit_exact(gpu_gemm(Ai, Bi, **opts), oracle.gemm_f32(Ai, Bi))


STREAM_K_CHAIN_CASES = [
    ((1792, 1792, 1792), {}),
    ((2048, 2048, 2048), {}),
    ((1000, 1100, 700), {}),
    ((300, 200, 150), {}),
    ((256, 256, 4096), {}),                      # one pair tile spread over many units
    ((128, 4096, 8192), {"cta_group": 1, "tile_n": 128}),
    ((128, 4096, 8192), {"cta_group": 2}),       # the pair's second 128 rows are empty
    ((3000, 2052, 1500), {"cta_group": 1, "tile_n": 256}),
    ((4096, 4096, 1024), {}),
    ((777, 1500, 515), {"max_ctas": 40}),
    ((129, 68, 64 * 33), {"cta_group": 1, "tile_n": 128}),
    ((1000, 1000, 3000), {"cta_group": 2, "tile_n": 192}),
]


@pytest.mark.parametrize("shape,opts", STREAM_K_CHAIN_CASES)
def test_stream_k_chain(shape, opts):
    """Stream-K plans (balanced k-ranges per unit, a tile's pieces chained into C last-first
    by TMA store and reduce-adds): the oracle's result over the whole matrix, bit for bit on
    integer inputs, and the same bits on every run (the chain fixes the order of the sums)."""
    M, N, K = shape
    opts = dict(opts, stream_k=3)
    plan = tct.gemm_f16_f32_plan(M, N, K, **opts)
    assert plan["split_form"] == 2
    rng = np.random.default_rng(47)
    A, B = inputs.normal_pair(rng, M, N, K)
    dA, dB = dev16(A), dev16(B)
    C = tct.matmul(dA, dB, **opts)
    torch.cuda.synchronize()
    first = C.clone()
    for _ in range(3):
        tct.matmul(dA, dB, C, **opts)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int32), first.view(torch.int32))
    assert within_tol(C.cpu().numpy(), oracle.gemm_f32(A, B), K)
    Ai, Bi = inputs.integer_pair(rng, M, N, K)
    assert bit_exact(gpu_gemm(Ai, Bi, **opts), oracle.gemm_f32(Ai, Bi))


def test_stream_k_chain_padding_bits_untouched():
    """The chain's TMA stores and reduce-adds write only the M x N block: -0.0 in the gap
    columns (ldc > N) and around C keeps its bits."""
    M, N, K, ldc = 1000, 1100, 700, 1108
    rng = np.random.default_rng(53)
    A, B = inputs.normal_pair(rng, M, N, K)
    guard = 1024
    c_buf = torch.full((guard + M * ldc + guard,), -0.0, dtype=torch.float32, device="cuda")
    c_base = c_buf.data_ptr() + guard * 4
    dA, dB = dev16(A), dev16(B)
    st = tct.gemm_f16_f32_ex(dA.data_ptr(), dB.data_ptr(), c_base, M, N, K, K, N, ldc,
                             torch.cuda.current_stream().cuda_stream, stream_k=3)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    bits = c_buf.view(torch.int32).cpu().numpy()
    neg0 = np.int32(-2 ** 31)
    assert np.all(bits[:guard] == neg0) and np.all(bits[guard + M * ldc:] == neg0)
    body = bits[guard:guard + M * ldc].reshape(M, ldc)
    assert np.all(body[:, N:] == neg0)
    assert within_tol(body[:, :N].view(np.float32), oracle.gemm_f32(A, B), K)


def test_stream_k_and_whole_tiles_agree_on_integers():
    rng = np.random.default_rng(43)
    A, B = inputs.integer_pair(rng, 2048, 2304, 3000)
    whole = gpu_gemm(A, B, stream_k=1)
    split = gpu_gemm(A, B, stream_k=2)
    assert bit_exact(whole, split) and bit_exact(split, oracle.gemm_f32(A, B))


# ---- full-size workloads: every element -----------------------------------------------

def check_whole(A, B, C_dev, integer=False):
    """Every element of C against the oracle, computed in blocks of rows so that host memory
    stays bounded (about 64 MiB of FP32 per block): the tolerance for N(0,1) inputs, bit for
    bit for integer inputs."""
    M, K = A.shape
    N = B.shape[1]
    step = max(1, (64 << 20) // (4 * max(1, N)))
    for r0 in range(0, M, step):
        n = min(step, M - r0)
        want = oracle.gemm_rows_f32(A, B, r0, n)
        got = C_dev[r0:r0 + n].cpu().numpy()
        if integer:
            assert bit_exact(got, want), f"rows {r0}..{r0 + n - 1} differ"
        else:
            assert within_tol(got, want, K), f"rows {r0}..{r0 + n - 1}: worst {worst_ratio(got, want, K):.3g}"


def test_square_4096_seed2_whole():
    (M, N, K), A, B = inputs.workload("square4096")[0]
    C = tct.matmul(dev16(A), dev16(B))
    torch.cuda.synchronize()
    check_whole(A, B, C)


def test_wave_sweep_seed3_whole():
    for (M, N, K), A, B in inputs.workload("wave_sweep"):
        C = tct.matmul(dev16(A), dev16(B))
        torch.cuda.synchronize()
        check_whole(A, B, C)
        del C


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_large_seed4_whole(idx):
    (M, N, K), A, B = inputs.workload(f"large:{idx}")[idx]
    C = tct.matmul(dev16(A), dev16(B))
    torch.cuda.synchronize()
    check_whole(A, B, C)


@pytest.mark.parametrize("n,seed", [(4096, 2), (8192, 4)])
def test_square_integer_bit_exact_whole(n, seed):
    """Integer inputs in [-4, 4] at the headline sizes: every partial sum is an integer below
    16 n <= 2^17 < 2^24, so the FP32 result is unique and compared bit for bit."""
    A, B = inputs.integer_pair(np.random.default_rng(seed), n, n, n)
    C = tct.matmul(dev16(A), dev16(B))
    torch.cuda.synchronize()
    check_whole(A, B, C, integer=True)


# ---- C that TMA cannot write ------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,off,pad", [(1793, 1793, 1793, 0, 0), (300, 201, 150, 1, 2), (129, 65, 700, 3, 0),
                                           (1000, 1100, 2000, 1, 1), (17, 4097, 31, 2, 5), (2048, 4097, 256, 1, 0)])
def test_unaligned_c_guard_zones(M, N, K, off, pad):
    """C whose rows do not start on 16-byte boundaries or end inside a 16-byte unit (a unit's
    last tile staged as whole rows and bulk-copied, its other tiles by per-lane stores): the
    oracle's result in the M x N block, bit for bit on integer inputs, and NaN guard zones
    before, after and between the rows untouched."""
    rng = np.random.default_rng(61)
    A, B = inputs.normal_pair(rng, M, N, K)
    ldc = N + pad
    guard = 4096
    c_buf = torch.full((guard + off + M * ldc + guard,), float("nan"), dtype=torch.float32, device="cuda")
    c_base = c_buf.data_ptr() + (guard + off) * 4
    dA, dB = dev16(A), dev16(B)
    st = tct.gemm_f16_f32(dA.data_ptr(), dB.data_ptr(), c_base, M, N, K, K, N, ldc,
                          torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    host = c_buf.cpu().numpy()
    assert np.all(np.isnan(host[:guard + off])) and np.all(np.isnan(host[guard + off + M * ldc:]))
    body = host[guard + off:guard + off + M * ldc].reshape(M, ldc)
    assert np.all(np.isnan(body[:, N:]))
    assert within_tol(body[:, :N], oracle.gemm_f32(A, B), K)
    Ai, Bi = inputs.integer_pair(rng, M, N, K)
    dAi, dBi = dev16(Ai), dev16(Bi)  # kept alive until the call has run
    st = tct.gemm_f16_f32(dAi.data_ptr(), dBi.data_ptr(), c_base, M, N, K, K, N, ldc,
                          torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    body = c_buf.cpu().numpy()[guard + off:guard + off + M * ldc].reshape(M, ldc)
    assert bit_exact(body[:, :N], oracle.gemm_f32(Ai, Bi))
