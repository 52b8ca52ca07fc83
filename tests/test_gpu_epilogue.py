"""GPU parity of the epilogue (gemm_ex through the C ABI): C = alpha * op(A) op(B) + beta * C
+ bias, C in FP32, FP16 or BF16, against the oracle's epilogue."""
import numpy as np
import pytest

import oracle
import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TYPES = {"f32": (oracle.F32, tct.GEMM_DTYPE_F32), "f16": (oracle.F16, tct.GEMM_DTYPE_F16),
         "bf16": (oracle.BF16, tct.GEMM_DTYPE_BF16)}


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK


def _as_float(x, t):
    if t == "f32":
        return np.asarray(x, np.float64)
    tt = torch.float16 if t == "f16" else torch.bfloat16
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(tt).double().numpy()


def _typed_random(rng, shape, t, integer=False):
    v = rng.integers(-40, 40, size=shape).astype(np.float64) if integer else rng.standard_normal(shape)
    if t == "f32":
        return v.astype(np.float32)
    if t == "f16":
        return v.astype(np.float16).view(np.uint16)
    return inputs.to_bf16_bits(v)


def _dev(x, t):
    if t == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    tt = torch.float16 if t == "f16" else torch.bfloat16
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(tt)


def run_gpu(A, B, ab, ta, tb, M, N, K, ct, alpha, beta, Cin, bias, bt, **opts):
    dA = _dev(A, ab)
    dB = _dev(B, ab)
    dC = _dev(Cin, ct) if Cin is not None else _dev(_typed_random(np.random.default_rng(0), (M, N), ct), ct)
    dbias = _dev(bias, bt) if bias is not None else None
    st = tct.gemm_ex(TYPES[ab][1], int(ta), int(tb), dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), TYPES[ct][1], M, N,
                     K, A.shape[1], B.shape[1], N, alpha=alpha, beta=beta,
                     bias=dbias.data_ptr() if dbias is not None else 0, bias_type=TYPES[bt][1],
                     stream=torch.cuda.current_stream().cuda_stream, **opts)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    out = dC.cpu()
    return out.numpy() if ct == "f32" else out.view(torch.int16).numpy().view(np.uint16)


def run_ref(A, B, ab, ta, tb, ct, alpha, beta, Cin, bias, bt):
    return oracle.gemm_epilogue(A, B, dtype=TYPES[ab][0], trans_a=ta, trans_b=tb, alpha=alpha, beta=beta, Cin=Cin,
                                cin_type=TYPES[ct][0], bias=bias, bias_type=TYPES[bt][0], out_type=TYPES[ct][0])


def close(got, want, ct, K, alpha, S_scale):
    g, w = _as_float(got, ct), _as_float(want, ct)
    ulp = {"f32": 0.0, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}[ct]
    tol = abs(alpha) * 1e-3 * np.sqrt(K) * np.maximum(1.0, S_scale) + 2 * ulp * np.abs(w) + 1e-30
    return bool(np.all(np.abs(g - w) <= tol) and np.all(np.isfinite(g)))


CASES = [
    # (ab, ta, tb, ct, alpha, beta, bias_type or None)
    ("f16", False, False, "f32", 1.0, 0.0, "f32"),
    ("f16", False, False, "f32", 0.5, -1.25, None),
    ("f16", False, False, "f16", 1.0, 0.0, None),
    ("f16", False, False, "bf16", 2.0, 1.0, "bf16"),
    ("bf16", True, False, "bf16", -1.0, 0.5, "f16"),
    ("bf16", False, True, "f16", 0.25, 0.0, "f32"),
    ("f16", True, True, "f32", 3.0, 2.0, "f16"),
]


@pytest.mark.parametrize("ab,ta,tb,ct,alpha,beta,bt", CASES)
def test_epilogue_random(ab, ta, tb, ct, alpha, beta, bt):
    rng = np.random.default_rng(71)
    for (M, N, K) in [(300, 200, 150), (129, 65, 33), (777, 1500, 515), (17, 4097, 31)]:
        A, B = inputs.pair_ex(rng, M, N, K, dtype=ab, trans_a=ta, trans_b=tb)
        Cin = _typed_random(rng, (M, N), ct)
        bias = _typed_random(rng, (N,), bt) if bt else None
        got = run_gpu(A, B, ab, ta, tb, M, N, K, ct, alpha, beta, Cin, bias, bt or "f32")
        want = run_ref(A, B, ab, ta, tb, ct, alpha, beta, Cin, bias, bt or "f32")
        S = np.abs(oracle.gemm_ex_f32(A, B, dtype=TYPES[ab][0], trans_a=ta, trans_b=tb))
        assert close(got, want, ct, K, alpha, S), (M, N, K)


@pytest.mark.parametrize("ct", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("opts", [{}, dict(stream_k=2, cta_group=2, tile_n=256), dict(cta_group=1, tile_n=128)])
def test_epilogue_integer_bit_exact(ct, opts):
    """Integer operands, C and bias with integer alpha and beta: every FP32 intermediate is
    exact, so the stored value is the exact result rounded once to C's type -- the same bits
    as the oracle, split tiles included (their owner applies the epilogue once)."""
    rng = np.random.default_rng(72)
    M, N, K = 700, 904, 300  # N % 8 == 0: C of every type goes out by TMA stores
    A, B = inputs.pair_ex(rng, M, N, K, dtype="f16", integer=True)
    Cin = _typed_random(rng, (M, N), ct, integer=True)
    bias = _typed_random(rng, (N,), "f16", integer=True)
    got = run_gpu(A, B, "f16", False, False, M, N, K, ct, 3.0, -2.0, Cin, bias, "f16", **opts)
    want = run_ref(A, B, "f16", False, False, ct, 3.0, -2.0, Cin, bias, "f16")
    assert np.array_equal(got, want)


def _gemm_ex_at(A, B, M, N, K, ct, alpha, beta, Cin, bias, bt, offset, ldc, **opts):
    """gemm_ex with C stored at `offset` elements into its buffer with row pitch ldc; returns
    C's M x N block and the buffer's other elements, as raw bits."""
    esz = 4 if ct == "f32" else 2
    buf = torch.full((offset + M * ldc + 64,), -1, dtype=torch.int32 if ct == "f32" else torch.int16, device="cuda")
    body = buf[offset:offset + M * ldc].view(M, ldc)
    src = torch.from_numpy(np.ascontiguousarray(Cin).view(np.int32 if ct == "f32" else np.int16)).cuda()
    body[:, :N] = src
    dA, dB = _dev(A, "f16"), _dev(B, "f16")
    dbias = _dev(bias, bt) if bias is not None else None
    st = tct.gemm_ex(tct.GEMM_DTYPE_F16, 0, 0, dA.data_ptr(), dB.data_ptr(), buf.data_ptr() + esz * offset,
                     TYPES[ct][1], M, N, K, K, N, ldc, alpha=alpha, beta=beta,
                     bias=dbias.data_ptr() if dbias is not None else 0, bias_type=TYPES[bt][1],
                     stream=torch.cuda.current_stream().cuda_stream, **opts)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    rest = np.concatenate([host[:offset], host[offset:offset + M * ldc].reshape(M, ldc)[:, N:].ravel(),
                           host[offset + M * ldc:]])
    return host[offset:offset + M * ldc].reshape(M, ldc)[:, :N].copy(), rest


@pytest.mark.parametrize("ct", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("alpha,beta,bt", [(1.0, 0.0, None), (1.0, 1.0, None), (0.5, 0.0, "bf16"),
                                           (-1.5, 0.75, "f32"), (2.0, -1.0, "f16")])
@pytest.mark.parametrize("opts", [{}, dict(stream_k=2)])
def test_tma_and_lane_store_paths_agree(ct, alpha, beta, bt, opts):
    """The same problem with C where TMA can write it (16-byte aligned base and pitch, rows of
    whole 16-byte units: the tile goes out through swizzled staging and TMA stores, C read by
    TMA when beta != 0) and one element off that alignment (per-lane stores): the same bits,
    since both paths apply the same operations; nothing outside the M x N block changes."""
    rng = np.random.default_rng(75)
    M, N, K = 333, 520, 200
    A, B = inputs.pair_ex(rng, M, N, K, dtype="f16")
    Cin = _typed_random(rng, (M, N), ct)
    bias = _typed_random(rng, (N,), bt) if bt else None
    ldc = N + 8
    tma, rest_t = _gemm_ex_at(A, B, M, N, K, ct, alpha, beta, Cin, bias, bt or "f32", 0, ldc, **opts)
    lane, rest_l = _gemm_ex_at(A, B, M, N, K, ct, alpha, beta, Cin, bias, bt or "f32", 1, ldc, **opts)
    assert np.all(rest_t == -1) and np.all(rest_l == -1)
    assert np.array_equal(tma, lane)
    want = run_ref(A, B, "f16", False, False, ct, alpha, beta, Cin, bias, bt or "f32")
    S = np.abs(oracle.gemm_ex_f32(A, B))
    got = tma if ct == "f32" else tma.view(np.uint16)
    assert close(got.view(np.float32) if ct == "f32" else got, want, ct, K, alpha, S)


@pytest.mark.parametrize("ct,N", [("f16", 1500), ("bf16", 1500), ("f16", 1504), ("f32", 1502)])
def test_padding_untouched_when_rows_end_inside_16_bytes(ct, N):
    """Aligned base and pitch: rows of whole 16-byte units go through TMA stores, others
    through per-lane stores; the columns between N and ldc keep their bits either way."""
    rng = np.random.default_rng(76)
    M, K = 300, 96
    A, B = inputs.pair_ex(rng, M, N, K, dtype="f16", integer=True)
    Cin = _typed_random(rng, (M, N), ct, integer=True)
    bias = _typed_random(rng, (N,), "f16", integer=True)
    ldc = N + (8 - N % 8) + 8
    got, rest = _gemm_ex_at(A, B, M, N, K, ct, 2.0, -1.0, Cin, bias, "f16", 0, ldc)
    assert np.all(rest == -1)
    want = run_ref(A, B, "f16", False, False, ct, 2.0, -1.0, Cin, bias, "f16")
    assert np.array_equal(got.view(np.uint32 if ct == "f32" else np.uint16), np.asarray(want).view(np.uint32 if ct == "f32" else np.uint16))


def test_beta_zero_never_reads_c_and_k_zero_is_the_empty_sum():
    rng = np.random.default_rng(73)
    M, N, K = 200, 300, 64
    A, B = inputs.pair_ex(rng, M, N, K, dtype="f16", integer=True)
    nan_c = np.full((M, N), np.nan, np.float32)
    got = run_gpu(A, B, "f16", False, False, M, N, K, "f32", 1.0, 0.0, nan_c, None, "f32")
    assert np.array_equal(got, oracle.gemm_ex_f32(A, B))
    # K == 0: C = beta * C + bias
    Cin = _typed_random(rng, (M, N), "f32", integer=True)
    bias = _typed_random(rng, (N,), "f32", integer=True)
    dC = torch.from_numpy(Cin.copy()).cuda()
    dbias = torch.from_numpy(bias).cuda()
    dA = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    dB = torch.empty((0, N), dtype=torch.float16, device="cuda")
    st = tct.gemm_ex(tct.GEMM_DTYPE_F16, 0, 0, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), tct.GEMM_DTYPE_F32, M, N,
                     0, 0, N, N, alpha=5.0, beta=-3.0, bias=dbias.data_ptr(), bias_type=tct.GEMM_DTYPE_F32,
                     stream=torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    assert np.array_equal(dC.cpu().numpy(), (-3.0 * Cin + bias[None, :]).astype(np.float32))


def test_unaligned_c_and_padded_ldc():
    rng = np.random.default_rng(74)
    M, N, K, pad = 130, 250, 100, 3
    A, B = inputs.pair_ex(rng, M, N, K, dtype="bf16")
    Cbuf = torch.full((M * (N + pad) + 1,), float("nan"), dtype=torch.float16, device="cuda")
    base = Cbuf.data_ptr() + 2  # 2-byte aligned only: scalar stores
    dA = _dev(A, "bf16")
    dB = _dev(B, "bf16")
    st = tct.gemm_ex(tct.GEMM_DTYPE_BF16, 0, 0, dA.data_ptr(), dB.data_ptr(), base, tct.GEMM_DTYPE_F16, M, N, K, K, N,
                     N + pad, alpha=1.0, beta=0.0, stream=torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    host = Cbuf.cpu().view(torch.int16).numpy().view(np.uint16)
    body = host[1:1 + M * (N + pad)].reshape(M, N + pad)
    assert np.all(np.isnan(host[:1].view(np.float16)))
    assert np.all(np.isnan(body[:, N:].view(np.float16)))
    want = run_ref(A, B, "bf16", False, False, "f16", 1.0, 0.0, None, None, "f32")
    S = np.abs(oracle.gemm_ex_f32(A, B, dtype=oracle.BF16))
    assert close(body[:, :N], want, "f16", K, 1.0, S)


def test_torch_helper():
    """The torch-facing helper (tct.gemm) gives the oracle's epilogue result."""
    rng = np.random.default_rng(75)
    M, N, K = 256, 384, 128
    A, B = inputs.pair_ex(rng, M, N, K, dtype="f16")
    dA, dB = _dev(A, "f16"), _dev(B, "f16")
    bias = rng.standard_normal(N).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    out = tct.gemm(dA, dB, _dev(C0, "f32"), alpha=2.0, beta=0.5, bias=_dev(bias, "f32"))
    torch.cuda.synchronize()
    want = run_ref(A, B, "f16", False, False, "f32", 2.0, 0.5, C0, bias, "f32")
    S = np.abs(oracle.gemm_ex_f32(A, B, dtype=oracle.F16))
    assert close(out.cpu().numpy(), want, "f32", K, 2.0, S)
    # A given as a transposed view, BF16 output: the stored layout is read in place
    out16 = tct.gemm(dA.t().contiguous().t(), dB, out_dtype=torch.bfloat16)
    assert out16.dtype == torch.bfloat16
    got16 = out16.cpu().view(torch.int16).numpy().view(np.uint16)
    want16 = run_ref(A, B, "f16", False, False, "bf16", 1.0, 0.0, None, None, "f32")
    assert close(got16, want16, "bf16", K, 1.0, S)


@pytest.mark.parametrize("ct", ["f32", "f16", "bf16"])
def test_beta_with_unaligned_c(ct):
    """beta != 0 on a C that TMA cannot write (one element off a 16-byte boundary, a row pitch
    that is not a 16-byte multiple): the per-lane epilogue reads C's current values and stores
    the result; gap columns and the elements around C keep their bits."""
    rng = np.random.default_rng(77)
    M, N, K, pad = 301, 203, 160, 3
    A, B = inputs.pair_ex(rng, M, N, K, dtype="f16")
    Cin = _typed_random(rng, (M, N + pad), ct)
    bias = _typed_random(rng, (N,), "f32")
    esz = 4 if ct == "f32" else 2
    off = 1  # one element past an aligned address
    total = off + M * (N + pad) + 8
    if ct == "f32":
        buf = torch.full((total,), float("nan"), dtype=torch.float32, device="cuda")
        buf[off:off + M * (N + pad)] = torch.from_numpy(np.ascontiguousarray(Cin).reshape(-1)).cuda()
    else:
        tt = torch.float16 if ct == "f16" else torch.bfloat16
        buf = torch.full((total,), float("nan"), dtype=tt, device="cuda")
        buf[off:off + M * (N + pad)] = torch.from_numpy(np.ascontiguousarray(Cin).view(np.int16).reshape(-1)).cuda().view(tt)
    before = buf.clone()
    dA, dB = _dev(A, "f16"), _dev(B, "f16")
    dbias = _dev(bias, "f32")
    st = tct.gemm_ex(TYPES["f16"][1], 0, 0, dA.data_ptr(), dB.data_ptr(), buf.data_ptr() + off * esz, TYPES[ct][1],
                     M, N, K, K, N, N + pad, alpha=0.75, beta=-1.5, bias=dbias.data_ptr(), bias_type=TYPES["f32"][1],
                     stream=torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    if ct == "f32":
        got_all = buf.cpu().numpy()
        was = before.cpu().numpy()
    else:
        got_all = buf.cpu().view(torch.int16).numpy().view(np.uint16)
        was = before.cpu().view(torch.int16).numpy().view(np.uint16)
    body = got_all[off:off + M * (N + pad)].reshape(M, N + pad)
    assert np.array_equal(got_all[:off].view(np.uint8), was[:off].view(np.uint8))
    assert np.array_equal(got_all[off + M * (N + pad):].view(np.uint8), was[off + M * (N + pad):].view(np.uint8))
    assert np.array_equal(body[:, N:].view(np.uint8), np.ascontiguousarray(Cin)[:, N:].view(np.uint8))
    want = run_ref(A, B, "f16", False, False, ct, 0.75, -1.5, np.ascontiguousarray(Cin[:, :N]), bias, "f32")
    S = np.abs(oracle.gemm_ex_f32(A, B, dtype=oracle.F16))
    assert close(body[:, :N], want, ct, K, 0.75, S + 1.5 * np.abs(_as_float(Cin[:, :N], ct)) + 4)
