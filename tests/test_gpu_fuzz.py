"""Seeded random problems through the C ABI, each checked against the oracle.

Every case draws, from its own seed: a shape (log-uniform sizes, occasionally K = 0), the
operand type and storage (gemm_f32acc's four layouts, FP16 or BF16), padded leading
dimensions and element offsets of the bases (so some operands are repacked and some C
matrices are stored without 16-byte vectors), and planner options (tile width, CTA pairs,
grid caps, GROUP_M, forced or forbidden split tails, stream-K where a plan for it exists).  A quarter of the GEMM cases use
integer inputs and must match bit for bit; the rest must meet the parity tolerance.  Every
case also checks that nothing outside the M x N block of C was written.  The epilogue cases
add random alpha, beta, bias and output types (gemm_ex); the softmax cases draw row lengths
from 1 to 300000 columns with padded, offset and in-place rows.
"""
import numpy as np
import pytest

import oracle
import tensor_core_tiled_gb300 as tct
from tensor_core_tiled_gb300 import inputs
from tests.parity import bit_exact, within_tol

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
TYPES = {"f32": (oracle.F32, tct.GEMM_DTYPE_F32), "f16": (oracle.F16, tct.GEMM_DTYPE_F16),
         "bf16": (oracle.BF16, tct.GEMM_DTYPE_BF16)}


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK


def _logu(rng, lo, hi):
    return int(np.exp(rng.uniform(np.log(lo), np.log(hi + 1)))) if hi > lo else lo


def _strided_device(x16, pad, offset, torch_dtype):
    """A device copy of the 2-D 16-bit array x16 with rows padded by `pad` elements, starting
    `offset` elements into its buffer; returns (buffer, pointer, leading dimension)."""
    rows, cols = x16.shape
    ld = cols + pad
    buf = torch.zeros(offset + max(rows * ld, 1) + 8, dtype=torch.int16, device="cuda")
    if rows and cols:
        view = buf[offset:offset + rows * ld].view(rows, ld)
        view[:, :cols] = torch.from_numpy(np.ascontiguousarray(x16).view(np.int16)).cuda()
    return buf.view(torch_dtype), buf.data_ptr() + 2 * offset, max(ld, 1)


def _draw_gemm(seed):
    rng = np.random.default_rng(seed)
    while True:
        M, N = _logu(rng, 1, 2048), _logu(rng, 1, 2048)
        K = 0 if rng.random() < 0.05 else _logu(rng, 1, 2048)
        if M * N * max(K, 1) <= 1 << 31:
            break
    case = dict(M=M, N=N, K=K, dt=str(rng.choice(["f16", "bf16"])), ta=bool(rng.random() < 0.4),
                tb=bool(rng.random() < 0.4), integer=bool(rng.random() < 0.25),
                pad_a=int(rng.choice([0, 0, 0, 1, 3, 8])), pad_b=int(rng.choice([0, 0, 0, 2, 5, 8])),
                off_a=int(rng.choice([0, 0, 0, 1, 8])), off_b=int(rng.choice([0, 0, 0, 3, 8])),
                pad_c=int(rng.choice([0, 0, 1, 4])), off_c=int(rng.choice([0, 0, 0, 1, 4])))
    opts = {}
    if rng.random() < 0.5:
        opts["stream_k"] = int(rng.choice([1, 2, 3]))
    if rng.random() < 0.3:
        opts["cta_group"] = int(rng.choice([1, 2]))
    if rng.random() < 0.3:
        opts["tile_n"] = int(rng.choice([128, 192, 256]))
    if rng.random() < 0.3:
        opts["max_ctas"] = int(rng.integers(2, 153))
    if rng.random() < 0.3:
        opts["group_m"] = int(rng.integers(1, 17))
    if opts.get("tile_n") == 192 and opts.get("cta_group") == 1:
        opts["tile_n"] = 256  # 192-column tiles: CTA pairs only
    if opts.get("stream_k") == 3:
        # stream-K adds pieces into C by TMA reduce-add: give it a C that TMA can write (rows of
        # whole 16-byte units on a 16-byte grid), so that most of these cases run it
        case["N"] = -(-N // 4) * 4
        case["pad_c"] = case["pad_c"] // 4 * 4
        case["off_c"] = case["off_c"] // 4 * 4
    case["opts"] = opts
    return rng, case


def _call(fn, opts):
    """fn(**opts); stream-K asked for (stream_k 3) is rejected with GEMM_ERR_INVALID_ARG where no
    stream-K plan exists (C not TMA-writable, an epilogue other than the plain FP32 one, too
    few k-blocks): then the call is repeated with the planner's own choice."""
    st = fn(**opts)
    if st == tct.GEMM_ERR_INVALID_ARG and opts.get("stream_k") == 3:
        st = fn(**{k: v for k, v in opts.items() if k != "stream_k"})
    return st


def _operands(rng, c):
    M, N, K, dt = c["M"], c["N"], c["K"], c["dt"]
    return inputs.pair_ex(rng, M, N, K, dtype=dt, integer=c["integer"], trans_a=c["ta"], trans_b=c["tb"])


def _device_operands(A, B, c):
    tdt = torch.float16 if c["dt"] == "f16" else torch.bfloat16
    bufA, pA, lda = _strided_device(A, c["pad_a"], c["off_a"], tdt)
    bufB, pB, ldb = _strided_device(B, c["pad_b"], c["off_b"], tdt)
    if c["K"] == 0:  # an empty operand still needs a legal leading dimension
        lda = max(lda, c["M"] if c["ta"] else 0, 1)
        ldb = max(ldb, 0 if c["tb"] else c["N"], 1)
    return (bufA, bufB), pA, lda, pB, ldb


@pytest.mark.parametrize("seed", range(1000, 1160))
def test_gemm_fuzz(seed):
    rng, c = _draw_gemm(seed)
    M, N, K = c["M"], c["N"], c["K"]
    A, B = _operands(rng, c)
    keep, pA, lda, pB, ldb = _device_operands(A, B, c)
    ldc = N + c["pad_c"]
    C = torch.full((c["off_c"] + M * ldc + 8,), float("nan"), device="cuda")
    pC = C.data_ptr() + 4 * c["off_c"]
    st = _call(lambda **o: tct.gemm_f32acc(TYPES[c["dt"]][1], int(c["ta"]), int(c["tb"]), pA, pB, pC, M, N, K, lda,
                                           ldb, ldc, torch.cuda.current_stream().cuda_stream, **o), c["opts"])
    assert st == tct.GEMM_OK, c
    torch.cuda.synchronize()
    host = C.cpu().numpy()
    block = host[c["off_c"]:c["off_c"] + M * ldc].reshape(M, ldc)
    got = block[:, :N]
    assert np.isnan(host[:c["off_c"]]).all() and np.isnan(host[c["off_c"] + M * ldc:]).all(), c
    assert np.isnan(block[:, N:]).all(), c
    if K == 0:
        assert np.all(got == 0), c
        return
    R = oracle.gemm_ex_f32(A, B, dtype=TYPES[c["dt"]][0], trans_a=c["ta"], trans_b=c["tb"])
    if c["integer"]:
        assert bit_exact(got, R), c
    else:
        assert within_tol(got, R, K), c


@pytest.mark.parametrize("seed", range(2000, 2040))
def test_gemm_ex_fuzz(seed):
    rng, c = _draw_gemm(seed)
    M, N, K = c["M"], c["N"], max(c["K"], 1)
    c["K"] = K
    ct = str(rng.choice(["f32", "f16", "bf16"]))
    alpha = float(rng.choice([1.0, 0.5, -2.0]))
    beta = float(rng.choice([0.0, 1.0, -0.75]))
    bt = str(rng.choice(["f32", "f16", "bf16"])) if rng.random() < 0.5 else None
    A, B = _operands(rng, c)
    keep, pA, lda, pB, ldb = _device_operands(A, B, c)
    if ct == "f32":
        Cin = rng.standard_normal((M, N)).astype(np.float32)
        dC = torch.from_numpy(Cin).cuda()
    else:
        Cin = (rng.standard_normal((M, N)).astype(np.float16).view(np.uint16) if ct == "f16"
               else inputs.to_bf16_bits(rng.standard_normal((M, N))))
        dC = torch.from_numpy(Cin.view(np.int16)).cuda()
    bias = None
    if bt:
        b = rng.standard_normal(N)
        bias = (b.astype(np.float32) if bt == "f32" else b.astype(np.float16).view(np.uint16) if bt == "f16"
                else inputs.to_bf16_bits(b))
        dbias = torch.from_numpy(bias.view(np.int32 if bt == "f32" else np.int16)).cuda()
    st = _call(lambda **o: tct.gemm_ex(TYPES[c["dt"]][1], int(c["ta"]), int(c["tb"]), pA, pB, dC.data_ptr(),
                                       TYPES[ct][1], M, N, K, lda, ldb, N, alpha=alpha, beta=beta,
                                       bias=dbias.data_ptr() if bt else 0, bias_type=TYPES[bt or "f32"][1],
                                       stream=torch.cuda.current_stream().cuda_stream, **o), c["opts"])
    assert st == tct.GEMM_OK, c
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    want = oracle.gemm_epilogue(A, B, dtype=TYPES[c["dt"]][0], trans_a=c["ta"], trans_b=c["tb"], alpha=alpha,
                                beta=beta, Cin=Cin, cin_type=TYPES[ct][0], bias=bias, bias_type=TYPES[bt or "f32"][0],
                                out_type=TYPES[ct][0])

    def as_f64(x):
        if ct == "f32":
            return x.astype(np.float64)
        tdt = torch.float16 if ct == "f16" else torch.bfloat16
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(tdt).double().numpy()

    S = np.abs(oracle.gemm_ex_f32(A, B, dtype=TYPES[c["dt"]][0], trans_a=c["ta"], trans_b=c["tb"]))
    ulp = {"f32": 0.0, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}[ct]
    g, w = as_f64(got), as_f64(want)
    tol = abs(alpha) * 1e-3 * np.sqrt(K) * np.maximum(1.0, S) + 2 * ulp * np.abs(w) + 1e-30
    assert np.all(np.abs(g - w) <= tol) and np.all(np.isfinite(g)), (c, ct, alpha, beta, bt)


@pytest.mark.parametrize("seed", range(3000, 3100))
def test_softmax_fuzz(seed):
    rng = np.random.default_rng(seed)
    N = _logu(rng, 1, 300000)
    M = max(1, min(_logu(rng, 1, 3000), (4 << 20) // N))
    pad = int(rng.choice([0, 0, 0, 1, 3, 4]))
    off = int(rng.choice([0, 0, 0, 1, 2, 4]))
    inplace = bool(rng.random() < 0.25)
    ld = N + pad
    X = inputs.normal_f32(rng, M, N) * np.float32(rng.choice([1.0, 1.0, 10.0]))
    X = X.astype(np.float32)
    if rng.random() < 0.2:  # special values in a few rows
        X[rng.integers(0, M)] = -np.inf
        X[rng.integers(0, M), rng.integers(0, N)] = np.inf
    buf = torch.full((off + M * ld + 8,), -3.0, device="cuda")
    view = buf[off:off + M * ld].view(M, ld)
    view[:, :N] = torch.from_numpy(X).cuda()
    ybuf = buf if inplace else torch.full_like(buf, -3.0)
    px = buf.data_ptr() + 4 * off
    py = ybuf.data_ptr() + 4 * off
    st = tct.softmax_rows_f32(px, py, M, N, ld, ld, torch.cuda.current_stream().cuda_stream)
    assert st == tct.GEMM_OK
    torch.cuda.synchronize()
    host = ybuf.cpu().numpy()
    block = host[off:off + M * ld].reshape(M, ld)
    y = block[:, :N]
    if pad:
        assert np.all(block[:, N:] == -3.0)
    assert np.all(host[:off] == -3.0) and np.all(host[off + M * ld:] == -3.0)
    ref = oracle.softmax_rows_f32(X)
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    valid = ~np.isnan(ref).any(axis=1)
    with np.errstate(invalid="ignore"):
        d = X.astype(np.float64) - X.max(axis=1, keepdims=True).astype(np.float64)
    ad = np.where(np.isfinite(d), np.abs(d), 0)
    staged = off % 4 == 0 and ld % 4 == 0
    n = 64 + (np.ceil(N / 4096) if staged else np.ceil(N / 256))
    tol = U * (32 + 3 * ad + 6 * ad.max(axis=1, keepdims=True) + 7 * n) * ref + 1e-37
    err = np.abs(y.astype(np.float64) - ref.astype(np.float64))
    assert not (~(err <= tol) & valid[:, None]).any(), (M, N, ld, off, inplace)
