"""Pins for the oracle's epilogue D = round_out(alpha * S + beta * Cin + bias[j]).

  * FP32 -> FP16 rounding against numpy's conversion, FP32 -> BF16 against torch's, on
    millions of bit patterns including every float32 near binary16's binade edges and ties;
  * alpha = 1, beta = 0, no bias, FP32 out equals the pinned generalised oracle;
  * integer-valued operands, C and bias with integer alpha and beta: the exact int64 result
    of numpy, rounded by numpy/torch to the output type.
"""
import numpy as np
import pytest

import oracle
from tensor_core_tiled_gb300 import inputs

torch = pytest.importorskip("torch")


def _sample_f32(n, seed):
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    # concentrate half the sample on binary16's range and its subnormals
    fp16_range = (rng.integers(0x33000000, 0x47800000, n // 2, dtype=np.uint64).astype(np.uint32)
                  | (rng.integers(0, 2, n // 2, dtype=np.uint64).astype(np.uint32) << 31))
    # exact binary16 ties: a 1 bit just below binary16's last significand bit
    k = rng.integers(0, 2 ** 10, 4096, dtype=np.uint64).astype(np.uint32)
    e = rng.integers(103, 142, 4096, dtype=np.uint64).astype(np.uint32)
    ties = (e << 23) | (k << 13) | (1 << 12)
    return np.concatenate([u, fp16_range, ties]).view(np.float32)


def test_f32_to_f16_matches_numpy():
    x = _sample_f32(2_000_000, 1)
    mine = oracle.f32_to_16bit_array(x, oracle.F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all((mine[nan] & 0x7c00) == 0x7c00) and np.all(mine[nan] & 0x3ff)


def test_f32_to_bf16_matches_torch():
    x = _sample_f32(2_000_000, 2)
    mine = oracle.f32_to_16bit_array(x, oracle.BF16)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_identity_epilogue_equals_the_product(dtype):
    rng = np.random.default_rng(3)
    A, B = inputs.pair_ex(rng, 129, 65, 33, dtype="f16" if dtype == oracle.F16 else "bf16")
    assert np.array_equal(oracle.gemm_epilogue(A, B, dtype=dtype), oracle.gemm_ex_f32(A, B, dtype=dtype))


@pytest.mark.parametrize("out_type", [oracle.F32, oracle.F16, oracle.BF16])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True)])
def test_integer_epilogue_exact(out_type, ta, tb):
    rng = np.random.default_rng(4)
    M, N, K = 70, 90, 40
    A, B = inputs.pair_ex(rng, M, N, K, dtype="f16", integer=True, trans_a=ta, trans_b=tb)
    Cin = rng.integers(-50, 50, size=(M, N)).astype(np.float32)
    bias = rng.integers(-20, 20, size=N).astype(np.float32)
    Ai = A.astype(np.int64).T if ta else A.astype(np.int64)
    Bi = B.astype(np.int64).T if tb else B.astype(np.int64)
    exact = 3 * (Ai @ Bi) - 2 * Cin.astype(np.int64) + bias.astype(np.int64)[None, :]
    D = oracle.gemm_epilogue(A, B, trans_a=ta, trans_b=tb, alpha=3.0, beta=-2.0, Cin=Cin, cin_type=oracle.F32,
                             bias=bias, bias_type=oracle.F32, out_type=out_type)
    if out_type == oracle.F32:
        assert np.array_equal(D, exact.astype(np.float32))
    elif out_type == oracle.F16:
        assert np.array_equal(D, exact.astype(np.float32).astype(np.float16).view(np.uint16))
    else:
        ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(D, ref)


def test_beta_zero_ignores_cin_and_bias_types_decode():
    rng = np.random.default_rng(5)
    A, B = inputs.pair_ex(rng, 16, 24, 8, dtype="f16", integer=True)
    nan_c = np.full((16, 24), np.nan, np.float32)
    base = oracle.gemm_epilogue(A, B)
    assert np.array_equal(oracle.gemm_epilogue(A, B, beta=0.0, Cin=nan_c), base)
    bias16 = np.arange(24, dtype=np.float16)
    with_b = oracle.gemm_epilogue(A, B, bias=bias16, bias_type=oracle.F16)
    assert np.array_equal(with_b, base + np.arange(24, dtype=np.float32)[None, :])
