"""Pins for the oracle's generalised operands: BF16 storage and transposed A and/or B.

  * the BF16 decoder against torch's own bfloat16 -> float64 conversion, all 65536 patterns;
  * exact Python-integer sums on 16x8x16 BF16 tiles (values taken from torch, not from the
    oracle), rounded to FP32 by integer arithmetic;
  * FP16 with both operands as stored agrees bit for bit with the pinned FP16 oracle;
  * each transposed storage gives the bits of the untransposed definition (numpy transposes);
  * integer-valued inputs in every layout and both types against numpy's int64 matmul.
"""
import itertools

import numpy as np
import pytest

import oracle
from tensor_core_tiled_gb300 import inputs
from tests import exact

torch = pytest.importorskip("torch")


def test_bf16_decoder_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = np.array([oracle.bf16_to_f64(b) for b in bits.tolist()])
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def _bf16_values(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _exact_units(vals, unit_exp):
    out = np.empty(vals.shape, dtype=object)
    for idx, v in np.ndenumerate(vals):
        f = exact.Fraction(float(v)) * (exact.Fraction(2) ** -unit_exp)
        assert f.denominator == 1
        out[idx] = int(f)
    return out


def test_bf16_brute_force_tiles_exact():
    rng = np.random.default_rng(2)
    for _ in range(30):
        A = inputs.normal_bf16(rng, 16, 16)
        B = inputs.normal_bf16(rng, 16, 8)
        # N(0,1) BF16 values are multiples of 2^-133 at worst; use 2^-40 units (exact here)
        a = _exact_units(_bf16_values(A), -40)
        b = _exact_units(_bf16_values(B), -40)
        want = np.empty((16, 8), np.float32)
        for i in range(16):
            for j in range(8):
                want[i, j] = exact.round_to_f32(sum(a[i, k] * b[k, j] for k in range(16)), unit_exp=-80)
        got = oracle.gemm_ex_f32(A, B, dtype=oracle.BF16)
        assert np.array_equal(got, want)


def test_f16_as_stored_equals_the_pinned_fp16_oracle():
    for (M, N, K), A, B in inputs.workload("ragged"):
        assert np.array_equal(oracle.gemm_ex_f32(A, B, dtype=oracle.F16), oracle.gemm_f32(A, B))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
def test_transposed_storage_gives_the_same_product(dtype, ta, tb):
    rng = np.random.default_rng(7)
    M, N, K = 37, 45, 29
    A, B = inputs.pair_ex(rng, M, N, K, dtype=dtype)
    d = oracle.F16 if dtype == "f16" else oracle.BF16
    ref = oracle.gemm_ex_f32(A, B, dtype=d)
    As = np.ascontiguousarray(A.T) if ta else A
    Bs = np.ascontiguousarray(B.T) if tb else B
    got = oracle.gemm_ex_f32(As, Bs, dtype=d, trans_a=ta, trans_b=tb)
    assert np.array_equal(got, ref)
    if M != K:
        # a planted mistake: reading a transposed A as if it were not transposed fails
        with pytest.raises(Exception):
            bad = oracle.gemm_ex_f32(As, Bs, dtype=d, trans_a=not ta, trans_b=tb)
            assert np.array_equal(bad, ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("ta,tb", list(itertools.product([False, True], repeat=2)))
def test_integer_inputs_every_layout_bit_exact(dtype, ta, tb):
    rng = np.random.default_rng(1)
    for (M, N, K) in [(300, 200, 150), (17, 4097, 31), (64, 64, 64)]:
        A, B = inputs.pair_ex(rng, M, N, K, dtype=dtype, integer=True, trans_a=ta, trans_b=tb)
        vals = (lambda x: _bf16_values(x)) if dtype == "bf16" else (lambda x: x.astype(np.float64))
        Ai = vals(A).astype(np.int64)
        Bi = vals(B).astype(np.int64)
        Ai = Ai.T if ta else Ai
        Bi = Bi.T if tb else Bi
        want = (Ai @ Bi).astype(np.float32)
        d = oracle.F16 if dtype == "f16" else oracle.BF16
        assert np.array_equal(oracle.gemm_ex_f32(A, B, dtype=d, trans_a=ta, trans_b=tb), want)
        rows = np.array([0, M - 1, M // 2])
        cols = np.array([N - 1, 0, N // 3])
        _, o32 = oracle.gemm_ex_elems(A, B, rows, cols, dtype=d, trans_a=ta, trans_b=tb)
        assert np.array_equal(o32, want[rows, cols])


def test_bf16_rounding_of_inputs():
    # the recipe rounds float64 -> float32 -> bf16, each to nearest even (torch's conversion)
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40])
    got = _bf16_values(inputs.to_bf16_bits(x))
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 + 2 ** -6 and got[3] == -2.5
