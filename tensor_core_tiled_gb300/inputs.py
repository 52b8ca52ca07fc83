"""Seeded synthetic inputs for the FP16 -> FP32 GEMM workloads.

This module draws random operands and nothing else: it holds none of the GEMM's
arithmetic, and both the CUDA path's tests/benchmark and the CPU oracle take their
inputs from it.  The recipe follows the lecture pages' own idiom
("04_tensor_cores.py" demos 1-2, "06_triton_style.py" demos 1 and 4): a numpy
``default_rng(seed)``, ``standard_normal`` drawn in float64 and rounded to FP16
(numpy rounds to nearest, ties to even), A (M x K) first, then B (K x N), from the same
generator; a list of shapes shares one generator in list order.

Integer-valued operands (for bit-exact checks) come from a fresh ``default_rng(seed)``
with ``integers(-4, 4, endpoint=True)``, i.e. uniform on -4..4, A then B per shape.
"""
import numpy as np

# Workload shapes, named by what they are.
SQUARE_256 = (256, 256, 256)
RAGGED_SHAPES = ((300, 200, 150), (129, 65, 33), (1, 1000, 64), (17, 4097, 31))
SQUARE_4096 = (4096, 4096, 4096)
WAVE_SWEEP_SIZES = (1792, 1793, 2048, 3072, 6144)
LARGE_SHAPES = ((8192, 8192, 8192), (16384, 16384, 4096), (128, 16384, 16384))

# Rows drawn per numpy call; drawing in chunks yields the same stream as one call
# and bounds the float64 temporary.
_CHUNK_ELEMS = 1 << 24


def normal_f16(rng, rows, cols):
    """A rows x cols FP16 matrix of N(0,1) draws, taken row-major from ``rng``."""
    out = np.empty((rows, cols), np.float16)
    if rows == 0 or cols == 0:
        return out
    step = max(1, _CHUNK_ELEMS // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = rng.standard_normal((r1 - r0, cols)).astype(np.float16)
    return out


def normal_pair(rng, M, N, K):
    """(A, B) with A = M x K then B = K x N drawn from ``rng`` in that order."""
    A = normal_f16(rng, M, K)
    B = normal_f16(rng, K, N)
    return A, B


def integer_pair(rng, M, N, K, lo=-4, hi=4):
    """(A, B) of integer values in [lo, hi] stored as FP16 (exact), A then B."""
    A = rng.integers(lo, hi, size=(M, K), endpoint=True).astype(np.float16)
    B = rng.integers(lo, hi, size=(K, N), endpoint=True).astype(np.float16)
    return A, B


def square(seed, n):
    """Square N(0,1) operands of side n from ``default_rng(seed)``."""
    return normal_pair(np.random.default_rng(seed), n, n, n)


def shape_set(seed, shapes, integer=False):
    """Yield ((M, N, K), A, B) for each shape, one generator shared in list order."""
    rng = np.random.default_rng(seed)
    for (M, N, K) in shapes:
        if integer:
            A, B = integer_pair(rng, M, N, K)
        else:
            A, B = normal_pair(rng, M, N, K)
        yield (M, N, K), A, B


def workload(name):
    """Operands of a named workload: returns a list of ((M, N, K), A, B).

    Names: ``square256`` (seed 0), ``ragged`` and ``ragged_int`` (seed 1),
    ``square4096`` (seed 2), ``wave_sweep`` (seed 3), ``large`` (seed 4, shapes in
    order), or ``large:<i>`` for the first i+1 shapes of ``large`` (the stream is
    sequential, so shape i needs the draws of the shapes before it).
    """
    if name == "square256":
        return list(shape_set(0, [SQUARE_256]))
    if name == "ragged":
        return list(shape_set(1, RAGGED_SHAPES))
    if name == "ragged_int":
        return list(shape_set(1, RAGGED_SHAPES, integer=True))
    if name == "square4096":
        return list(shape_set(2, [SQUARE_4096]))
    if name == "wave_sweep":
        return list(shape_set(3, [(n, n, n) for n in WAVE_SWEEP_SIZES]))
    if name == "large":
        return list(shape_set(4, LARGE_SHAPES))
    if name.startswith("large:"):
        i = int(name.split(":")[1])
        return list(shape_set(4, LARGE_SHAPES[: i + 1]))
    raise KeyError(name)


# ---- BF16 operands and transposed storage ------------------------------------------------

def to_bf16_bits(x):
    """float array -> BF16 bit patterns (uint16): rounded to FP32, then to BF16, each to
    nearest with ties to even (torch's conversion)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def normal_bf16(rng, rows, cols):
    """A rows x cols BF16 matrix (bit patterns) of N(0,1) draws, row-major from ``rng``."""
    out = np.empty((rows, cols), np.uint16)
    if rows == 0 or cols == 0:
        return out
    step = max(1, _CHUNK_ELEMS // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = to_bf16_bits(rng.standard_normal((r1 - r0, cols)))
    return out


def pair_ex(rng, M, N, K, dtype="f16", integer=False, trans_a=False, trans_b=False):
    """(A, B) for C = op(A) . op(B): the logical A (M x K) is drawn first, then the logical B
    (K x N), exactly as in normal_pair / integer_pair; then each is stored transposed if asked
    (A as K x M, B as N x K).  FP16 arrays are float16, BF16 arrays are uint16 bit patterns."""
    if integer:
        A = rng.integers(-4, 4, size=(M, K), endpoint=True)
        B = rng.integers(-4, 4, size=(K, N), endpoint=True)
        if dtype == "f16":
            A, B = A.astype(np.float16), B.astype(np.float16)
        else:
            A, B = to_bf16_bits(A), to_bf16_bits(B)
    elif dtype == "f16":
        A, B = normal_pair(rng, M, N, K)
    else:
        A = normal_bf16(rng, M, K)
        B = normal_bf16(rng, K, N)
    if trans_a:
        A = np.ascontiguousarray(A.T)
    if trans_b:
        B = np.ascontiguousarray(B.T)
    return A, B


# ---- row softmax inputs -------------------------------------------------------------------

# The page's softmax workload ("06_triton_style.py" demo 3): a 4096 x 1024 FP32 matrix of
# N(0,1) draws; the larger case is the same recipe at 32768 x 4096 (512 MiB, above L2).
SOFTMAX_PAGE = (4096, 1024)
SOFTMAX_LARGE = (32768, 4096)


def normal_f32(rng, rows, cols):
    """A rows x cols FP32 matrix of N(0,1) draws (float64 rounded to nearest), row-major."""
    out = np.empty((rows, cols), np.float32)
    if rows == 0 or cols == 0:
        return out
    step = max(1, _CHUNK_ELEMS // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = rng.standard_normal((r1 - r0, cols)).astype(np.float32)
    return out
