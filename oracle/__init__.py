"""CPU oracle for the FP16 -> FP32 blocked GEMM (ctypes binding of ``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package; the product library never does, and the
two share no code.  See ``oracle.c`` for what is computed and which passages of the
lecture pages each part follows.

Arrays are numpy ``float16`` (or their ``uint16`` bit views); a leading dimension
larger than the row length is expressed by passing a wider array and the logical
(M, N, K) separately.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force=False):
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (OpenMP, IEEE arithmetic)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    subprocess.check_call(cmd)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64 = ctypes.c_int64
    vp = ctypes.c_void_p
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_f16.restype = None
    lib.oracle_decode_f16.argtypes = [vp, vp, i64]
    for name in ("oracle_gemm_f64", "oracle_gemm_f32"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64]
    for name in ("oracle_gemm_rows_f64", "oracle_gemm_rows_f32"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64]
    lib.oracle_gemm_elems.restype = ctypes.c_int
    lib.oracle_gemm_elems.argtypes = [vp, vp, i64, i64, i64, i64, i64, vp, vp, i64, vp, vp]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_gemm_ex_rows_f32.restype = ctypes.c_int
    lib.oracle_gemm_ex_rows_f32.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, i64, i64, i64, i64,
                                            i64, i64, i64, i64]
    lib.oracle_gemm_ex_elems.restype = ctypes.c_int
    lib.oracle_gemm_ex_elems.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, i64, i64, i64,
                                         vp, vp, i64, vp, vp]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16_n.restype = None
    lib.oracle_f32_to_f16_n.argtypes = [vp, vp, i64]
    lib.oracle_f32_to_bf16_n.restype = None
    lib.oracle_f32_to_bf16_n.argtypes = [vp, vp, i64]
    lib.oracle_gemm_epilogue.restype = ctypes.c_int
    lib.oracle_gemm_epilogue.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, i64, i64, i64, i64, i64,
                                         ctypes.c_double, ctypes.c_double, vp, ctypes.c_int, i64, vp, ctypes.c_int,
                                         vp, ctypes.c_int, i64]
    lib.oracle_softmax_rows_f32.restype = ctypes.c_int
    lib.oracle_softmax_rows_f32.argtypes = [vp, vp, i64, i64, i64, i64]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _bits(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("oracle operands are FP16 (or their uint16 bit patterns)")
    return x


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def f16_to_f64(bits):
    """Decode one FP16 bit pattern (int) with the oracle's own decoder."""
    return _load().oracle_f16_to_f64(int(bits) & 0xFFFF)


def decode_f16(x):
    """Decode an array of FP16 values (or bit patterns) to float64 with the oracle's decoder."""
    b = _bits(x)
    out = np.empty(b.shape, np.float64)
    _load().oracle_decode_f16(_ptr(b), _ptr(out), b.size)
    return out


def _shape(A, B, M, N, K):
    if A.ndim != 2 or B.ndim != 2:
        raise ValueError("A and B must be 2-D")
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[1] if N is None else N
    if M > A.shape[0] or K > A.shape[1] or K > B.shape[0] or N > B.shape[1]:
        raise ValueError("logical shape exceeds the arrays")
    return M, N, K


def gemm_f64(A, B, M=None, N=None, K=None):
    """FP64 sums R[i,j] = sum_k A[i,k]*B[k,j] in increasing k (no final rounding)."""
    A, B = _bits(A), _bits(B)
    M, N, K = _shape(A, B, M, N, K)
    R = np.zeros((M, max(N, 1)), np.float64)
    rc = _load().oracle_gemm_f64(_ptr(A), _ptr(B), _ptr(R), M, N, K, A.shape[1], B.shape[1], R.shape[1])
    if rc:
        raise ValueError(f"oracle_gemm_f64 rejected the arguments (rc={rc})")
    return R[:, :N]


def gemm_f32(A, B, M=None, N=None, K=None):
    """The oracle proper: FP64 sums rounded once to FP32 (round to nearest even)."""
    A, B = _bits(A), _bits(B)
    M, N, K = _shape(A, B, M, N, K)
    C = np.zeros((M, max(N, 1)), np.float32)
    rc = _load().oracle_gemm_f32(_ptr(A), _ptr(B), _ptr(C), M, N, K, A.shape[1], B.shape[1], C.shape[1])
    if rc:
        raise ValueError(f"oracle_gemm_f32 rejected the arguments (rc={rc})")
    return C[:, :N]


def gemm_rows_f32(A, B, row0, nrows, M=None, N=None, K=None):
    """Rows [row0, row0+nrows) of :func:`gemm_f32` (for bounded CPU samples of big products)."""
    A, B = _bits(A), _bits(B)
    M, N, K = _shape(A, B, M, N, K)
    C = np.zeros((nrows, max(N, 1)), np.float32)
    rc = _load().oracle_gemm_rows_f32(_ptr(A), _ptr(B), _ptr(C), M, N, K, A.shape[1], B.shape[1],
                                      C.shape[1], row0, nrows)
    if rc:
        raise ValueError(f"oracle_gemm_rows_f32 rejected the arguments (rc={rc})")
    return C[:, :N]


def gemm_elems(A, B, rows, cols, M=None, N=None, K=None):
    """Selected outputs: returns (fp64 sums, fp32 results) at positions (rows[t], cols[t])."""
    A, B = _bits(A), _bits(B)
    M, N, K = _shape(A, B, M, N, K)
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    n = rows.size
    o64 = np.zeros(n, np.float64)
    o32 = np.zeros(n, np.float32)
    rc = _load().oracle_gemm_elems(_ptr(A), _ptr(B), M, N, K, A.shape[1], B.shape[1], _ptr(rows),
                                   _ptr(cols), n, _ptr(o64), _ptr(o32))
    if rc:
        raise ValueError(f"oracle_gemm_elems rejected the arguments (rc={rc})")
    return o64, o32


def num_threads():
    return _load().oracle_num_threads()


def set_num_threads(n):
    _load().oracle_set_num_threads(int(n))


# ---- generalised operands: FP16 or BF16 storage, either operand stored transposed ---------

F16, BF16 = 0, 1


def bf16_to_f64(bits):
    """Decode one BF16 bit pattern (int) with the oracle's own decoder."""
    return _load().oracle_bf16_to_f64(int(bits) & 0xFFFF)


def _bits16(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError("oracle operands are 16-bit patterns (uint16) or float16")


def gemm_ex_f32(A, B, dtype=F16, trans_a=False, trans_b=False, M=None, N=None, K=None, row0=0, nrows=None):
    """C = op(A) . op(B) rounded once to FP32.  A, B are 16-bit patterns of `dtype` (F16 or
    BF16) stored row-major: A is M x K (trans_a False) or K x M (True), B is K x N (trans_b
    False) or N x K (True); wider arrays give leading dimensions.  Rows [row0, row0+nrows)."""
    A, B = _bits16(A), _bits16(B)
    Mi = A.shape[1] if trans_a else A.shape[0]
    Ki = A.shape[0] if trans_a else A.shape[1]
    Ni = B.shape[0] if trans_b else B.shape[1]
    M = Mi if M is None else M
    K = Ki if K is None else K
    N = Ni if N is None else N
    nrows = M - row0 if nrows is None else nrows
    C = np.zeros((nrows, max(N, 1)), np.float32)
    rc = _load().oracle_gemm_ex_rows_f32(int(dtype), int(bool(trans_a)), int(bool(trans_b)), _ptr(A), _ptr(B),
                                         _ptr(C), M, N, K, A.shape[1], B.shape[1], C.shape[1], row0, nrows)
    if rc:
        raise ValueError(f"oracle_gemm_ex_rows_f32 rejected the arguments (rc={rc})")
    return C[:, :N]


def gemm_ex_elems(A, B, rows, cols, dtype=F16, trans_a=False, trans_b=False, M=None, N=None, K=None):
    """Selected outputs of op(A) . op(B): (fp64 sums, fp32 results)."""
    A, B = _bits16(A), _bits16(B)
    M = (A.shape[1] if trans_a else A.shape[0]) if M is None else M
    K = (A.shape[0] if trans_a else A.shape[1]) if K is None else K
    N = (B.shape[0] if trans_b else B.shape[1]) if N is None else N
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    o64 = np.zeros(rows.size, np.float64)
    o32 = np.zeros(rows.size, np.float32)
    rc = _load().oracle_gemm_ex_elems(int(dtype), int(bool(trans_a)), int(bool(trans_b)), _ptr(A), _ptr(B), M, N, K,
                                      A.shape[1], B.shape[1], _ptr(rows), _ptr(cols), rows.size, _ptr(o64), _ptr(o32))
    if rc:
        raise ValueError(f"oracle_gemm_ex_elems rejected the arguments (rc={rc})")
    return o64, o32


# ---- epilogue: D = round_out(alpha * S + beta * Cin + bias[j]) ------------------------------

F32 = 2


def f32_to_f16_bits(x):
    """binary16 bit pattern of a float32 value, the oracle's own rounding."""
    return _load().oracle_f32_to_f16(float(np.float32(x)))


def f32_to_bf16_bits(x):
    return _load().oracle_f32_to_bf16(float(np.float32(x)))


def _typed(x, t):
    """Contiguous array of the given oracle type code (F16/BF16 as uint16 bits, F32)."""
    x = np.ascontiguousarray(x)
    if t == F32:
        if x.dtype != np.float32:
            raise TypeError("expected float32")
        return x
    return _bits16(x)


def gemm_epilogue(A, B, dtype=F16, trans_a=False, trans_b=False, alpha=1.0, beta=0.0, Cin=None, cin_type=F32,
                  bias=None, bias_type=F32, out_type=F32):
    """D = round_out(alpha * op(A).op(B) + beta * Cin + bias[j]) -- see oracle.c.  Returns a
    float32 array (out F32) or uint16 bit patterns (out F16/BF16)."""
    A, B = _bits16(A), _bits16(B)
    M = A.shape[1] if trans_a else A.shape[0]
    K = A.shape[0] if trans_a else A.shape[1]
    N = B.shape[0] if trans_b else B.shape[1]
    D = np.zeros((M, max(N, 1)), np.float32 if out_type == F32 else np.uint16)
    cin = _typed(Cin, cin_type) if (beta != 0.0 and Cin is not None) else None
    bs = _typed(bias, bias_type) if bias is not None else None
    rc = _load().oracle_gemm_epilogue(int(dtype), int(bool(trans_a)), int(bool(trans_b)), _ptr(A), _ptr(B), M, N, K,
                                      A.shape[1], B.shape[1], float(alpha), float(beta), _ptr(cin), int(cin_type),
                                      cin.shape[1] if cin is not None else N, _ptr(bs), int(bias_type), _ptr(D),
                                      int(out_type), D.shape[1])
    if rc:
        raise ValueError(f"oracle_gemm_epilogue rejected the arguments (rc={rc})")
    return D[:, :N]


def f32_to_16bit_array(x, out_type):
    """Vectorised oracle rounding of float32 values to F16 or BF16 bit patterns."""
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    fn = _load().oracle_f32_to_f16_n if out_type == F16 else _load().oracle_f32_to_bf16_n
    fn(_ptr(x), _ptr(out), x.size)
    return out


# ---- row softmax ------------------------------------------------------------------------

def softmax_rows_f32(X):
    """Row softmax of a 2-D float32 array: FP64 arithmetic, one final round to FP32."""
    X = np.ascontiguousarray(X, np.float32)
    M, N = X.shape
    Y = np.zeros((M, max(N, 1)), np.float32)
    rc = _load().oracle_softmax_rows_f32(_ptr(X), _ptr(Y), M, N, N, Y.shape[1])
    if rc:
        raise ValueError(f"oracle_softmax_rows_f32 rejected the arguments (rc={rc})")
    return Y[:, :N]
