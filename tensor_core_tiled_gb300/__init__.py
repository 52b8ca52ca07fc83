"""Python binding of the GB300 FP16 -> FP32 tiled tensor-core GEMM (``libtensor_core_tiled.so``).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  The names mirror the C ABI in ``include/tensor_core_tiled.h``.  Importing this
package does not load the library; the first call does, and raises ``GemmError`` if the
library has not been built (``python -m tensor_core_tiled_gb300.build``) -- there is no
fallback implementation.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtensor_core_tiled.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED_DEVICE = 2
GEMM_ERR_CUDA = 3
GEMM_ERR_DEVICE_TIMEOUT = 4

GEMM_DTYPE_F16, GEMM_DTYPE_BF16, GEMM_DTYPE_F32 = 0, 1, 2
GEMM_OP_N, GEMM_OP_T = 0, 1

# Every function the header declares (checked by the test-suite against the .so).
EXPORTED = (
    "gemm_f16_f32",
    "gemm_f16_f32_ex",
    "gemm_f16_f32_noalloc",
    "gemm_f32acc",
    "gemm_ex",
    "softmax_rows_f32",
    "gemm_f16_f32_host",
    "softmax_rows_f32_host",
    "gemm_f16_f32_plan",
    "gemm_f16_f32_work_item",
    "gemm_tile_coord",
    "gemm_wave_model",
    "gemm_f16_f32_get_error",
    "gemm_tensor_rate_probe",
    "gemm_status_string",
    "gemm_version",
)


class GemmError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})" if what else status_string(status))


class GemmOptions(ctypes.Structure):
    _fields_ = [("group_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("timeout_ms", ctypes.c_int32), ("cta_group", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("fault_inject", ctypes.c_int32)]


class GemmPlan(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("group_m", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("tiles", ctypes.c_int64), ("waves", ctypes.c_int64), ("wave_efficiency", ctypes.c_double),
                ("smem_bytes", ctypes.c_int32), ("pack_a", ctypes.c_int32), ("pack_b", ctypes.c_int32),
                ("cta_group", ctypes.c_int32), ("units", ctypes.c_int32), ("stream_k_tiles", ctypes.c_int32),
                ("effective_waves", ctypes.c_double), ("split_kb", ctypes.c_int32),
                ("split_parts_per_unit", ctypes.c_int32), ("split_form", ctypes.c_int32),
                ("sk_units", ctypes.c_int32)]


class GemmEpilogue(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("bias_type", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class GemmWork(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int32), ("kb0", ctypes.c_int32), ("kb1", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("part", ctypes.c_int32)]


WORK_STORE, WORK_FIXUP, WORK_PARTIAL, WORK_CHAIN = 0, 1, 2, 3

_lib = None


def load():
    """Load the shared library (once).  Raises GemmError if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise GemmError(GEMM_ERR_CUDA, f"{LIB_PATH} is not built; run tensor_core_tiled_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.gemm_f16_f32.restype = ctypes.c_int
    lib.gemm_f16_f32.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
    lib.gemm_f16_f32_noalloc.restype = ctypes.c_int
    lib.gemm_f16_f32_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
    lib.gemm_f32acc.restype = ctypes.c_int
    lib.gemm_f32acc.argtypes = [i32, i32, i32, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp,
                                ctypes.POINTER(GemmOptions)]
    lib.gemm_ex.restype = ctypes.c_int
    lib.gemm_ex.argtypes = [i32, i32, i32, vp, vp, vp, i32, i64, i64, i64, i64, i64, i64,
                            ctypes.POINTER(GemmEpilogue), vp, ctypes.POINTER(GemmOptions)]
    lib.softmax_rows_f32.restype = ctypes.c_int
    lib.softmax_rows_f32.argtypes = [vp, vp, i64, i64, i64, i64, vp]
    lib.softmax_rows_f32_host.restype = ctypes.c_int
    lib.softmax_rows_f32_host.argtypes = [vp, vp, i64, i64, i64, i64, vp]
    lib.gemm_f16_f32_host.restype = ctypes.c_int
    lib.gemm_f16_f32_host.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
    lib.gemm_f16_f32_ex.restype = ctypes.c_int
    lib.gemm_f16_f32_ex.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, ctypes.POINTER(GemmOptions)]
    lib.gemm_f16_f32_plan.restype = ctypes.c_int
    lib.gemm_f16_f32_plan.argtypes = [i64, i64, i64, i64, i64, i32, ctypes.POINTER(GemmOptions),
                                      ctypes.POINTER(GemmPlan)]
    lib.gemm_f16_f32_work_item.restype = ctypes.c_int
    lib.gemm_f16_f32_work_item.argtypes = [i64, i64, i64, i32, ctypes.POINTER(GemmOptions), i32, i32,
                                           ctypes.POINTER(GemmWork)]
    lib.gemm_tile_coord.restype = ctypes.c_int
    lib.gemm_tile_coord.argtypes = [i64, i64, i64, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.gemm_wave_model.restype = ctypes.c_int
    lib.gemm_wave_model.argtypes = [i64, i64, i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                    ctypes.POINTER(ctypes.c_double)]
    lib.gemm_f16_f32_get_error.restype = ctypes.c_int
    lib.gemm_f16_f32_get_error.argtypes = []
    lib.gemm_tensor_rate_probe.restype = ctypes.c_int
    lib.gemm_tensor_rate_probe.argtypes = [i32, vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_double)]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_version.restype = ctypes.c_char_p
    lib.gemm_version.argtypes = []
    _lib = lib
    return lib


def status_string(status):
    try:
        return load().gemm_status_string(int(status)).decode()
    except GemmError:
        return f"status {status}"


def version():
    return load().gemm_version().decode()


def _options(group_m=0, tile_n=0, stages=0, max_ctas=0, timeout_ms=0, cta_group=0, stream_k=0, fault_inject=0):
    o = GemmOptions()
    o.group_m, o.tile_n, o.stages, o.max_ctas, o.timeout_ms = group_m, tile_n, stages, max_ctas, timeout_ms
    o.cta_group, o.stream_k, o.fault_inject = cta_group, stream_k, fault_inject
    return o


def gemm_f16_f32(A, B, C, M, N, K, lda, ldb, ldc, stream=0):
    """Raw C-ABI call with integer device pointers; returns the status code."""
    return load().gemm_f16_f32(A, B, C, M, N, K, lda, ldb, ldc, stream or None)


def gemm_f16_f32_noalloc(A, B, C, M, N, K, lda, ldb, ldc, stream=0):
    """Raw C-ABI call of the allocation-free entry point (library-owned scratch array)."""
    return load().gemm_f16_f32_noalloc(A, B, C, M, N, K, lda, ldb, ldc, stream or None)


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def gemm_f16_f32_ex(A, B, C, M, N, K, lda, ldb, ldc, stream=0, **options):
    """Raw C-ABI call with tuning options (group_m, tile_n, stages, max_ctas, timeout_ms, cta_group,
    stream_k)."""
    opt = _options(**options)
    return load().gemm_f16_f32_ex(A, B, C, M, N, K, lda, ldb, ldc, stream or None, ctypes.byref(opt))


def gemm_f32acc(ab_type, op_a, op_b, A, B, C, M, N, K, lda, ldb, ldc, stream=0, **options):
    """Raw C-ABI call for FP16/BF16 operands stored as given (op = GEMM_OP_N or GEMM_OP_T)."""
    opt = _options(**options)
    return load().gemm_f32acc(ab_type, op_a, op_b, A, B, C, M, N, K, lda, ldb, ldc, stream or None,
                              ctypes.byref(opt))


def gemm_ex(ab_type, op_a, op_b, A, B, C, c_type, M, N, K, lda, ldb, ldc, alpha=1.0, beta=0.0, bias=0,
            bias_type=GEMM_DTYPE_F32, stream=0, **options):
    """Raw C-ABI call with the epilogue C = alpha * op(A) op(B) + beta * C + bias (pointers as ints)."""
    epi = GemmEpilogue()
    epi.alpha, epi.beta, epi.bias, epi.bias_type, epi.reserved = alpha, beta, bias or None, bias_type, 0
    opt = _options(**options)
    return load().gemm_ex(ab_type, op_a, op_b, A, B, C, c_type, M, N, K, lda, ldb, ldc, ctypes.byref(epi),
                          stream or None, ctypes.byref(opt))


def gemm_f16_f32_plan(M, N, K, lda=None, ldb=None, num_sms=0, **options):
    """The launch plan (tile shape, stages, grid, waves) as a dict."""
    opt = _options(**options)
    pl = GemmPlan()
    st = load().gemm_f16_f32_plan(M, N, K, K if lda is None else lda, N if ldb is None else ldb, num_sms,
                                  ctypes.byref(opt), ctypes.byref(pl))
    if st:
        raise GemmError(st, "gemm_f16_f32_plan")
    return {name: getattr(pl, name) for name, _ in GemmPlan._fields_}


def gemm_f16_f32_work_item(M, N, K, num_sms, unit, idx, **options):
    """Work item idx of a persistent unit as a dict, or None when the unit has no more."""
    opt = _options(**options)
    w = GemmWork()
    st = load().gemm_f16_f32_work_item(M, N, K, num_sms, ctypes.byref(opt), unit, idx, ctypes.byref(w))
    if st == GEMM_ERR_INVALID_ARG:
        return None
    if st:
        raise GemmError(st, "gemm_f16_f32_work_item")
    return {name: getattr(w, name) for name, _ in GemmWork._fields_}


def gemm_tile_coord(t, num_m, num_n, group_m):
    r, c = ctypes.c_int64(), ctypes.c_int64()
    st = load().gemm_tile_coord(t, num_m, num_n, group_m, ctypes.byref(r), ctypes.byref(c))
    if st:
        raise GemmError(st, "gemm_tile_coord")
    return r.value, c.value


def gemm_wave_model(M, N, tile_m, tile_n, slots):
    t, w, u = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_double()
    st = load().gemm_wave_model(M, N, tile_m, tile_n, slots, ctypes.byref(t), ctypes.byref(w), ctypes.byref(u))
    if st:
        raise GemmError(st, "gemm_wave_model")
    return t.value, w.value, u.value


def gemm_f16_f32_get_error():
    return load().gemm_f16_f32_get_error()


def gemm_tensor_rate_probe(n_mma=1 << 16, stream=0):
    """Measured dense FP16 tensor FLOP per SM per clock: (median, min, max) over the SMs."""
    med, lo, hi = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    st = load().gemm_tensor_rate_probe(n_mma, stream or None, ctypes.byref(med), ctypes.byref(lo), ctypes.byref(hi))
    if st:
        raise GemmError(st, "gemm_tensor_rate_probe")
    return med.value, lo.value, hi.value


def _current_stream_ptr(device):
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _operand(t, rows, cols, name):
    """(op, ld) of a 2-D tensor holding a rows x cols operand: row-major (unit column stride)
    is op N with ld = row stride; column-major (unit row stride) is op T, i.e. the transpose
    stored row-major, with ld = column stride."""
    r_stride, c_stride = t.stride()
    if cols <= 1 or c_stride == 1:
        return GEMM_OP_N, max(r_stride if rows > 1 else cols, cols, 1)
    if rows <= 1 or r_stride == 1:
        return GEMM_OP_T, max(c_stride if cols > 1 else rows, rows, 1)
    raise ValueError(f"{name} must be row-major or column-major (one unit stride)")


def matmul(A, B, C=None, stream=None, **options):
    """C = A @ B for torch CUDA tensors: A (M x K) and B (K x N) both float16 or both bfloat16,
    each row-major or column-major (e.g. a transposed view), C (M x N) float32 row-major
    (allocated if None).  Runs on ``stream`` (a torch.cuda.Stream) or the current stream;
    raises GemmError on a non-zero status."""
    import torch
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    if A.dtype != B.dtype or A.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("A and B must both be float16 or both bfloat16")
    if not (A.is_cuda and B.is_cuda) or A.device != B.device:
        raise ValueError("A and B must be CUDA tensors on one device")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if C.dtype != torch.float32 or tuple(C.shape) != (M, N) or C.device != A.device:
        raise ValueError("C must be a float32 M x N tensor on A's device")
    if C.numel() and N > 1 and C.stride(1) != 1:
        raise ValueError("C must be row-major (unit column stride)")
    op_a, lda = _operand(A, M, K, "A")
    op_b, ldb = _operand(B, K, N, "B")
    ldc = C.stride(0) if M > 1 else max(N, 1)
    s = stream.cuda_stream if stream is not None else _current_stream_ptr(A.device)
    dt = GEMM_DTYPE_BF16 if A.dtype == torch.bfloat16 else GEMM_DTYPE_F16
    with torch.cuda.device(A.device):
        if dt == GEMM_DTYPE_F16 and op_a == GEMM_OP_N and op_b == GEMM_OP_N:
            if options:
                st = gemm_f16_f32_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, ldc, s, **options)
            else:
                st = gemm_f16_f32(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, ldc, s)
        else:
            st = gemm_f32acc(dt, op_a, op_b, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, ldc, s,
                             **options)
    if st:
        raise GemmError(st, "gemm_f32acc" if (dt or op_a or op_b) else "gemm_f16_f32")
    return C


def gemm(A, B, C=None, alpha=1.0, beta=0.0, bias=None, out_dtype=None, stream=None, **options):
    """C = alpha * A @ B + beta * C + bias for torch CUDA tensors (A, B float16 or bfloat16,
    row- or column-major; bias None or a length-N float32/float16/bfloat16 vector; C row-major
    float32/float16/bfloat16, allocated as out_dtype (default float32) when None)."""
    import torch
    types = {torch.float16: GEMM_DTYPE_F16, torch.bfloat16: GEMM_DTYPE_BF16, torch.float32: GEMM_DTYPE_F32}
    if A.dim() != 2 or B.dim() != 2 or A.dtype != B.dtype or A.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("A and B must be 2-D, both float16 or both bfloat16")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    if C.dtype not in types or tuple(C.shape) != (M, N) or (C.numel() and N > 1 and C.stride(1) != 1):
        raise ValueError("C must be a row-major M x N float32/float16/bfloat16 tensor")
    if bias is not None and (bias.dim() != 1 or bias.numel() != N or bias.dtype not in types or
                             (N > 1 and bias.stride(0) != 1)):
        raise ValueError("bias must be a contiguous length-N float32/float16/bfloat16 vector")
    op_a, lda = _operand(A, M, K, "A")
    op_b, ldb = _operand(B, K, N, "B")
    ldc = C.stride(0) if M > 1 else max(N, 1)
    s = stream.cuda_stream if stream is not None else _current_stream_ptr(A.device)
    with torch.cuda.device(A.device):
        st = gemm_ex(types[A.dtype], op_a, op_b, A.data_ptr(), B.data_ptr(), C.data_ptr(), types[C.dtype], M, N, K,
                     lda, ldb, ldc, alpha, beta, bias.data_ptr() if bias is not None else 0,
                     types[bias.dtype] if bias is not None else GEMM_DTYPE_F32, s, **options)
    if st:
        raise GemmError(st, "gemm_ex")
    return C


def softmax_rows_f32(X, Y, M, N, ldx, ldy, stream=0):
    """Raw C-ABI call of the row softmax (pointers as ints); returns the status code."""
    return load().softmax_rows_f32(X, Y, M, N, ldx, ldy, stream or None)


def softmax(X, out=None, stream=None):
    """Row softmax of a 2-D float32 CUDA tensor (row-major; out may be X for in place)."""
    import torch
    if X.dim() != 2 or X.dtype != torch.float32 or not X.is_cuda:
        raise TypeError("X must be a 2-D float32 CUDA tensor")
    M, N = X.shape
    if N > 1 and X.stride(1) != 1:
        raise ValueError("X must be row-major")
    if out is None:
        out = torch.empty_like(X)
    if out.shape != X.shape or out.dtype != torch.float32 or (N > 1 and out.stride(1) != 1):
        raise ValueError("out must be a row-major float32 tensor of X's shape")
    s = stream.cuda_stream if stream is not None else _current_stream_ptr(X.device)
    with torch.cuda.device(X.device):
        st = softmax_rows_f32(X.data_ptr(), out.data_ptr(), M, N, X.stride(0) if M > 1 else max(N, 1),
                              out.stride(0) if M > 1 else max(N, 1), s)
    if st:
        raise GemmError(st, "softmax_rows_f32")
    return out


def gemm_f16_f32_host(A, B, C, M, N, K, lda, ldb, ldc, stream=0):
    """Raw C-ABI call of the host-buffer GEMM (host pointers as ints); returns the status."""
    return load().gemm_f16_f32_host(A, B, C, M, N, K, lda, ldb, ldc, stream or None)


def softmax_rows_f32_host(X, Y, M, N, ldx, ldy, stream=0):
    """Raw C-ABI call of the host-buffer row softmax (host pointers as ints); returns the status."""
    return load().softmax_rows_f32_host(X, Y, M, N, ldx, ldy, stream or None)
