/*
 * oracle.c -- CPU oracle for C[MxN] = A[MxK] . B[KxN], FP16 inputs, FP32 output.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through the seeded input arrays.
 *
 * What it computes (the plain definition of the product the lecture pages
 * centre on):
 *
 *     R[i][j] = (float) sum_{k=0}^{K-1} (double) A[i*lda + k] * (double) B[k*ldb + j]
 *
 *   - "04_tensor_cores.py", demo 2 (block tensor-core GEMM) and "06_triton_style.py",
 *     demos 1 and 4: every kernel on the pages is checked against the product of the
 *     FP16 inputs widened to float64, which is exactly this sum.
 *   - "04_tensor_cores.py", demo 1 observation 3: an FP16 x FP16 product has at most
 *     11 + 11 significand bits, so each product below is exact in FP64; the only
 *     rounding is in the FP64 running sum and in the single final cast to FP32.
 *   - Summation order: increasing k, one running FP64 accumulator per output,
 *     i-k-j loop order (rows in parallel), no blocking, no reordering.
 *   - The final FP64 -> FP32 conversion is a plain C cast, i.e. IEEE round to
 *     nearest, ties to even (the pages are silent; this is the plainest reading).
 *   - K == 0 gives the empty sum 0 for every output; M == 0 or N == 0 writes nothing.
 *
 * FP16 values are decoded from their bit patterns by oracle_f16_to_f64(), written
 * from the IEEE 754 binary16 definition (1 sign bit, 5 exponent bits with bias 15,
 * 10 fraction bits; exponent 0 = zero/subnormal, exponent 31 = inf/NaN).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, exact for every one of the 65536 patterns. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        /* zero or subnormal: 0.frac x 2^-14 */
        mag = ldexp((double)frac, -24);
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        /* normal: 1.frac x 2^(expo-15) */
        mag = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -mag : mag;
}

void oracle_decode_f16(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f16_to_f64(h[i]);
}

/* Decoding through a table built from oracle_f16_to_f64 keeps the triple loop plain
 * while avoiding a ldexp per operand read. */
static double g_f16_table[65536];
static int g_f16_table_ready = 0;

static const double *f16_table(void)
{
    if (!g_f16_table_ready) {
        for (int i = 0; i < 65536; ++i)
            g_f16_table[i] = oracle_f16_to_f64((uint16_t)i);
        g_f16_table_ready = 1;
    }
    return g_f16_table;
}

static int check_args(const void *A, const void *B, const void *C, int64_t M, int64_t N,
                      int64_t K, int64_t lda, int64_t ldb, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (lda < K || ldb < N || ldc < N) return 1;
    if (M > 0 && N > 0 && !C) return 1;
    if (M > 0 && K > 0 && !A) return 1;
    if (N > 0 && K > 0 && !B) return 1;
    return 0;
}

/*
 * Rows [row0, row0 + nrows) of the FP64 sums, written to R (leading dimension ldr).
 * This is the whole definition; the other entry points round or sample it.
 */
int oracle_gemm_rows_f64(const uint16_t *A, const uint16_t *B, double *R, int64_t M, int64_t N,
                         int64_t K, int64_t lda, int64_t ldb, int64_t ldr, int64_t row0,
                         int64_t nrows)
{
    if (check_args(A, B, R, M, N, K, lda, ldb, ldr)) return 1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > M) return 1;
    const double *T = f16_table();
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = row0; i < row0 + nrows; ++i) {
        double *r = R + (i - row0) * ldr;
        for (int64_t j = 0; j < N; ++j) r[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = T[A[i * lda + k]];
            const uint16_t *b = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) r[j] += a * T[b[j]];
        }
    }
    return 0;
}

int oracle_gemm_f64(const uint16_t *A, const uint16_t *B, double *R, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldr)
{
    return oracle_gemm_rows_f64(A, B, R, M, N, K, lda, ldb, ldr, 0, M);
}

/* Rows [row0, row0 + nrows) of the FP64 sums rounded once to FP32. */
int oracle_gemm_rows_f32(const uint16_t *A, const uint16_t *B, float *C, int64_t M, int64_t N,
                         int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t row0,
                         int64_t nrows)
{
    if (check_args(A, B, C, M, N, K, lda, ldb, ldc)) return 1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > M) return 1;
    const double *T = f16_table();
    int bad = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = row0; i < row0 + nrows; ++i) {
            if (!acc) continue;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = T[A[i * lda + k]];
                const uint16_t *b = B + k * ldb;
                for (int64_t j = 0; j < N; ++j) acc[j] += a * T[b[j]];
            }
            float *c = C + (i - row0) * ldc;
            for (int64_t j = 0; j < N; ++j) c[j] = (float)acc[j];
        }
        free(acc);
    }
    return bad ? 2 : 0;
}

int oracle_gemm_f32(const uint16_t *A, const uint16_t *B, float *C, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldc)
{
    return oracle_gemm_rows_f32(A, B, C, M, N, K, lda, ldb, ldc, 0, M);
}

/*
 * Selected outputs (rows[t], cols[t]) for t < n: the same FP64 sum in the same
 * order, for checking single elements of products too large to compute whole.
 * out64 (may be NULL) receives the FP64 sums, out32 (may be NULL) the FP32 casts.
 */
int oracle_gemm_elems(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, const int64_t *rows, const int64_t *cols,
                      int64_t n, double *out64, float *out32)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || n < 0) return 1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return 1;
    const double *T = f16_table();
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = rows[t], j = cols[t];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += T[A[i * lda + k]] * T[B[k * ldb + j]];
        if (out64) out64[t] = s;
        if (out32) out32[t] = (float)s;
    }
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Generalised operands (still the plain definition, one FP64 running sum per output):
 *
 *     R[i][j] = (float) sum_k  opA(i, k) * opB(k, j)
 *
 *   dtype 0: FP16 (binary16, decoded as above); dtype 1: BF16, whose 16 bits are the upper
 *   half of an IEEE binary32 value (1 sign, 8 exponent, 7 fraction bits), so its value is
 *   that binary32 value, exact in double.  A BF16 x BF16 product has at most 8 + 8
 *   significand bits, so it too is exact in FP64.
 *   trans_a 0: opA(i, k) = A[i*lda + k] (A stored M x K); 1: opA(i, k) = A[k*lda + i]
 *   (A stored K x M).  trans_b 0: opB(k, j) = B[k*ldb + j] (B stored K x N); 1:
 *   opB(k, j) = B[j*ldb + k] (B stored N x K).
 * --------------------------------------------------------------------------------- */
double oracle_bf16_to_f64(uint16_t h)
{
    union {
        uint32_t u;
        float f;
    } v;
    v.u = (uint32_t)h << 16;
    return (double)v.f;
}

static double g_bf16_table[65536];
static int g_bf16_table_ready = 0;

static const double *bf16_table(void)
{
    if (!g_bf16_table_ready) {
        for (int i = 0; i < 65536; ++i)
            g_bf16_table[i] = oracle_bf16_to_f64((uint16_t)i);
        g_bf16_table_ready = 1;
    }
    return g_bf16_table;
}

int oracle_gemm_ex_rows_f32(int dtype, int trans_a, int trans_b, const uint16_t *A, const uint16_t *B, float *C,
                            int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t row0,
                            int64_t nrows)
{
    if (dtype != 0 && dtype != 1) return 1;
    if (M < 0 || N < 0 || K < 0 || ldc < N) return 1;
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? K : N)) return 1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > M) return 1;
    if (M > 0 && N > 0 && (!C || (K > 0 && (!A || !B)))) return 1;
    const double *T = dtype ? bf16_table() : f16_table();
    int bad = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = row0; i < row0 + nrows; ++i) {
            if (!acc) continue;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = T[trans_a ? A[k * lda + i] : A[i * lda + k]];
                if (trans_b) {
                    for (int64_t j = 0; j < N; ++j) acc[j] += a * T[B[j * ldb + k]];
                } else {
                    const uint16_t *b = B + k * ldb;
                    for (int64_t j = 0; j < N; ++j) acc[j] += a * T[b[j]];
                }
            }
            float *c = C + (i - row0) * ldc;
            for (int64_t j = 0; j < N; ++j) c[j] = (float)acc[j];
        }
        free(acc);
    }
    return bad ? 2 : 0;
}

int oracle_gemm_ex_elems(int dtype, int trans_a, int trans_b, const uint16_t *A, const uint16_t *B, int64_t M,
                         int64_t N, int64_t K, int64_t lda, int64_t ldb, const int64_t *rows, const int64_t *cols,
                         int64_t n, double *out64, float *out32)
{
    if (dtype != 0 && dtype != 1) return 1;
    if (M < 0 || N < 0 || K < 0 || n < 0) return 1;
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? K : N)) return 1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return 1;
    const double *T = dtype ? bf16_table() : f16_table();
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += T[trans_a ? A[k * lda + i] : A[i * lda + k]] * T[trans_b ? B[j * ldb + k] : B[k * ldb + j]];
        if (out64) out64[t] = s;
        if (out32) out32[t] = (float)s;
    }
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Epilogue (the plain reading of a scaled, biased product written in a chosen type):
 *
 *     D[i][j] = round_out( alpha * S[i][j] + beta * Cin[i][j] + bias[j] )
 *
 *   S is the FP64 sum of oracle_gemm_ex_rows_f32 before its final rounding; the scaled sum,
 *   the FP64 values of Cin and bias (decoded from their types) are combined in FP64 and
 *   rounded once to FP32; a narrower output type is then produced from that FP32 value by
 *   round-to-nearest-even (FP16 through a C conversion of the FP32 value, which is exact
 *   to double and then rounded by the binary16 rule below; BF16 by rounding the FP32 bit
 *   pattern to its upper 16 bits).  beta == 0 does not read Cin; bias may be NULL.
 *   Types: 0 FP16, 1 BF16, 2 FP32.
 * --------------------------------------------------------------------------------- */
static double decode_any(const void *p, int type, int64_t idx)
{
    if (type == 2) return (double)((const float *)p)[idx];
    const uint16_t h = ((const uint16_t *)p)[idx];
    return type == 1 ? oracle_bf16_to_f64(h) : oracle_f16_to_f64(h);
}

/* binary16 of a float by round to nearest, ties to even (IEEE 754: 11-bit significands,
 * exponents -14..15, subnormals in steps of 2^-24, overflow to infinity).  The float is
 * m * 2^p exactly; its binary16 quantum at that magnitude is 2^qe with
 * qe = max(floor(log2|f|) - 10, -24); q = m * 2^(p - qe) rounded to an integer. */
uint16_t oracle_f32_to_f16(float f)
{
    union {
        float f;
        uint32_t u;
    } v;
    v.f = f;
    const uint16_t sign = (uint16_t)((v.u >> 16) & 0x8000u);
    const uint32_t ex = (v.u >> 23) & 0xffu, man = v.u & 0x7fffffu;
    if (ex == 0xffu) return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0u));
    if (ex == 0 && man == 0) return sign;
    const uint64_t m = ex ? (man | 0x800000u) : man;
    const int p = ex ? (int)ex - 150 : -149;
    const int bl = 64 - __builtin_clzll(m);
    const int e = p + bl - 1;
    int qe = e - 10 < -24 ? -24 : e - 10;
    uint64_t q;
    if (qe > p) {
        const int rs = qe - p;
        if (rs > 63) {
            q = 0;
        } else {
            q = m >> rs;
            const uint64_t rem = m & ((1ull << rs) - 1), half = 1ull << (rs - 1);
            if (rem > half || (rem == half && (q & 1))) ++q;
        }
    } else {
        q = m << (p - qe);
    }
    if (q == 2048) { /* rounded up into the next binade */
        q = 1024;
        ++qe;
    }
    if (q < 1024) return (uint16_t)(sign | q); /* subnormal, qe == -24 */
    const int field = qe + 25;
    if (field >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | ((uint32_t)field << 10) | (uint32_t)(q - 1024));
}

/* bfloat16 of a float: its upper 16 bits after round to nearest, ties to even on the lower
 * 16 bits (NaN stays NaN). */
uint16_t oracle_f32_to_bf16(float f)
{
    union {
        float f;
        uint32_t u;
    } v;
    v.f = f;
    if (((v.u >> 23) & 0xffu) == 0xffu) return (uint16_t)((v.u >> 16) | ((v.u & 0xffffu) ? 0x40u : 0u));
    const uint32_t lower = v.u & 0xffffu, upper = v.u >> 16;
    uint32_t r = upper;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) ++r;
    return (uint16_t)r;
}

void oracle_f32_to_f16_n(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(x[i]);
}

void oracle_f32_to_bf16_n(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(x[i]);
}

int oracle_gemm_epilogue(int ab_type, int trans_a, int trans_b, const uint16_t *A, const uint16_t *B, int64_t M,
                         int64_t N, int64_t K, int64_t lda, int64_t ldb, double alpha, double beta,
                         const void *Cin, int cin_type, int64_t ldcin, const void *bias, int bias_type, void *D,
                         int d_type, int64_t ldd)
{
    if (d_type < 0 || d_type > 2 || cin_type < 0 || cin_type > 2 || bias_type < 0 || bias_type > 2) return 1;
    if (M < 0 || N < 0 || ldd < N || (beta != 0.0 && (!Cin || ldcin < N))) return 1;
    if (M == 0 || N == 0) return 0;
    float *S = (float *)malloc((size_t)M * (size_t)N * sizeof(float));
    double *S64 = (double *)malloc((size_t)M * (size_t)N * sizeof(double));
    if (!S || !S64) {
        free(S);
        free(S64);
        return 2;
    }
    /* the FP64 sums, row by row, through the generalised definition's element routine */
    int64_t *rows = (int64_t *)malloc((size_t)N * sizeof(int64_t));
    int64_t *cols = (int64_t *)malloc((size_t)N * sizeof(int64_t));
    int rc = (!rows || !cols) ? 2 : 0;
    for (int64_t i = 0; i < M && !rc; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            rows[j] = i;
            cols[j] = j;
        }
        rc = oracle_gemm_ex_elems(ab_type, trans_a, trans_b, A, B, M, N, K, lda, ldb, rows, cols, N, S64 + i * N,
                                  S + i * N);
    }
    free(rows);
    free(cols);
    if (!rc) {
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j) {
                double x = alpha * S64[i * N + j];
                if (beta != 0.0) x += beta * decode_any(Cin, cin_type, i * ldcin + j);
                if (bias) x += decode_any(bias, bias_type, j);
                const float f = (float)x;
                if (d_type == 2)
                    ((float *)D)[i * ldd + j] = f;
                else if (d_type == 1)
                    ((uint16_t *)D)[i * ldd + j] = oracle_f32_to_bf16(f);
                else
                    ((uint16_t *)D)[i * ldd + j] = oracle_f32_to_f16(f);
            }
    }
    free(S);
    free(S64);
    return rc;
}

/* ---------------------------------------------------------------------------------
 * Row softmax ("06_triton_style.py", demo 3: the fused softmax workload): for each row x
 * of an M x N FP32 matrix,
 *
 *     y[j] = exp(x[j] - max_k x[k]) / sum_k exp(x[k] - max_k x[k])
 *
 * in FP64 (the max subtracted first, as the page's kernels do, so exp never overflows),
 * rounded once to FP32.  exp(-inf) = 0; a row whose maximum is +inf or NaN, or that is
 * all -inf, has no finite softmax and yields NaN in every element.
 * --------------------------------------------------------------------------------- */
int oracle_softmax_rows_f32(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy)
{
    if (M < 0 || N < 0 || ldx < N || ldy < N) return 1;
    if (M > 0 && N > 0 && (!X || !Y)) return 1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < M; ++i) {
        const float *x = X + i * ldx;
        float *y = Y + i * ldy;
        double m = -INFINITY;
        int bad = 0;
        for (int64_t j = 0; j < N; ++j) {
            if (isnan(x[j])) bad = 1;
            if ((double)x[j] > m) m = (double)x[j];
        }
        if (bad || isinf(m)) {
            for (int64_t j = 0; j < N; ++j) y[j] = NAN;
            continue;
        }
        double s = 0.0;
        for (int64_t j = 0; j < N; ++j) s += exp((double)x[j] - m);
        for (int64_t j = 0; j < N; ++j) y[j] = (float)(exp((double)x[j] - m) / s);
    }
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
