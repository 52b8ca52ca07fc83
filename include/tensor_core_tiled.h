/*
 * tensor_core_tiled.h -- C ABI of the GB300 (sm_103a) FP16 -> FP32 tiled tensor-core GEMM.
 *
 * The operation is the blocked tensor-core matrix multiply that the lecture pages
 * centre on: C[M x N] = A[M x K] . B[K x N] with FP16 inputs, FP32 accumulation and an
 * FP32 result ("04_tensor_cores.py", function tc_matmul and demo 2: FP16 inputs, FP32
 * accumulation), correct for any shape, ragged edges included ("06_triton_style.py",
 * matmul_kernel and demo 1: out-of-range loads read as zero, out-of-range stores are
 * skipped).  All matrices are row-major with explicit leading dimensions.
 *
 * Conventions shared by every entry point below:
 *   - Pointers A, B, C are device-accessible addresses (cudaMalloc, torch CUDA tensors),
 *     except in the *_host entry points, which take host memory.  The caller owns all
 *     memory.  C must not overlap A or B.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All
 *     work is enqueued on it; no call synchronises the host.
 *   - C is overwritten (gemm_ex adds the beta * C term).  M == 0 or N == 0 is a no-op.
 *     K == 0 writes zeros (the empty sum) into the M x N block of C.  Only the M x N block
 *     is written: the elements between N and ldc, and memory outside the block, keep
 *     their bits.
 *   - Errors in the arguments are reported immediately through the return value and
 *     nothing is enqueued.  Device-side errors (a pipeline wait that exceeded its time
 *     limit) are recorded in a per-device error word read by gemm_f16_f32_get_error().
 *   - Calls may come from several host threads: per-device state (properties, memory
 *     pool, copy streams of the *_host calls) is created once under a lock.
 */
#ifndef TENSOR_CORE_TILED_H
#define TENSOR_CORE_TILED_H

#include <stdint.h>

#if defined(__GNUC__)
#define TCT_API __attribute__((visibility("default")))
#else
#define TCT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* bad size, leading dimension, pointer or option */
    GEMM_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not sm_103 (GB300)            */
    GEMM_ERR_CUDA = 3,               /* a CUDA runtime/driver call failed               */
    GEMM_ERR_DEVICE_TIMEOUT = 4      /* a device pipeline wait exceeded its time limit  */
} gemm_status;

/*
 * gemm_f16_f32 -- C = A . B, FP16 x FP16 -> FP32 accumulate -> FP32 C.
 *   A   : FP16, M x K, row-major, element (i, k) at A[i*lda + k]; lda >= K.
 *   B   : FP16, K x N, row-major, element (k, j) at B[k*ldb + j]; ldb >= N.
 *   C   : FP32, M x N, row-major, element (i, j) at C[i*ldc + j]; ldc >= N.
 *   M, N, K : 0 <= M, N, K < 2^31.
 * Any alignment and any leading dimension are accepted.  When lda or ldb is not a
 * multiple of 8 elements, or A or B is not 16-byte aligned, the operand is first copied
 * on `stream` into a stream-ordered temporary whose rows are 16-byte aligned.  Temporaries
 * (these copies, and the flags -- with an epilogue also the parts -- of split tiles, see
 * gemm_options) come from a library-owned stream-ordered memory pool per device
 * (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`) that keeps freed memory for reuse
 * until the process exits.  The result does not depend on which path ran.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (negative or oversized dims, lda < K, ldb < N,
 * ldc < N, NULL pointer with a non-empty extent), GEMM_ERR_UNSUPPORTED_DEVICE or
 * GEMM_ERR_CUDA.
 */
TCT_API gemm_status gemm_f16_f32(const void *A, const void *B, float *C, int64_t M, int64_t N,
                         int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void *stream);

/*
 * Tuning options for gemm_f16_f32_ex.  Zero in any field selects the library default.
 *   group_m   : output tile rows per launch-order group ("06_triton_style.py",
 *               matmul_kernel and demo 2: GROUP_M program order for L2 reuse); 1 gives
 *               row-major tile order.  Range 1..256.
 *   tile_n    : output tile width in columns: 128 or 256, or 192 (CTA pairs only).
 *   stages    : shared-memory pipeline depth (a compiled depth for the chosen tile).
 *   max_ctas  : cap on the persistent grid in CTAs (default: every co-resident CTA).
 *   timeout_ms: limit on any single device pipeline wait (default 2000 ms).
 *   cta_group : 1 = one CTA per 128-row tile, 2 = a CTA pair per 256-row tile.
 *   stream_k  : 1 = whole tiles only; 2 = split each tile of the last, partial wave into
 *               two k-parts: its owner unit takes the first split_kb k-blocks and one of the
 *               units left over takes the rest (a helper may take several tiles' second
 *               parts in turn; see gemm_plan).  With the plain FP32 epilogue, a C whose
 *               base and row pitch are 16-byte multiples and N a multiple of 4 (the TMA
 *               writes whole 16-byte units of a row), the owner zeroes the tile in C and
 *               both parts are added into it by TMA reduce-add; otherwise the second part goes
 *               through a stream-ordered workspace and the owner adds it.  Every tile has two
 *               contributions, so the sum does not depend on their order and results are
 *               reproducible.
 *               3 = stream-K (plain FP32 epilogue and a C that TMA writes, as above; else
 *               GEMM_ERR_INVALID_ARG at launch): after whole waves of tiles, the k-blocks of
 *               the remaining tiles are cut into contiguous ranges of balanced length, one per
 *               unit, so that every unit finishes together even when there are fewer tiles
 *               than units ("02_gpu_execution_model.py", part 5: a partial wave leaves SMs
 *               idle).  A tile's k-loop may then be spread over several consecutive units;
 *               its pieces reach C in a fixed order, the last piece stored first and each
 *               earlier piece added by TMA reduce-add once the next one is in C, so results
 *               are reproducible bit for bit.  No workspace is used.
 *               0 = let the planner decide among whole tiles, 2 and 3.
 *   fault_inject: test hook for the device-side timeout path; 0 in normal use.  Bit 0: split
 *               tiles are never published (the owner neither zeroes nor flags its tile, the
 *               helper never flags its part, or a stream-K piece that starts inside a tile
 *               never flags it), so the waits for them run until timeout_ms,
 *               record GEMM_ERR_DEVICE_TIMEOUT (read by gemm_f16_f32_get_error) and return
 *               without storing those tiles.  Bit 1 (gemm_ex with beta != 0 on a C that TMA
 *               writes): the epilogue never loads C's blocks, so its waits for them run out
 *               the same way and no tile is stored.  Nothing faults, traps or hangs; later
 *               calls are unaffected.  Values above 3 are rejected.
 */
typedef struct gemm_options {
    int32_t group_m;
    int32_t tile_n;
    int32_t stages;
    int32_t max_ctas;
    int32_t timeout_ms;
    int32_t cta_group;
    int32_t stream_k;
    int32_t fault_inject;
} gemm_options;

/* gemm_f16_f32 with explicit tuning options (opt may be NULL = all defaults). */
TCT_API gemm_status gemm_f16_f32_ex(const void *A, const void *B, float *C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void *stream,
                            const gemm_options *opt);

/* Operand element type and storage of gemm_f32acc. */
typedef enum gemm_dtype { GEMM_DTYPE_F16 = 0, GEMM_DTYPE_BF16 = 1, GEMM_DTYPE_F32 = 2 } gemm_dtype;
typedef enum gemm_op { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op;

/*
 * gemm_f32acc -- C = op(A) . op(B) with FP16 or BF16 operands, FP32 accumulation, FP32 C.
 * The same blocked tensor-core product as gemm_f16_f32, with the operand storage and type
 * chosen by the caller:
 *   ab_type : GEMM_DTYPE_F16 or GEMM_DTYPE_BF16 (both operands).
 *   op_a    : GEMM_OP_N -- A stored M x K row-major, op(A)(i, k) = A[i*lda + k], lda >= K;
 *             GEMM_OP_T -- A stored K x M row-major (column-major M x K), op(A)(i, k) =
 *             A[k*lda + i], lda >= M.
 *   op_b    : GEMM_OP_N -- B stored K x N row-major, op(B)(k, j) = B[k*ldb + j], ldb >= N;
 *             GEMM_OP_T -- B stored N x K row-major, op(B)(k, j) = B[j*ldb + k], ldb >= K.
 *   C       : FP32, M x N row-major, ldc >= N.
 * Everything else (alignment handling, options, errors, stream semantics) is as for
 * gemm_f16_f32_ex; the stages option must name a variant compiled for the layout (the
 * planner's defaults always are).
 */
TCT_API gemm_status gemm_f32acc(int32_t ab_type, int32_t op_a, int32_t op_b, const void *A, const void *B,
                                float *C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                int64_t ldc, void *stream, const gemm_options *opt);

/*
 * Epilogue of gemm_ex: C = alpha * op(A).op(B) + beta * C + bias[j] for every row, computed
 * in FP32 and stored in C's type (narrower types by round to nearest even).
 *   alpha, beta : finite scale factors; beta == 0 means C is not read (any content, NaN
 *                 included, is overwritten).
 *   bias        : NULL, or N values of bias_type added to each row (aligned to its type).
 *   bias_type   : GEMM_DTYPE_F32, GEMM_DTYPE_F16 or GEMM_DTYPE_BF16.
 *   reserved    : must be zero.
 */
typedef struct gemm_epilogue {
    float alpha;
    float beta;
    const void *bias;
    int32_t bias_type;
    int32_t reserved;
} gemm_epilogue;

/*
 * gemm_ex -- C = alpha * op(A).op(B) + beta * C + bias, FP16/BF16 operands stored as for
 * gemm_f32acc, FP32 accumulation, C of c_type (GEMM_DTYPE_F32, F16 or BF16), row-major with
 * ldc >= N and aligned to its type.  epi may be NULL (alpha 1, beta 0, no bias).  With
 * K == 0 the product is the empty sum, so C = beta * C + bias.  Stream semantics, options
 * and errors as for gemm_f16_f32_ex.
 */
TCT_API gemm_status gemm_ex(int32_t ab_type, int32_t op_a, int32_t op_b, const void *A, const void *B, void *C,
                            int32_t c_type, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                            int64_t ldc, const gemm_epilogue *epi, void *stream, const gemm_options *opt);

/*
 * Launch plan the library would use for a problem (host only, no GPU needed when
 * num_sms > 0 is given; num_sms <= 0 queries the current device), for gemm_f16_f32 with
 * 16-byte aligned bases and ldc a multiple of 4: split tiles are planned as combined by TMA
 * reduce-add when N is a multiple of 4, through workspace otherwise.
 */
typedef struct gemm_plan {
    int32_t tile_m, tile_n, tile_k; /* output tile and k-block                        */
    int32_t stages;                 /* shared-memory pipeline depth                   */
    int32_t group_m;                /* launch-order group height (tiles)              */
    int32_t grid;                   /* persistent CTAs launched                       */
    int64_t tiles;                  /* output tiles                                   */
    int64_t waves;                  /* ceil(tiles / grid)                             */
    double wave_efficiency;         /* M*N / (waves * grid * tile_m * tile_n)          */
    int32_t smem_bytes;             /* dynamic shared memory per CTA                  */
    int32_t pack_a, pack_b;         /* 1 if the operand would be repacked first       */
    int32_t cta_group;              /* CTAs sharing one tile (1 or 2)                 */
    int32_t units;                  /* persistent work units (CTAs or CTA pairs)      */
    int32_t stream_k_tiles;         /* tiles whose k-loop may be split across units   */
    double effective_waves;         /* tile-times per unit: whole waves + split share */
    int32_t split_kb;               /* form 1: k-block where a split tile's second part
                                       starts; form 2: the shortest unit range (k-blocks) */
    int32_t split_parts_per_unit;   /* form 1: second parts a helper unit takes in turn;
                                       form 2: most pieces one tile is cut into */
    int32_t split_form;             /* 0 whole tiles, 1 two-part split tail (stream_k 2),
                                       2 stream-K ranges (stream_k 3)                    */
    int32_t sk_units;               /* form 2: units sharing the stream-K k-blocks     */
} gemm_plan;

TCT_API gemm_status gemm_f16_f32_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                              int32_t num_sms, const gemm_options *opt, gemm_plan *out);

/*
 * Launch-order map of the tile scheduler (host copy of the device function): linear tile
 * index t -> (tile row, tile column) with GROUP_M grouping ("06_triton_style.py",
 * matmul_kernel: groups of group_m tile rows, walked down the rows first).  Returns
 * GEMM_ERR_INVALID_ARG when t is out of range or a count is not positive.
 */
TCT_API gemm_status gemm_tile_coord(int64_t t, int64_t num_m, int64_t num_n, int32_t group_m,
                            int64_t *tile_row, int64_t *tile_col);

/*
 * One work item of a persistent unit (a CTA, or a CTA pair when cta_group is 2): k-blocks
 * [kb0, kb1) of linear tile `tile`.  mode 0: store the tile to C.  A tile of the last,
 * partial wave may be split into two k-parts: mode 1 is its owner (k-blocks [0, split_kb)),
 * mode 2 the helper computing the rest; `part` numbers the split tile (its flag, and its
 * workspace slot when the parts are combined through workspace).  mode 3: a stream-K piece
 * of a tile (split_form 2), `part` = the unit, whose flag it raises when kb0 > 0.
 */
typedef struct gemm_work {
    int32_t tile, kb0, kb1;
    int32_t mode;
    int32_t part; /* -1 when mode == 0 */
} gemm_work;

/*
 * Work item `idx` of unit `unit` in the plan the library would use for (M, N, K) on num_sms
 * SMs (host only).  Returns GEMM_ERR_INVALID_ARG when the unit has no such item.  Every
 * (tile, k-block) pair belongs to exactly one item of one unit.
 */
TCT_API gemm_status gemm_f16_f32_work_item(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                                           const gemm_options *opt, int32_t unit, int32_t idx,
                                           gemm_work *out);

/*
 * Wave model ("02_gpu_execution_model.py", part 5, wave_utilization): tiles =
 * ceil(M/tile_m)*ceil(N/tile_n), waves = ceil(tiles/slots), utilisation = tiles /
 * (waves*slots).  Host only.
 */
TCT_API gemm_status gemm_wave_model(int64_t M, int64_t N, int64_t tile_m, int64_t tile_n, int64_t slots,
                            int64_t *tiles, int64_t *waves, double *utilization);

/*
 * gemm_f16_f32_noalloc -- gemm_f16_f32 for callers that cannot allocate device memory.
 * The lecture pages have no counterpart to this entry point; it exists for callers whose
 * device memory is owned by another allocator (a framework's caching pool, a server that
 * reserves the whole GPU at start-up), where a new driver allocation mid-run can fail or
 * stall, and for callers whose interface forbids using the CUDA allocator (an operator or
 * plugin API that provides only the input and output buffers).
 *   Arguments, layouts and results are those of gemm_f16_f32; the caller still provides A,
 *   B and C.  The call makes no cudaMalloc/cudaFree or other allocating call.  The only
 *   scratch it can need -- the aligned copy of A and/or B made when lda or ldb is not a
 *   multiple of 8 or a base is not 16-byte aligned -- lives in one library-owned device
 *   array of GEMM_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library keeps
 *   until the process exits.  GEMM_ERR_INVALID_ARG is returned, before any work is
 *   enqueued, when the repacked operands would need more than that (M * roundup(K, 8) * 2
 *   bytes for A plus K * roundup(N, 8) * 2 bytes for B, each rounded up to 256).
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *   with that device current; make that first call before any stream capture.
 *   All calls share the one array and it keeps the last call's contents (nothing in it
 *   needs to start at zero): calls that may run at the same time on the GPU (different
 *   streams without ordering between them) race on it and must be serialised by the caller.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
TCT_API gemm_status gemm_f16_f32_noalloc(const void *A, const void *B, float *C, int64_t M, int64_t N,
                                         int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void *stream);

/*
 * softmax_rows_f32 -- Y[i][j] = exp(X[i][j] - max_k X[i][k]) / sum_k exp(X[i][k] - max_k X[i][k])
 * for every row of an M x N FP32 matrix: the fused row softmax of "06_triton_style.py"
 * demo 3: one read of X and one write of Y, except for rows too long to stage on chip
 * (beyond 393216 columns when X and Y rows start on 16-byte boundaries, beyond 51200
 * otherwise), which are read twice.
 *   X, Y : FP32 device pointers, row-major, leading dimensions ldx, ldy >= N, 4-byte
 *          aligned; Y may be X itself (ldy == ldx), other overlaps are undefined.
 * exp(-inf) = 0; a row holding a NaN, whose maximum is +inf, or whose entries are all -inf
 * is written as NaN.  M == 0 or N == 0 is a no-op.  Stream-ordered, no host sync.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED_DEVICE or GEMM_ERR_CUDA.
 */
TCT_API gemm_status softmax_rows_f32(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                                     void *stream);

/*
 * gemm_f16_f32_host -- gemm_f16_f32 with A, B and C in host memory (same layouts, leading
 * dimensions and conventions).  A is cut into up to 4 row blocks and B into up to 4 column
 * blocks (whole 256-wide tiles); they are copied to the device interleaved (A0, B0, B1, A1,
 * A2, B2, ...), each block of C is multiplied on `stream` as soon as its row block of A and
 * column block of B have arrived, and copied back while later blocks are still in flight, so
 * the two copy directions and the tensor-core work overlap.  The copies run on two library
 * streams; the device copies of A, B and C come from the library's stream-ordered pool.  Host
 * memory should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to be
 * asynchronous; pageable memory gives the same result with serialised copies.
 * Stream-ordered: the work starts after everything queued on `stream` before the call, and
 * work queued on `stream` after it starts once C is complete in host memory; A, B and C must
 * stay valid until then.  The pages have no such call: they time device-resident operands;
 * this is the end-to-end form of the product for callers whose data lives in host memory.
 * Returns the statuses of gemm_f16_f32.
 */
TCT_API gemm_status gemm_f16_f32_host(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                                      int64_t lda, int64_t ldb, int64_t ldc, void *stream);

/*
 * softmax_rows_f32_host -- softmax_rows_f32 with X and Y in host memory (Y may be X with
 * ldy == ldx).  X is copied to one device buffer in 8 row blocks, each block is softmaxed in
 * place on `stream` as soon as it has arrived, and copied back to Y while later blocks are in
 * flight.  Stream and memory rules as for gemm_f16_f32_host; the page's fused softmax has no
 * host-buffer form.  Returns the statuses of softmax_rows_f32.
 */
TCT_API gemm_status softmax_rows_f32_host(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                                          void *stream);

/*
 * Dense FP16 tensor rate of this device per SM and clock, measured (the per-clock factor of
 * the GEMM's roofline, SMs x FLOP/clk/SM x SM clock, "04_tensor_cores.py" demo 3: the
 * arithmetic a tensor core delivers per SM per clock).  One CTA per SM issues n_mma
 * back-to-back tcgen05.mma.kind::f16 of 128 x 256 x 16 (FP32 accumulation in tensor memory,
 * operands in shared memory) from one thread and times them with the SM clock counter;
 * FLOP = n_mma x 2 x 128 x 256 x 16.  Writes the median over SMs to *flop_per_clk_sm and,
 * when not NULL, the smallest and largest to *min_flop_per_clk_sm / *max_flop_per_clk_sm.
 * Runs on `stream` and synchronises it.  n_mma in 1 .. 2^22, else GEMM_ERR_INVALID_ARG;
 * GEMM_ERR_DEVICE_TIMEOUT if the MMAs did not complete within 2 s (bounded wait).
 */
TCT_API gemm_status gemm_tensor_rate_probe(int32_t n_mma, void *stream, double *flop_per_clk_sm,
                                           double *min_flop_per_clk_sm, double *max_flop_per_clk_sm);

/*
 * Reads and clears the device error word of the current device: GEMM_OK, or
 * GEMM_ERR_DEVICE_TIMEOUT if a kernel launched since the last read gave up on a pipeline
 * wait (its output is then incomplete).  Synchronises the current device first.
 */
TCT_API gemm_status gemm_f16_f32_get_error(void);

/* Static description of a status code (never NULL). */
TCT_API const char *gemm_status_string(int status);

/* Library version string, e.g. "tensor_core_tiled 0.1 sm_103a". */
TCT_API const char *gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TENSOR_CORE_TILED_H */
