// gemm_internal.h -- declarations shared by the kernel translation unit and the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tct {

// Matches GEMM_ERR_DEVICE_TIMEOUT in the public header; the device word stores
// code | (wait site << 8).
constexpr unsigned GEMM_ERR_DEVICE_TIMEOUT_CODE = 4u;

struct KernelParams {
    void *C;  // element type c_type
    int64_t ldc;
    int32_t M, N, K;
    int32_t num_m, num_n, num_kb, num_tiles;
    int32_t group_m;
    int32_t vec_store;  // 1 when C is aligned to 4 elements and ldc % 4 == 0
    // Epilogue: C = alpha * acc + beta * C + bias[col], in c_type (0 FP16, 1 BF16, 2 FP32).
    // epi == 0 means alpha 1, beta 0, no bias (C is not read).
    int32_t c_type;
    int32_t epi;
    float alpha, beta;
    const void *bias;
    int32_t bias_type;
    int32_t bias_vec;  // 1 when bias is aligned for 4-element vector loads
    uint64_t timeout_ns;
    // Work split.  `units` CTAs (cta_group 1) or CTA pairs (cta_group 2) first take whole
    // tiles 0 .. dp_tiles-1 (tile u + i * units goes to unit u).  The last split_tiles tiles
    // (the partial last wave; 2 * split_tiles <= units) are each split into two halves of
    // the k-loop: unit j does the first half of tail tile j and owns it, unit split_tiles + j
    // the second half, which it writes to workspace slot j (tile_rows x tile_n FP32) before
    // raising flag[j * cta_group + rank]; the owner then adds that part to its own and
    // stores the tile.
    int32_t units;
    int32_t dp_tiles;
    int32_t split_tiles;
    int32_t split_kb;  // first k-block of a split tile's second part (the owner takes [0, split_kb))
    float *workspace;
    unsigned int *flags;
    int32_t fault_inject;  // bit 0: never publish a split tile (its part, or its zeroed C rows);
                           // bit 1: never issue the TMA loads of C (beta != 0)
    // How split tiles are combined.  0: the second half goes through workspace and the owner
    // adds it (any epilogue).  1 (plain FP32 epilogue, C TMA-addressable): the owner zeroes
    // its rows of the tile in C at kernel start and raises flag[part * cta_group + rank]; both
    // halves then add their accumulators into C with TMA reduce-add (the tensor map over C),
    // so C = (0 + a) + b = (0 + b) + a whichever half lands first.
    int32_t split_mode;
    // 1 when the tensor map over C is valid (C's base and row pitch 16-byte aligned, N a
    // whole number of 16-byte units): whole tiles are then written by TMA stores.
    int32_t c_tma;
    // split_mode 2 (stream-K; plain FP32 epilogue, C TMA-writable): after dp_tiles whole
    // tiles, the k-blocks of the last split_tiles tiles -- split_tiles * num_kb iterations in
    // tile order -- are cut into sk_units contiguous ranges of balanced length, one per unit
    // (sk_units <= units, every range non-empty).  A unit walks its range in order, so only
    // its first piece can start inside a tile and only its last can end inside one.  The
    // pieces of one tile lie on consecutive units and are combined in C in a fixed order, the
    // last piece first: a piece that reaches the tile's end is stored; a piece that ends
    // inside the tile waits until the next unit's piece is in C (flag[(u + 1) * cta_group +
    // rank]) and adds itself by TMA reduce-add; a piece that starts inside the tile raises
    // flag[u * cta_group + rank] once its rows are in C.  C = ((p_last + ...) + p_1) + p_0,
    // the same bits on every run.
    // split_mode 3: the same ranges when every range is at least a tile long less one k-block,
    // so that no tile has more than two pieces: the piece that starts the tile zeroes its
    // rows of C at kernel start and raises flag[(tile - dp_tiles) * cta_group + rank]; both
    // pieces add into C by TMA reduce-add once they see it, in either order, since
    // (0 + a) + b = (0 + b) + a.
    int32_t sk_units;
    // 1 when every B element is read by one tile only (a single row of tiles, num_m == 1):
    // B's TMA loads then mark their L2 lines evict-first, so that the stream of B does not
    // push out the A rows every tile re-reads (measured on GB300 at 128 x 16384 x 16384:
    // 94.3 -> 90.6 us).
    int32_t b_stream;
    // 1 when the operands do not fit in L2 and A's rows are re-read by several column tiles:
    // A's TMA loads then mark three quarters of their L2 lines evict-last, so that a GROUP_M
    // group's A rows survive the B columns streaming past them across its waves (measured on
    // GB300: DRAM reads -5 to -10% at 8192^3, 6144^3 and 16384 x 16384 x 4096, time unchanged).
    int32_t a_keep;
};

enum WorkMode : int32_t {
    WORK_STORE = 0,    // store the accumulator to C
    WORK_FIXUP = 1,    // add the part in workspace slot `part`, then store to C
    WORK_PARTIAL = 2,  // store the accumulator to workspace slot `part`, raise its flag
    WORK_CHAIN = 3,    // stream-K piece of a tile (split_mode 2 or 3); `part` is the unit
};

// One piece of work of a unit: k-blocks [kb0, kb1) of linear tile `tile`.
struct WorkItem {
    int32_t tile;
    int32_t kb0, kb1;
    int32_t mode;
    int32_t part;  // workspace slot (split tiles), else -1
};

// The idx-th work item of unit u (false when the unit has no more).
#if defined(__CUDACC__)
__host__ __device__
#endif
inline bool work_item(const KernelParams &p, int32_t u, int32_t idx, WorkItem &it)
{
    // whole tiles u, u + units, ... below dp_tiles
    const int32_t waves = u < p.dp_tiles ? (p.dp_tiles - 1 - u) / p.units + 1 : 0;
    it.part = -1;
    if (idx < waves) {
        it.tile = u + idx * p.units;
        it.kb0 = 0;
        it.kb1 = p.num_kb;
        it.mode = WORK_STORE;
        return true;
    }
    if (p.split_mode == 2 || p.split_mode == 3) {
        // Stream-K: the idx - waves-th tile piece of this unit's range [a, b) of iterations.
        if (u >= p.sk_units || p.split_tiles <= 0) return false;
        const int64_t iters = static_cast<int64_t>(p.split_tiles) * p.num_kb;
        const int64_t a = static_cast<int64_t>(u) * iters / p.sk_units;
        const int64_t b = static_cast<int64_t>(u + 1) * iters / p.sk_units;
        const int64_t t = a / p.num_kb + (idx - waves);
        const int64_t t0 = t * p.num_kb;
        const int64_t lo = a > t0 ? a : t0;
        const int64_t hi = b < t0 + p.num_kb ? b : t0 + p.num_kb;
        if (lo >= hi) return false;
        it.tile = p.dp_tiles + static_cast<int32_t>(t);
        it.kb0 = static_cast<int32_t>(lo - t0);
        it.kb1 = static_cast<int32_t>(hi - t0);
        const bool whole = it.kb0 == 0 && it.kb1 == p.num_kb;
        it.mode = whole ? WORK_STORE : WORK_CHAIN;
        it.part = whole ? -1 : u;
        return true;
    }
    // Split tail tile j = dp_tiles + j' (j' < split_tiles): unit j' owns k-blocks
    // [0, split_kb); the units_left = units - split_tiles other units are helpers, helper h
    // taking [split_kb, num_kb) of tails h, h + units_left, h + 2 * units_left, ... in turn.
    if (p.split_tiles <= 0) return false;
    if (u < p.split_tiles) {
        if (idx != waves) return false;
        it.tile = p.dp_tiles + u;
        it.part = u;
        it.kb0 = 0;
        it.kb1 = p.split_kb;
        it.mode = WORK_FIXUP;
        return true;
    }
    const int32_t helpers = p.units - p.split_tiles;
    const int32_t j = (u - p.split_tiles) + (idx - waves) * helpers;
    if (j >= p.split_tiles) return false;
    it.tile = p.dp_tiles + j;
    it.part = j;
    it.kb0 = p.split_kb;
    it.kb1 = p.num_kb;
    it.mode = WORK_PARTIAL;
    return true;
}

// Compiled (cta_group, tile_n, stages) variants of the main kernel.  cta_group 1: 128 x
// tile_n tiles, one CTA each; per stage 16 KB of A + tile_n * 128 B of B.  cta_group 2:
// 256 x tile_n tiles on a CTA pair; per CTA and stage 16 KB of A + tile_n * 64 B of B.
// The epilogue staging takes 16 KB more.
#define TCT_VARIANTS(X) \
    X(2, 192, 6)        \
    X(1, 256, 2)        \
    X(1, 256, 3)        \
    X(1, 256, 4)        \
    X(1, 128, 4)        \
    X(1, 128, 6)        \
    X(2, 256, 3)        \
    X(2, 256, 4)        \
    X(2, 256, 5)        \
    X(2, 256, 6)        \
    X(2, 128, 6)        \
    X(2, 128, 8)

// Variants compiled for the other operand layouts and BF16 (the planner's candidates).
#define TCT_VARIANTS_EX(X) \
    X(2, 256, 6)           \
    X(2, 192, 6)           \
    X(1, 256, 4)           \
    X(1, 128, 6)           \
    X(2, 128, 8)

// Operand layout and type of a launch: bit 0 = A stored K x M, bit 1 = B stored N x K,
// bit 2 = BF16 (else FP16).  0 is the FP16, untransposed form.
int variant_exists(int layout, int cta_group, int tile_n, int stages);

int variant_smem_bytes(int cta_group, int tile_n, int stages);

// 1 if the variant's stage buffers can hold a split tile's other half in its epilogue.
int variant_split_ok(int cta_group, int tile_n, int stages);

// Co-resident clusters of the variant on the current device (-1 if the query fails).
int variant_max_clusters(int cta_group, int tile_n, int stages);

// tp: 2-D FP32 map of the split-tile parts (box tile_n x 32), used when split tiles combine
// through workspace (split_mode 0).  tc: 2-D map over C in its own type (boxes of 128 bytes
// x 32 rows, 128-byte swizzle), used when p.c_tma is set.
cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tp, const CUtensorMap &tc,
                        const KernelParams &p, int layout, int cta_group, int tile_n, int stages, int grid,
                        cudaStream_t stream);
// The layouts 3..7 of launch_gemm, compiled in the second object of the kernel source.
cudaError_t launch_gemm_part1(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tp,
                              const CUtensorMap &tc, const KernelParams &p, int layout, int cta_group, int tile_n,
                              int stages, int grid, cudaStream_t stream);

// One matrix of a row copy: rows x cols elements of esz bytes (2 or 4), leading dimensions
// in elements; a NULL src skips it.
struct RowCopy {
    const void *src;
    int64_t ld_src;
    void *dst;
    int64_t ld_dst;
    int64_t rows, cols;
    int32_t esz;
};

// Copies up to two matrices in one launch between layouts whose rows may start on any element
// boundary (programmatic dependent launch: it waits for the kernel before it).
cudaError_t launch_copy_rows(const RowCopy &m0, const RowCopy &m1, cudaStream_t stream, int num_sms);

// Copies up to two FP16 operands (a NULL src skips one) into buffers with 16-byte aligned rows,
// in one launch.
cudaError_t launch_pack2(const void *src0, int64_t ld_src0, void *dst0, int64_t ld_dst0, int64_t rows0, int64_t cols0,
                         const void *src1, int64_t ld_src1, void *dst1, int64_t ld_dst1, int64_t rows1, int64_t cols1,
                         cudaStream_t stream);

// K == 0: C = beta * C + bias[col] (the empty sum), or zeros when epi == 0.
cudaError_t launch_fill_epilogue(const KernelParams &p, int num_sms, cudaStream_t stream);

cudaError_t read_and_clear_error(unsigned *out);
// The second object's error word, read and cleared (read_and_clear_error reads both).
cudaError_t read_and_clear_error_part1(unsigned *out);

// Device address of the library's error word (code | wait site << 8) on the current device.
cudaError_t error_word_address(unsigned **out);

// Row softmax of an M x N FP32 matrix (softmax_sm103a.cu).  `err` is the error word that
// a timed-out wait records into; `timeout_ns` bounds every wait.
cudaError_t launch_softmax_rows(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy, int num_sms,
                                unsigned *err, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace tct
