// gemm_sm103a.cu -- persistent, warp-specialised FP16 x FP16 -> FP32 GEMM for GB300 (sm_103a).
//
// C[M x N] = A[M x K] . B[K x N], all row-major, FP32 accumulation in tensor memory.
// This is the blocked tensor-core matrix multiply of the lecture pages ("04_tensor_cores.py",
// tc_matmul and demo 2; "06_triton_style.py", matmul_kernel), re-designed for the
// 5th-generation tensor core instead of the mma.sync/ldmatrix and Triton realisations the
// pages describe:
//
//   * Block tiling with a K loop: each tile is (128 * CG) x BN outputs, K is walked in
//     64-element blocks ("04_tensor_cores.py", tc_matmul: BM x BN blocks, a BK loop).
//     CG = 1: one CTA per tile.  CG = 2: a CTA pair (cluster of 2) shares one 256-row tile;
//     each CTA loads its own 128 rows of A and half of the tile's B columns, the even CTA
//     issues M = 256 MMAs that read both CTAs' shared memory, and each CTA's TMEM receives
//     its 128 rows -- half the B bytes per SM of the CG = 1 form for the same work.
//   * Operand tiles reach shared memory through TMA with the 128-byte swizzle, the
//     hardware form of the XOR swizzle of demo 2 (16-byte chunk index XOR row mod 8), so
//     tensor-core reads of any 8 rows hit distinct banks.  A (K-major) and B (row-major,
//     i.e. N-major) are consumed as stored: B needs no transposed copy.
//   * A ring of STAGES shared-memory stages guarded by mbarriers, sized by the Little's-law
//     argument of "04_tensor_cores.py" demo 4 (data in flight = consumption rate x latency,
//     capped by the 227 KB of shared memory).
//   * Warp specialisation (demo 4, observation 4: one producer issues TMA, consumers only
//     compute): warp 0 issues TMA, warp 1 issues tcgen05.mma from one thread, warps 2..5
//     drain the FP32 accumulators from TMEM.  Two TMEM accumulator buffers let the
//     epilogue of one tile overlap the main loop of the next.
//   * A persistent grid walks the tiles in GROUP_M launch order ("06_triton_style.py",
//     matmul_kernel / demo 2) for L2 reuse.
//   * Ragged shapes ("06_triton_style.py", matmul_kernel masks): TMA fills out-of-range
//     operand elements with zeros (the masked load with other = 0); the epilogue writes C
//     with TMA stores from swizzled staging blocks where the hardware clips rows >= M and
//     columns >= N (the masked store), or, where TMA cannot write C, with per-lane stores
//     predicated on row < M and column < N.
//   * Every pipeline wait sleeps in hardware (mbarrier try_wait with a suspend-time hint)
//     and is bounded in wall time; on expiry the CTA records an error code in a device
//     word, drains its own copies and MMAs, frees TMEM and returns.
//   * Launched as a programmatic dependent launch: the set-up may overlap the previous
//     kernel on the stream; global memory is touched only after waiting for it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "gemm_internal.h"
#include "ptx_sm103a.cuh"
#include "tile_sched.h"

// The file compiles as two objects that run in parallel: TCT_PART 0 holds the kernels of the
// row-major and single-transpose FP16 layouts and every host-side function, TCT_PART 1 the
// kernels of the other layouts (each object keeps its own device error word; the host reads
// and clears both).
#ifndef TCT_PART
#define TCT_PART 0
#endif

namespace tct {

static __device__ unsigned int g_error_word;

template <int CG_, int BN_, int STAGES_, bool AT_ = false, bool BT_ = false, bool BF16_ = false>
struct Cfg {
    static constexpr bool AT = AT_;      // A stored K x M (transposed): MN-major A tiles
    static constexpr bool BT = BT_;      // B stored N x K (transposed): K-major B tiles
    static constexpr bool BF16 = BF16_;  // BF16 operands instead of FP16
    static constexpr int CG = CG_;            // CTAs per tile (1 or 2)
    static constexpr int BM = 128;            // tile rows held by one CTA
    static constexpr int BN = BN_;            // tile columns (the MMA's N)
    static constexpr int BN_CTA = BN_ / CG_;  // B columns loaded by one CTA
    static constexpr int BK = 64;             // 64 FP16 = 128 bytes = one swizzle row
    static constexpr int STAGES = STAGES_;
    static constexpr int UMMA_K = 16;         // K of one kind::f16 MMA
    static constexpr int A_STAGE = BM * BK * 2;
    static constexpr int B_SUB = BK * 64 * 2;  // one 64-column TMA box of B
    // TMA boxes of B per stage: B as K x N arrives in 64-column boxes (a CTA of a 192-column
    // pair tile holds 96 columns: two boxes, the second one's last 32 columns unused); B as
    // N x K arrives as one K-major box of BN_CTA rows.
    static constexpr int B_BOXES = BT_ ? 1 : (BN_CTA + 63) / 64;
    static constexpr int A_BOXES = AT_ ? 2 : 1;            // TMA boxes of A per stage
    static constexpr int B_STAGE = BT_ ? BK * BN_CTA * 2 : B_BOXES * B_SUB;
    static constexpr int STAGE_TX = CG * (A_STAGE + B_STAGE);  // bytes counted on one full barrier
    static constexpr int EPI_WARPS = 4;
    static constexpr int EPI_BYTES = EPI_WARPS * 32 * 32 * 4;
    static constexpr int BIAS_BYTES = EPI_WARPS * BN_ * 4;  // a tile's bias, per epilogue warp
    static constexpr int NUM_BARS = 2 * STAGES + 6 + 2 * EPI_WARPS;
    // A split tile's part (32 rows x BN FP32 per epilogue warp) is loaded into the stage
    // buffers, which are idle by then; only variants with room for it split tiles.
    static constexpr bool SPLIT_OK = STAGES * (A_STAGE + B_STAGE) >= EPI_WARPS * 32 * BN * 4;
    // The last tile of a unit, for a C that TMA cannot write, is staged as whole rows (32 per
    // epilogue warp, BN + 4 floats apart) in the idle stage buffers.
    static constexpr int ROW_PITCH = BN + 4;
    static constexpr bool ROWS_OK = STAGES * (A_STAGE + B_STAGE) >= EPI_WARPS * 32 * ROW_PITCH * 4;
    // two accumulator buffers of BN columns; the allocation is a power of two of at least 32
    static constexpr int TMEM_COLS = 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
    static constexpr int SMEM_BYTES =
        1024 + STAGES * (A_STAGE + B_STAGE) + EPI_BYTES + BIAS_BYTES + NUM_BARS * 8 + 16;
    static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair per tile");
    static_assert(BN_CTA % 32 == 0 && BN % 64 == 0 && BN <= 256, "B columns per CTA: a multiple of 32");
    static_assert(B_STAGE % 1024 == 0, "each stage's B starts on a 1024-byte swizzle boundary");
    static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM columns");
    static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory");
};

enum WaitSite : unsigned {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_FULL = 2,
    SITE_MMA_TMEM_EMPTY = 3,
    SITE_EPI_TMEM_FULL = 4,
    SITE_PRODUCER_TAIL = 5,
    SITE_EPI_PARTS = 6,
};

__device__ __forceinline__ void record_timeout(volatile int *abort_flag, unsigned site)
{
    atomicCAS(&g_error_word, 0u, (unsigned)GEMM_ERR_DEVICE_TIMEOUT_CODE | (site << 8));
    *abort_flag = 1;
    __threadfence_block();
}

template <bool kCluster>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity)
{
    if constexpr (kCluster)
        return mbar_try_wait_cluster(bar, parity);
    else
        return mbar_try_wait(bar, parity);
}

// Bounded wait that also gives up as soon as another role of this CTA has aborted.
template <bool kCluster>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int *abort_flag, unsigned site)
{
    if (try_wait<kCluster>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (true) {
        if (try_wait<kCluster>(bar, parity)) return true;
        if ((++spins & 15u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                record_timeout(abort_flag, site);
                return false;
            }
        }
    }
}

// Destination of one accumulator: element (r, c) of the tile goes to base[r * ld + c] for
// r < rows and c < cols (coordinates relative to `base`); `vec` allows 16-byte stores,
// `streaming` marks stores that are not read again.  When `part` is set, element (r, c) of
// this warp's 32 rows of the split tile's other half, staged in shared memory as 32 rows
// of BN floats, is added before the store.
struct TileDst {
    void *base;
    int64_t ld;
    int64_t rows, cols;
    bool vec;
    bool streaming;
    const float *part;
    // epilogue (C stores only): out_type 0 FP16, 1 BF16, 2 FP32; when epi, the stored value
    // is alpha * acc + beta * (current C) + bias[col]
    int out_type;
    bool epi;
    float alpha, beta;
    const void *bias;
    int bias_type;
    bool bias_vec;  // bias aligned for 4-element vector loads
};

__device__ __forceinline__ float load_typed(const void *p, int type, int64_t i)
{
    if (type == 2) return __ldg(static_cast<const float *>(p) + i);
    const unsigned short h = __ldg(static_cast<const unsigned short *>(p) + i);
    return type == 1 ? __bfloat162float(__ushort_as_bfloat16(h)) : __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ unsigned short to_16bit(float v, int type)
{
    return type == 1 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

// Elements i .. i+3 of a typed array (those below `count`; the rest read as 0), with one
// 16- or 8-byte load when `vec` allows it and all four are present.
__device__ __forceinline__ float4 load4_typed(const void *p, int type, int64_t i, bool vec, int64_t count)
{
    if (vec && count >= 4) {
        if (type == 2) return __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
        const uint2 h = __ldg(reinterpret_cast<const uint2 *>(static_cast<const unsigned short *>(p) + i));
        const unsigned short u[4] = {static_cast<unsigned short>(h.x & 0xffffu), static_cast<unsigned short>(h.x >> 16),
                                     static_cast<unsigned short>(h.y & 0xffffu), static_cast<unsigned short>(h.y >> 16)};
        float f[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            f[e] = type == 1 ? __bfloat162float(__ushort_as_bfloat16(u[e])) : __half2float(__ushort_as_half(u[e]));
        return make_float4(f[0], f[1], f[2], f[3]);
    }
    float f[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (e < count) f[e] = load_typed(p, type, i + e);
    return make_float4(f[0], f[1], f[2], f[3]);
}

// Four values from their loaded bits: FP32 bits, or (`packed16`) four 16-bit values packed
// in .x and .y.
__device__ __forceinline__ float4 raw_to_float4(uint4 r, int type, bool packed16)
{
    if (!packed16) return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
    const unsigned short u[4] = {static_cast<unsigned short>(r.x & 0xffffu), static_cast<unsigned short>(r.x >> 16),
                                 static_cast<unsigned short>(r.y & 0xffffu), static_cast<unsigned short>(r.y >> 16)};
    float f[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        f[e] = type == 1 ? __bfloat162float(__ushort_as_bfloat16(u[e])) : __half2float(__ushort_as_half(u[e]));
    return make_float4(f[0], f[1], f[2], f[3]);
}

// The epilogue on 4 outputs: alpha * acc + beta * c + bias (c and bias already loaded).
__device__ __forceinline__ float4 apply_epilogue(const TileDst &d, float4 v, float4 c, float4 b)
{
    float4 y = make_float4(d.alpha * v.x, d.alpha * v.y, d.alpha * v.z, d.alpha * v.w);
    if (d.beta != 0.0f)
        y = make_float4(fmaf(d.beta, c.x, y.x), fmaf(d.beta, c.y, y.y), fmaf(d.beta, c.z, y.z), fmaf(d.beta, c.w, y.w));
    if (d.bias) y = make_float4(y.x + b.x, y.y + b.y, y.z + b.z, y.w + b.w);
    return y;
}

// Epilogue and store of 4 consecutive outputs (row grow, columns gcol..gcol+3), any type.
// With `applied` the epilogue has been applied to v already.
__device__ __forceinline__ void store_general(const TileDst &d, int64_t grow, int64_t gcol, float4 v,
                                              bool applied = false)
{
    const bool full = d.vec && gcol + 3 < d.cols;
    if (d.epi && !applied) {
        const int64_t count = d.cols - gcol;
        const float4 c = d.beta != 0.0f ? load4_typed(d.base, d.out_type, grow * d.ld + gcol, d.vec, count)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 b = d.bias ? load4_typed(d.bias, d.bias_type, gcol, d.bias_vec, count)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        v = apply_epilogue(d, v, c, b);
    }
    float x[4] = {v.x, v.y, v.z, v.w};
    if (d.out_type == 2) {
        float *dst = static_cast<float *>(d.base) + grow * d.ld + gcol;
        if (full) {
            __stcs(reinterpret_cast<float4 *>(dst), make_float4(x[0], x[1], x[2], x[3]));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (gcol + e < d.cols) __stcs(dst + e, x[e]);
        }
    } else {
        unsigned short *dst = static_cast<unsigned short *>(d.base) + grow * d.ld + gcol;
        if (full) {
            uint2 w;
            w.x = static_cast<uint32_t>(to_16bit(x[0], d.out_type)) |
                  (static_cast<uint32_t>(to_16bit(x[1], d.out_type)) << 16);
            w.y = static_cast<uint32_t>(to_16bit(x[2], d.out_type)) |
                  (static_cast<uint32_t>(to_16bit(x[3], d.out_type)) << 16);
            __stcs(reinterpret_cast<uint2 *>(dst), w);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (gcol + e < d.cols) dst[e] = to_16bit(x[e], d.out_type);
        }
    }
}

// One accumulator buffer (this warp's 32 TMEM lanes x BN columns) to global memory.
// `release` is called by lane 0 once every column has been read from TMEM.
template <int BN, typename Release>
__device__ __forceinline__ void store_accumulator(uint32_t t_row, const TileDst &d, int64_t row_base,
                                                  int64_t col_base, float *stage, int lane, Release release)
{
    const bool read_c = d.epi && d.beta != 0.0f;
    const int jj = lane & 7;
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + ch * 32, r);
        tmem_wait_ld();
        if (ch == BN / 32 - 1) {
            // Accumulator fully read: hand the buffer back to the MMA issuer.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
        }
        // Row `lane` of this 32 x 32 block into the staging buffer, 16-byte chunks
        // XOR-swizzled by row so the transposed read below is conflict-free.
        float4 *srow = reinterpret_cast<float4 *>(stage + lane * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            srow[j ^ (lane & 7)] =
                make_float4(__uint_as_float(r[4 * j + 0]), __uint_as_float(r[4 * j + 1]),
                            __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        __syncwarp();
        if (!d.vec && !d.epi && !d.part && d.out_type == 2) {
            // FP32 C whose rows are not 16-byte aligned (no vector stores): one row per
            // store instruction, lane = column, so each instruction writes 128 contiguous bytes.
            const int64_t gc = col_base + ch * 32 + lane;
            const int swz = lane & 3;
#pragma unroll 8
            for (int rr = 0; rr < 32; ++rr) {
                const int64_t grow = row_base + rr;
                const float v = stage[rr * 32 + ((((lane >> 2) ^ (rr & 7)) << 2) | swz)];
                if (grow < d.rows && gc < d.cols) __stcs(static_cast<float *>(d.base) + grow * d.ld + gc, v);
            }
            __syncwarp();
            continue;
        }
        // Coalesced, predicated stores: 8 lanes cover one 128-byte row segment.
        const int64_t gcol = col_base + ch * 32 + jj * 4;
        // Epilogue inputs, loaded before any store of this block: the bias of this lane's 4
        // columns (the same for its 8 rows), and C's current values when beta != 0 -- all 8
        // rows at once and unconverted, so that the loads are in flight together instead of
        // waiting behind the stores to C or behind each other's conversions.
        float4 bias4 = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 cin[8];
        if (d.epi && d.bias) bias4 = load4_typed(d.bias, d.bias_type, gcol, d.bias_vec, d.cols - gcol);
        if (read_c) {
            if (d.out_type != 2 && d.vec && d.cols - gcol >= 4) {
                // 16-bit C: all eight loads first, then the conversions
                uint2 raw[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int64_t grow = row_base + t * 4 + (lane >> 3);
                    raw[t] = grow < d.rows ? __ldg(reinterpret_cast<const uint2 *>(
                                                 static_cast<const unsigned short *>(d.base) + grow * d.ld + gcol))
                                           : make_uint2(0u, 0u);
                }
#pragma unroll
                for (int t = 0; t < 8; ++t) cin[t] = raw_to_float4(make_uint4(raw[t].x, raw[t].y, 0u, 0u), d.out_type, true);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int64_t grow = row_base + t * 4 + (lane >> 3);
                    cin[t] = grow < d.rows ? load4_typed(d.base, d.out_type, grow * d.ld + gcol, d.vec, d.cols - gcol)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
#pragma unroll
        for (int rr0 = 0; rr0 < 32; rr0 += 4) {
            const int rr = rr0 + (lane >> 3);
            float4 v = reinterpret_cast<const float4 *>(stage + rr * 32)[jj ^ (rr & 7)];
            if (d.part) {
                const float4 a = *reinterpret_cast<const float4 *>(d.part + rr * BN + ch * 32 + jj * 4);
                v.x += a.x;
                v.y += a.y;
                v.z += a.z;
                v.w += a.w;
            }
            const int64_t grow = row_base + rr;
            if (grow < d.rows && d.epi) {
                const float4 c = read_c ? cin[rr0 / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
                store_general(d, grow, gcol, apply_epilogue(d, v, c, bias4), true);
            } else if (grow < d.rows && d.out_type != 2) {
                store_general(d, grow, gcol, v);
            } else if (grow < d.rows) {
                float *dst = static_cast<float *>(d.base) + grow * d.ld + gcol;
                if (d.vec && gcol + 3 < d.cols) {
                    if (d.streaming)
                        __stcs(reinterpret_cast<float4 *>(dst), v);
                    else
                        __stcg(reinterpret_cast<float4 *>(dst), v);
                } else {
                    if (gcol + 0 < d.cols) __stcs(dst + 0, v.x);
                    if (gcol + 1 < d.cols) __stcs(dst + 1, v.y);
                    if (gcol + 2 < d.cols) __stcs(dst + 2, v.z);
                    if (gcol + 3 < d.cols) __stcs(dst + 3, v.w);
                }
            }
        }
        __syncwarp();
    }
}

// One accumulator buffer to an FP32 C whose rows TMA cannot address (a row pitch or base
// off the 16-byte grid), plain epilogue: lane l's row of the tile goes whole into
// rows + l * PITCH, shifted by the row's offset from the 16-byte grid in C, so that its
// elements sit at the same address modulo 16 in shared and global memory.  The row's body
// between its first and last 16-byte boundaries in C then goes out as one bulk copy
// (cp.async.bulk, issued by the lane), the at most three elements on either side by plain
// stores.  `rows` is 16-byte aligned with room for 32 x PITCH floats.  Returns once the
// copies have completed.  `release` is called by lane 0 once every column has been read
// from TMEM.
template <int BN, int PITCH, typename Release>
__device__ __forceinline__ void store_rows_bulk(uint32_t t_row, const TileDst &d, int64_t row_base, int64_t col_base,
                                                float *rows, int lane, Release release)
{
    static_assert(PITCH % 4 == 0 && PITCH >= BN + 3, "rows of whole 16-byte units with room for the shift");
    const int64_t grow = row_base + lane;
    const bool row_in = grow < d.rows;
    float *gdst = static_cast<float *>(d.base) + (row_in ? grow : 0) * d.ld + col_base;
    const int shift = static_cast<int>((reinterpret_cast<uintptr_t>(gdst) >> 2) & 3u);
    float *srow = rows + lane * PITCH + shift;
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + ch * 32, r);
        tmem_wait_ld();
        if (ch == BN / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) srow[ch * 32 + j] = __uint_as_float(r[j]);
    }
    const int64_t ncols = d.cols - col_base < BN ? d.cols - col_base : BN;
    if (row_in && ncols > 0) {
        const int64_t head = ((4 - shift) & 3) < ncols ? ((4 - shift) & 3) : ncols;
        const int64_t body = (ncols - head) & ~int64_t(3);
        if (body > 0) {
            fence_proxy_async_smem();  // this lane's generic writes before the async-proxy read
            bulk_store(gdst + head, smem_u32(srow + head), static_cast<uint32_t>(body * 4));
            bulk_commit_group();
        }
        for (int64_t c = 0; c < head; ++c) __stcs(gdst + c, srow[c]);
        for (int64_t c = head + body; c < ncols; ++c) __stcs(gdst + c, srow[c]);
        if (body > 0) bulk_wait_all();
    }
    __syncwarp();
}

// Two floats rounded to the 16-bit type (FP16 0, BF16 1) and packed, the first in the low half.
__device__ __forceinline__ uint32_t pack_16bit(float a, float b, int type)
{
    return static_cast<uint32_t>(to_16bit(a, type)) | (static_cast<uint32_t>(to_16bit(b, type)) << 16);
}

// One accumulator buffer written to C by TMA, when the tensor map over C can write it (C's
// base and row pitch 16-byte aligned, rows of whole 16-byte units).  The warp's 32 rows go
// out in blocks of 32 rows x 128 bytes: 32 FP32 columns (kWide false) or 64 FP16/BF16
// columns (kWide true), staged in the 128-byte-swizzled layout the tensor map names.  Each
// lane holds one row of 32 accumulator columns at a time (tcgen05.ld 32x32b) and applies
// the epilogue, alpha * acc + beta * C + bias[col], with the same operations as
// store_general (the bias from `sbias`, the tile's bias columns as floats, staged by the
// warp before the tile's accumulator was ready).  When beta != 0, C's block is first TMA-loaded into the staging block
// (barrier `cbar`, phase count `cphase`) and each lane overwrites its row there.  Lane 0
// then stores the block (kReduce false) or adds it (kReduce true: either half of a split
// tile under split_mode 1, plain FP32 only) at (row0, first column of the block); the
// hardware clips boxes that reach past C.  With kOwnBlocks, `stage` holds one 4 KB block
// (1024-byte aligned) per block of the accumulator, all C loads are issued at once and the
// copies go out back to back; otherwise it is one block, reused once the previous copy has
// read it.  `skip_c_load` (fault injection) never issues the C loads, so their waits run
// out.  Returns false if a C load did not arrive in time (after recording the timeout);
// else once the copies have read shared memory, and with kOwnBlocks once they have completed.
// `release` is called by lane 0 once every column has been read from TMEM.
// With kStageOnly (kOwnBlocks, FP32, no epilogue inputs) the blocks are only staged: nothing
// is issued, and issue_staged_blocks sends them later (a stream-K piece stages its
// accumulator while it waits for the next piece to reach C).
template <int BN, bool kReduce, bool kOwnBlocks, bool kWide, typename Release, bool kStageOnly = false>
__device__ __forceinline__ bool bulk_accumulator(uint32_t t_row, const void *tmap_c, int64_t row0, int64_t col0,
                                                 const TileDst &d, const float *sbias, float *stage, int lane,
                                                 uint32_t cbar, uint32_t &cphase, uint64_t limit,
                                                 volatile int *abort_flag, bool skip_c_load, Release release)
{
    static_assert(!(kReduce && kWide), "reduce-add of FP32 only");
    static_assert(!kStageOnly || (kOwnBlocks && !kWide), "staging alone needs a block per 32 FP32 columns");
    constexpr int kCols = kWide ? 64 : 32;  // columns per staged block (128-byte rows)
    constexpr int kChunk = kWide ? 8 : 4;   // columns per 16-byte unit
    constexpr int kUnits = 32 / kChunk;     // 16-byte units per 32 accumulator columns
    constexpr int kBlocks = BN / kCols;
    const bool read_c = d.epi && d.beta != 0.0f;
    const bool rows_in = row0 < d.rows;
    auto block_in = [&](int blk) { return rows_in && col0 + blk * kCols < d.cols; };
    auto load_c = [&](int blk, float *dst) {  // lane 0: C's block into dst, counted on cbar
        tma_load_2d(smem_u32(dst), tmap_c, static_cast<int32_t>(col0 + blk * kCols), static_cast<int32_t>(row0), cbar);
    };
    bool ok = true;
    if (kOwnBlocks && read_c) {
        int n = 0;
        for (int blk = 0; blk < kBlocks; ++blk) n += block_in(blk) ? 1 : 0;
        if (n > 0) {
            if (lane == 0 && !skip_c_load) {
                mbar_arrive_expect_tx(cbar, n * 4096u);
                for (int blk = 0; blk < kBlocks; ++blk)
                    if (block_in(blk)) load_c(blk, stage + blk * 32 * 32);
            }
            ok = wait_or_abort<false>(cbar, cphase & 1u, limit, abort_flag, SITE_EPI_PARTS);
            ++cphase;
        }
    }
    // The accumulator is read 32 columns at a time (a wide block takes two reads).
    for (int sb = 0; sb < BN / 32; ++sb) {
        const int blk = kWide ? sb >> 1 : sb;
        const int half = kWide ? sb & 1 : 0;
        const int64_t c0 = col0 + blk * kCols;  // first column of the staged block
        float *block = kOwnBlocks ? stage + blk * 32 * 32 : stage;
        if (!kOwnBlocks && half == 0) {
            if (blk > 0) {  // the previous block has been read out of the staging buffer
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
            }
            if (read_c && block_in(blk)) {
                if (lane == 0 && !skip_c_load) {
                    mbar_arrive_expect_tx(cbar, 4096u);
                    load_c(blk, block);
                }
            }
        }
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + sb * 32, r);
        tmem_wait_ld();
        if (sb == BN / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
        }
        if (!kOwnBlocks && half == 0 && read_c && block_in(blk)) {
            ok = wait_or_abort<false>(cbar, cphase & 1u, limit, abort_flag, SITE_EPI_PARTS) && ok;
            ++cphase;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint4 *srow = reinterpret_cast<uint4 *>(block + lane * 32);
#pragma unroll
        for (int u = 0; u < kUnits; ++u) {
            const int j = half * kUnits + u;  // 16-byte unit of the staged row
            const float *bj = sbias + blk * kCols + j * kChunk;  // bias of the unit's columns
            const uint4 craw = read_c ? srow[j ^ (lane & 7)] : make_uint4(0u, 0u, 0u, 0u);
            uint4 out;
            if constexpr (!kWide) {
                float4 v = make_float4(__uint_as_float(r[4 * u + 0]), __uint_as_float(r[4 * u + 1]),
                                       __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
                if (d.epi) {
                    const float4 b = d.bias ? *reinterpret_cast<const float4 *>(bj) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v = apply_epilogue(d, v, raw_to_float4(craw, 2, false), b);
                }
                out = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w));
            } else {
                float4 lo = make_float4(__uint_as_float(r[8 * u + 0]), __uint_as_float(r[8 * u + 1]),
                                        __uint_as_float(r[8 * u + 2]), __uint_as_float(r[8 * u + 3]));
                float4 hi = make_float4(__uint_as_float(r[8 * u + 4]), __uint_as_float(r[8 * u + 5]),
                                        __uint_as_float(r[8 * u + 6]), __uint_as_float(r[8 * u + 7]));
                if (d.epi) {
                    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 b_lo = d.bias ? *reinterpret_cast<const float4 *>(bj) : z;
                    const float4 b_hi = d.bias ? *reinterpret_cast<const float4 *>(bj + 4) : z;
                    lo = apply_epilogue(d, lo, raw_to_float4(make_uint4(craw.x, craw.y, 0u, 0u), d.out_type, true), b_lo);
                    hi = apply_epilogue(d, hi, raw_to_float4(make_uint4(craw.z, craw.w, 0u, 0u), d.out_type, true), b_hi);
                }
                out = make_uint4(pack_16bit(lo.x, lo.y, d.out_type), pack_16bit(lo.z, lo.w, d.out_type),
                                 pack_16bit(hi.x, hi.y, d.out_type), pack_16bit(hi.z, hi.w, d.out_type));
            }
            srow[j ^ (lane & 7)] = out;
        }
        if (kWide && half == 0) continue;  // the block's second half is still to come
        if constexpr (kStageOnly) continue;
        fence_proxy_async_smem();          // this lane's generic writes before the async-proxy read
        __syncwarp();
        if (lane == 0 && block_in(blk)) {
            if constexpr (kReduce)
                tma_reduce_add_2d(tmap_c, static_cast<int32_t>(c0), static_cast<int32_t>(row0), smem_u32(block));
            else
                tma_store_2d(tmap_c, static_cast<int32_t>(c0), static_cast<int32_t>(row0), smem_u32(block));
            bulk_commit_group();
        }
    }
    if constexpr (kStageOnly) {
        fence_proxy_async_smem();  // every block's generic writes before the later async-proxy reads
        __syncwarp();
        return ok;
    }
    if (lane == 0) {
        if constexpr (kOwnBlocks)
            bulk_wait_all();
        else
            bulk_wait_read_all();
    }
    __syncwarp();
    return ok;
}

// The blocks bulk_accumulator<..., kStageOnly> staged (FP32, one 4 KB block per 32 columns),
// added into C by TMA reduce-add back to back; returns once the writes have completed.
template <int BN>
__device__ __forceinline__ void issue_staged_blocks(const void *tmap_c, int64_t row0, int64_t col0, const TileDst &d,
                                                    const float *stage, int lane)
{
    if (lane == 0) {
        if (row0 < d.rows) {
            for (int blk = 0; blk < BN / 32; ++blk) {
                const int64_t c0 = col0 + blk * 32;
                if (c0 < d.cols)
                    tma_reduce_add_2d(tmap_c, static_cast<int32_t>(c0), static_cast<int32_t>(row0),
                                      smem_u32(stage + blk * 32 * 32));
            }
        }
        bulk_commit_group();
        bulk_wait_all();
    }
    __syncwarp();
}

// Waits until *flag is raised (by another CTA), bounded like the pipeline waits.
__device__ __forceinline__ bool wait_flag(const unsigned int *flag, uint64_t limit_ns, volatile int *abort_flag)
{
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (flag_acquire_gpu(flag) == 0u) {
        if ((++spins & 15u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                record_timeout(abort_flag, SITE_EPI_PARTS);
                return false;
            }
        }
    }
    return true;
}

template <int CG, int BN, int STAGES, bool AT, bool BT, bool BF16>
__global__ void __launch_bounds__(192, 1)
    gemm_tcgen05_f32acc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmC,
                        const KernelParams p)
{
    using Cf = Cfg<CG, BN, STAGES, AT, BT, BF16>;
    constexpr bool kPair = CG == 2;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms must start on 1024-byte boundaries of the shared space.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = sA + STAGES * Cf::A_STAGE;
    float *sEpi = reinterpret_cast<float *>(sB + STAGES * Cf::B_STAGE);
    float *sBias = sEpi + Cf::EPI_BYTES / 4;
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sBias) + Cf::BIAS_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cf::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t part_bar = bar0 + 8u * (2 * STAGES + 5);  // epilogue warps done with a part
    auto pload_bar = [&](int e) { return bar0 + 8u * (2 * STAGES + 6 + e); };  // part load, warp e
    // C load of epilogue warp e (beta != 0 with TMA-written C)
    auto cload_bar = [&](int e) { return bar0 + 8u * (2 * STAGES + 6 + Cf::EPI_WARPS + e); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA rank inside the pair (0 = the CTA that issues the MMAs) and this CTA's work unit.
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), Cf::EPI_WARPS * CG);
        }
        mbar_init(drain_bar, 1);
        mbar_init(part_bar, Cf::EPI_WARPS);
        for (int e = 0; e < Cf::EPI_WARPS; ++e) {
            mbar_init(pload_bar(e), 1);
            mbar_init(cload_bar(e), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if constexpr (kPair) {
            tmem_alloc_pair(smem_u32(tmem_slot), Cf::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), Cf::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // peer barriers initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t limit = p.timeout_ns;
    // Everything above touched only shared memory, tensor memory and the parameters, so it
    // may overlap the end of the previous grid on the stream; global memory waits for it.
    griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_parity[STAGES];
            bool issued[STAGES];
            for (int i = 0; i < STAGES; ++i) issued[i] = false, issued_parity[i] = 0;
            bool ok = true;
            WorkItem w;
            const bool b_first_out = !kPair && p.b_stream != 0;  // B read by one tile only
            const uint64_t b_policy = l2_policy_evict_first();
            const bool a_keep = p.a_keep != 0;  // A rows re-read across a group's waves
            const uint64_t a_policy = l2_policy_evict_last(0.75f);
            for (int idx = 0; ok && work_item(p, unit, idx, w); ++idx) {
                const TileCoord c = tile_coord(w.tile, p.num_m, p.num_n, p.group_m);
                const int32_t m0 = c.m * (Cf::BM * CG) + static_cast<int32_t>(rank) * Cf::BM;
                const int32_t n0 = c.n * BN + static_cast<int32_t>(rank) * Cf::BN_CTA;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_or_abort<kPair>(empty_bar(s), ph ^ 1u, limit, abort_flag,
                                              SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const int32_t k0 = kb * Cf::BK;
                    // Box coordinates (innermost first) of this stage's operand tiles:
                    //   A as M x K: one 64(K) x 128(M) box; A as K x M: two 64(M) x 64(K) boxes;
                    //   B as K x N: 64(N) x 64(K) boxes; B as N x K: one 64(K) x BN_CTA(N) box.
                    uint32_t fb = full_bar(s);
                    if constexpr (kPair) {
                        // Both CTAs' bytes are counted on the even CTA's full barrier.
                        fb = map_to_cta(full_bar(s), 0);
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(s), Cf::STAGE_TX);
                    } else {
                        mbar_arrive_expect_tx(full_bar(s), Cf::STAGE_TX);
                    }
                    auto load = [&](uint32_t dst, const CUtensorMap *tm, int32_t c0, int32_t c1) {
                        if constexpr (kPair)
                            tma_load_2d_pair(dst, tm, c0, c1, fb);
                        else
                            tma_load_2d(dst, tm, c0, c1, fb);
                    };
                    auto load_hint = [&](uint32_t dst, const CUtensorMap *tm, int32_t c0, int32_t c1, uint64_t pol) {
                        if constexpr (kPair)
                            tma_load_2d_pair_hint(dst, tm, c0, c1, fb, pol);
                        else
                            tma_load_2d_hint(dst, tm, c0, c1, fb, pol);
                    };
#pragma unroll
                    for (int j = 0; j < Cf::A_BOXES; ++j) {
                        const uint32_t dst = smem_u32(sA + s * Cf::A_STAGE + j * Cf::B_SUB);
                        const int32_t ac0 = AT ? m0 + 64 * j : k0, ac1 = AT ? k0 : m0;
                        if (a_keep)
                            load_hint(dst, &tmA, ac0, ac1, a_policy);
                        else
                            load(dst, &tmA, ac0, ac1);
                    }
#pragma unroll
                    for (int j = 0; j < Cf::B_BOXES; ++j) {
                        const uint32_t dst = smem_u32(sB + s * Cf::B_STAGE + j * Cf::B_SUB);
                        const int32_t bc0 = BT ? k0 : n0 + 64 * j, bc1 = BT ? n0 : k0;
                        if (b_first_out)
                            load_hint(dst, &tmB, bc0, bc1, b_policy);
                        else
                            load(dst, &tmB, bc0, bc1);
                    }
                    issued[s] = true;
                    issued_parity[s] = ph;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            griddep_launch_dependents();  // every load issued: the next grid may start launching
            if (ok) {
                // Tail: wait until the MMAs have released every stage, so that no arrival is
                // still on its way to this CTA's shared memory when it exits.
                for (int i = 0; i < STAGES; ++i) {
                    if (!wait_or_abort<kPair>(empty_bar(s), ph ^ 1u, limit, abort_flag, SITE_PRODUCER_TAIL))
                        break;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            } else if (kPair && rank != 0) {
                // This CTA's loads signal the peer's barrier: give them time to land.
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) __nanosleep(1000);
            } else {
                // Let this CTA's loads land before shared memory is released.
                for (int i = 0; i < STAGES; ++i)
                    if (issued[i]) (void)mbar_wait(full_bar(i), issued_parity[i], limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_f32acc(Cf::BM * CG, BN, /*a_mn_major=*/AT, /*b_mn_major=*/!BT, BF16);
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            bool any_mma = false;
            WorkItem w;
            for (; ok && work_item(p, unit, it, w); ++it) {
                const int b = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!wait_or_abort<kPair>(tempty_bar(b), (use & 1u) ^ 1u, limit, abort_flag,
                                          SITE_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_or_abort<kPair>(full_bar(s), ph, limit, abort_flag, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + s * Cf::A_STAGE);
                    const uint32_t b_base = smem_u32(sB + s * Cf::B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < Cf::BK / Cf::UMMA_K; ++kk) {
                        // K-major tiles: 128-byte rows of K, 8-row groups 1024 B apart (stride
                        // offset); a K step of 16 elements is 32 bytes inside the swizzle row.
                        // MN-major tiles: 64-element MN boxes B_SUB bytes apart (leading
                        // offset), 8-row K groups 1024 B apart; 16 K rows = 2048 B.
                        const uint64_t adesc = AT ? smem_desc_sw128(a_base + kk * 2048, Cf::B_SUB, 1024)
                                                  : smem_desc_sw128(a_base + kk * 32, 16, 1024);
                        const uint64_t bdesc = BT ? smem_desc_sw128(b_base + kk * 32, 16, 1024)
                                                  : smem_desc_sw128(b_base + kk * 2048, Cf::B_SUB, 1024);
                        const uint32_t acc = (kb != w.kb0 || kk != 0) ? 1u : 0u;
                        if constexpr (kPair)
                            tc_mma_f16_pair(d_tmem, adesc, bdesc, idesc, acc);
                        else
                            tc_mma_f16(d_tmem, adesc, bdesc, idesc, acc);
                    }
                    any_mma = true;
                    if constexpr (kPair)
                        tc_commit_pair_multicast(empty_bar(s), 0x3);
                    else
                        tc_commit(empty_bar(s));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (kPair)
                    tc_commit_pair_multicast(tfull_bar(b), 0x3);
                else
                    tc_commit(tfull_bar(b));
            }
            if (!ok && any_mma) {
                // Wait for this thread's MMAs before TMEM is released.
                if constexpr (kPair)
                    tc_commit_pair_multicast(drain_bar, 0x1);
                else
                    tc_commit(drain_bar);
                (void)mbar_wait(drain_bar, 0, limit);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        float *stage = sEpi + (warp - 2) * 32 * 32;
        float *sbias = sBias + (warp - 2) * BN;  // the current tile's bias columns (TMA path)
        if ((p.split_mode == 1 || p.split_mode == 3) && !(p.fault_inject & 1)) {
            // The owner of a split tile (the piece that starts it) zeroes its rows of the tile
            // in C while the first tile's k-loop runs, then raises the tile's flag for this CTA
            // rank; both pieces add into C once they see it.  (A unit owns at most one split
            // tile.)  Fault injection skips this, so that both pieces' waits run out and C keeps
            // its old contents there.
            WorkItem z;
            for (int i = 0; work_item(p, unit, i, z); ++i) {
                const bool owned = p.split_mode == 1 ? z.mode == WORK_FIXUP : (z.mode == WORK_CHAIN && z.kb0 == 0);
                if (!owned) continue;
                const int32_t slot = p.split_mode == 1 ? z.part : z.tile - p.dp_tiles;
                const TileCoord c = tile_coord(z.tile, p.num_m, p.num_n, p.group_m);
                const int64_t r0 = static_cast<int64_t>(c.m) * (Cf::BM * CG) + rank * Cf::BM + q * 32;
                const int64_t c0 = static_cast<int64_t>(c.n) * BN;
                float *Cz = static_cast<float *>(p.C);
                for (int rr = 0; rr < 32 && r0 + rr < p.M; ++rr) {
                    float *crow = Cz + (r0 + rr) * p.ldc;
                    for (int cc = lane * 4; cc < BN; cc += 128) {
                        const int64_t col = c0 + cc;
                        if (col + 3 < p.N) {
                            *reinterpret_cast<float4 *>(crow + col) = make_float4(0.f, 0.f, 0.f, 0.f);
                        } else {
                            for (int e = 0; e < 4; ++e)
                                if (col + e < p.N) crow[col + e] = 0.f;
                        }
                    }
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) mbar_arrive(part_bar);
                if (warp == 2 && lane == 0 && wait_or_abort<false>(part_bar, 0u, limit, abort_flag, SITE_EPI_PARTS))
                    flag_release_gpu(p.flags + slot * CG + rank, 1u);
                break;
            }
        }
        int it = 0;
        uint32_t cphase = 0;  // C loads completed on this warp's cload barrier
        WorkItem w;
        for (; work_item(p, unit, it, w); ++it) {
            const int b = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            const TileCoord c = tile_coord(w.tile, p.num_m, p.num_n, p.group_m);
            if (p.c_tma && p.bias && w.mode == WORK_STORE) {
                // The tile's bias, as floats, into this warp's copy while the MMAs still run.
                for (int i = lane; i < BN; i += 32) {
                    const int64_t col = static_cast<int64_t>(c.n) * BN + i;
                    sbias[i] = col < p.N ? load_typed(p.bias, p.bias_type, col) : 0.0f;
                }
                __syncwarp();
            }
            bool ok = wait_or_abort<kPair>(tfull_bar(b), use & 1u, limit, abort_flag, SITE_EPI_TMEM_FULL);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int64_t lane_rows = static_cast<int64_t>(rank) * Cf::BM + q * 32;  // tile-local
            constexpr int64_t kTileElems = static_cast<int64_t>(Cf::BM * CG) * BN;
            TileDst d{p.C,      p.ldc,      p.M,     p.N,    p.vec_store != 0, true,        nullptr,
                      p.c_type, p.epi != 0, p.alpha, p.beta, p.bias,            p.bias_type, p.bias_vec != 0};
            int64_t row_base = static_cast<int64_t>(c.m) * (Cf::BM * CG) + lane_rows;
            int64_t col_base = static_cast<int64_t>(c.n) * BN;
            const uint32_t t_row0 = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
            // C that TMA can write: a whole tile goes out by TMA stores after its epilogue, and
            // (plain FP32 epilogue) either half of a split tile by TMA reduce-adds into C,
            // zeroed by the tile's owner.  A unit's last accumulator is staged in the stage
            // buffers -- its MMAs have completed, so no stage is read or written again -- with
            // a block of its own for each 128-byte column block; the others share this warp's
            // staging block.
            auto release = [&] {
                if constexpr (kPair)
                    mbar_arrive_cluster(map_to_cta(tempty_bar(b), 0));
                else
                    mbar_arrive(tempty_bar(b));
            };
            WorkItem next;
            const bool own_blocks = Cf::SPLIT_OK && !work_item(p, unit, it + 1, next);
            const uint32_t cb = cload_bar(warp - 2);
            const bool skip_c = (p.fault_inject & 2) != 0;
            float *blocks = reinterpret_cast<float *>(sA) + (warp - 2) * 32 * BN;
            // One accumulator out by TMA: reduce-add (split half, FP32) or store, 16-bit (wide) or
            // FP32 blocks; staged in its own blocks when it is the unit's last.
            auto bulk = [&](auto reduce, auto wide) {
                constexpr bool kReduce = decltype(reduce)::value, kWide = decltype(wide)::value;
                return own_blocks ? bulk_accumulator<BN, kReduce, true, kWide>(t_row0, &tmC, row_base, col_base, d, sbias,
                                                                              blocks, lane, cb, cphase, limit, abort_flag,
                                                                              skip_c, release)
                                  : bulk_accumulator<BN, kReduce, false, kWide>(t_row0, &tmC, row_base, col_base, d, sbias,
                                                                               stage, lane, cb, cphase, limit, abort_flag,
                                                                               skip_c, release);
            };
            if (w.mode == WORK_CHAIN && p.split_mode == 3) {
                // Stream-K piece of a tile cut in at most two: add into C, zeroed by the tile's
                // first piece, whichever piece comes first.
                ok = wait_flag(p.flags + (w.tile - p.dp_tiles) * CG + rank, limit, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                fence_proxy_async_all();  // the owner's zeros (generic writes) before the reduce
                if (!bulk(std::true_type{}, std::false_type{})) break;
                continue;
            }
            if (w.mode == WORK_CHAIN) {
                // Stream-K piece: the tile's pieces reach C last-first.  A piece that ends
                // inside the tile waits for the next unit's piece, then adds itself; the piece
                // that reaches the tile's end is the first and is stored.
                const bool add = w.kb1 < p.num_kb;
                if (add && own_blocks) {
                    // The unit's last item (a piece that ends inside its tile always is): stage
                    // the whole accumulator in the idle stage buffers while the next piece is on
                    // its way, then add it into C in one burst once the flag is seen.
                    ok = bulk_accumulator<BN, true, true, false, decltype(release), true>(
                        t_row0, &tmC, row_base, col_base, d, sbias, blocks, lane, cb, cphase, limit, abort_flag, skip_c,
                        release);
                    ok = ok && wait_flag(p.flags + (unit + 1) * CG + rank, limit, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    fence_proxy_async_all();  // the flag seen before the reduce reads C
                    issue_staged_blocks<BN>(&tmC, row_base, col_base, d, blocks, lane);
                } else {
                    if (add) {
                        ok = wait_flag(p.flags + (unit + 1) * CG + rank, limit, abort_flag);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        fence_proxy_async_all();  // the flag seen before the reduce reads C
                    }
                    ok = add ? bulk(std::true_type{}, std::false_type{}) : bulk(std::false_type{}, std::false_type{});
                    if (!ok) break;
                }
                if (w.kb0 > 0) {
                    // A unit's only piece that starts inside a tile (its first): publish it to
                    // the previous unit once all four warps' rows are in C.
                    if (lane == 0) {
                        bulk_wait_all();
                        fence_proxy_async_all();
                    }
                    __syncwarp();
                    __threadfence();
                    if (lane == 0) mbar_arrive(part_bar);
                    if (warp == 2 && lane == 0 && wait_or_abort<false>(part_bar, 0u, limit, abort_flag, SITE_EPI_PARTS) &&
                        !(p.fault_inject & 1))
                        flag_release_gpu(p.flags + unit * CG + rank, 1u);
                }
                continue;
            }
            if (p.split_mode == 1 && w.mode != WORK_STORE) {
                ok = wait_flag(p.flags + w.part * CG + rank, limit, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                fence_proxy_async_all();  // the owner's zeros (generic writes) before the reduce
                if (!bulk(std::true_type{}, std::false_type{})) break;
                continue;
            }
            if (p.c_tma && w.mode == WORK_STORE) {
                ok = p.c_type == 2 ? bulk(std::false_type{}, std::false_type{}) : bulk(std::false_type{}, std::true_type{});
                if (!ok) break;
                continue;
            }
            if (w.mode == WORK_PARTIAL) {
                // second half of a split tile for its owner: the whole tile, tile-local rows
                d = TileDst{p.workspace + w.part * kTileElems, BN, Cf::BM * CG, BN, true, false, nullptr,
                            2, false, 1.0f, 0.0f, nullptr, 2, false};
                row_base = lane_rows;
                col_base = 0;
            } else if (w.mode == WORK_FIXUP) {
                if constexpr (Cf::SPLIT_OK) {
                    // The other half, once its unit has published it, comes in by TMA: this
                    // warp's 32 rows into the (idle) stage buffers, then it is added below.
                    ok = wait_flag(p.flags + w.part * CG + rank, limit, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    float *part = reinterpret_cast<float *>(sA) + (warp - 2) * 32 * BN;
                    const uint32_t pb = pload_bar(warp - 2);
                    if (lane == 0) {
                        fence_proxy_async_all();
                        mbar_arrive_expect_tx(pb, 32 * BN * 4);
                        tma_load_2d(smem_u32(part), &tmP, 0,
                                    static_cast<int32_t>(w.part * (Cf::BM * CG) + lane_rows), pb);
                    }
                    ok = wait_or_abort<false>(pb, 0u, limit, abort_flag, SITE_EPI_PARTS);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    d.part = part;
                }
            }
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(b * BN);
            if constexpr (Cf::ROWS_OK) {
                if (own_blocks && w.mode == WORK_STORE && !p.c_tma && !d.epi && d.out_type == 2) {
                    float *rows = reinterpret_cast<float *>(sA) + (warp - 2) * 32 * Cf::ROW_PITCH;
                    if constexpr (kPair) {
                        const uint32_t te = map_to_cta(tempty_bar(b), 0);
                        store_rows_bulk<BN, Cf::ROW_PITCH>(t_row, d, row_base, col_base, rows, lane,
                                                           [&] { mbar_arrive_cluster(te); });
                    } else {
                        const uint32_t te = tempty_bar(b);
                        store_rows_bulk<BN, Cf::ROW_PITCH>(t_row, d, row_base, col_base, rows, lane,
                                                           [&] { mbar_arrive(te); });
                    }
                    continue;
                }
            }
            if constexpr (kPair) {
                const uint32_t te = map_to_cta(tempty_bar(b), 0);
                store_accumulator<BN>(t_row, d, row_base, col_base, stage, lane, [&] { mbar_arrive_cluster(te); });
            } else {
                const uint32_t te = tempty_bar(b);
                store_accumulator<BN>(t_row, d, row_base, col_base, stage, lane, [&] { mbar_arrive(te); });
            }
            if (w.mode == WORK_PARTIAL) {
                // Publish this CTA's rows of the part to the owner once all four warps have
                // written theirs (through workspace a helper writes one part at most, so the
                // barrier's first phase).
                __threadfence();
                fence_proxy_async_all();
                __syncwarp();
                if (lane == 0) mbar_arrive(part_bar);
                if (warp == 2 && lane == 0 && wait_or_abort<false>(part_bar, 0u, limit, abort_flag, SITE_EPI_PARTS) &&
                    !(p.fault_inject & 1))
                    flag_release_gpu(p.flags + w.part * CG + rank, 1u);
            }
        }
        if (lane == 0) bulk_wait_all();  // every TMA store or reduce of this warp has completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // the pair's MMAs and remote arrivals are done
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem_base, Cf::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, Cf::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- helper kernels

// Row copy between two layouts whose rows may start on any element boundary, for up to two
// matrices in one launch.  It repacks operands into rows that start on 16-byte boundaries
// (TMA's stride rule) and moves a product from an aligned temporary into a C that TMA cannot
// write.  Each destination row is written in whole, aligned 16-byte units; the few elements
// before its first and after its last aligned unit are copied one by one.  The work is
// flattened: index u of row r (u < units_max, one more than the most whole units a row of
// this length can hold) is one thread's work -- aligned unit u when the row has that many,
// else, for the first index past the row's units, the row's loose elements -- so every
// thread has a single, independent copy in flight and the grid strides over all rows of
// both matrices.  The 16 source bytes of a unit may straddle two aligned 16-byte blocks: both
// are loaded whole and the bytes realigned with funnel shifts.  Each of the two blocks holds
// at least one byte of the unit, which lies inside the source row, so no load reaches
// outside the 16-byte blocks the row occupies.
constexpr int kCopyThreads = 256;

struct CopyJob {
    const uint8_t *src;
    int64_t ld_src;  // bytes between rows
    uint8_t *dst;
    int64_t ld_dst;  // bytes between rows
    int64_t rows;
    int64_t row_bytes;
    int32_t esz;        // element size: 2 or 4 bytes
    int64_t units_max;  // work indices per row
};

// 16 bytes starting at any byte address p, realigned from the two aligned blocks they touch.
__device__ __forceinline__ uint4 load16_realigned(const uint8_t *p)
{
    const uintptr_t addr = reinterpret_cast<uintptr_t>(p);
    const uint32_t off = static_cast<uint32_t>(addr & 15u);
    const uint4 *blk = reinterpret_cast<const uint4 *>(addr - off);
    const uint4 lo = __ldg(blk);
    const uint4 hi = off ? __ldg(blk + 1) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t q = off >> 2, sh = (off & 3u) * 8u;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = q == 0 ? w[i] : q == 1 ? w[i + 1] : q == 2 ? w[i + 2] : w[i + 3];
        const uint32_t b = q == 0 ? w[i + 1] : q == 1 ? w[i + 2] : q == 2 ? w[i + 3] : w[i + 4];
        o[i] = __funnelshift_r(a, b, sh);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Elements [e0, e1) of a row, one at a time.
__device__ __forceinline__ void copy_elements(const uint8_t *s, uint8_t *d, int64_t e0, int64_t e1, int esz)
{
    for (int64_t e = e0; e < e1; ++e) {
        if (esz == 4)
            reinterpret_cast<uint32_t *>(d)[e] = reinterpret_cast<const uint32_t *>(s)[e];
        else
            reinterpret_cast<uint16_t *>(d)[e] = reinterpret_cast<const uint16_t *>(s)[e];
    }
}

// Work index u of row r of job j.
__device__ __forceinline__ void copy_unit(const CopyJob &j, int64_t r, int64_t u)
{
    const uint8_t *s = j.src + r * j.ld_src;
    uint8_t *d = j.dst + r * j.ld_dst;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(d), d1 = d0 + static_cast<uintptr_t>(j.row_bytes);
    const uintptr_t a0 = (d0 + 15u) & ~uintptr_t(15), a1 = d1 & ~uintptr_t(15);
    const int64_t units = a1 > a0 ? static_cast<int64_t>(a1 - a0) >> 4 : 0;
    const int64_t head = units > 0 ? static_cast<int64_t>(a0 - d0) : 0;  // bytes before the first aligned unit
    if (u < units) {
        *reinterpret_cast<uint4 *>(d + head + 16 * u) = load16_realigned(s + head + 16 * u);
    } else if (u == units) {  // the loose elements: all of a row without a whole aligned unit
        const int64_t n = j.row_bytes / j.esz;
        if (units == 0) {
            copy_elements(s, d, 0, n, j.esz);
        } else {
            copy_elements(s, d, 0, head / j.esz, j.esz);
            copy_elements(s, d, (head + 16 * units) / j.esz, n, j.esz);
        }
    }
}

#if TCT_PART == 0
__global__ void __launch_bounds__(kCopyThreads) copy_rows(const CopyJob j0, const CopyJob j1)
{
    // Launched as a programmatic dependent launch: wait for the kernel before it (which may
    // write the source), then let the next kernel start its set-up; that kernel reads these
    // rows only after its own dependency wait, i.e. after this grid has completed.
    griddep_wait();
    griddep_launch_dependents();
    const int64_t t0 = j0.rows * j0.units_max, total = t0 + j1.rows * j1.units_max;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total; g += stride) {
        const bool first = g < t0;
        const CopyJob &j = first ? j0 : j1;
        const int64_t x = first ? g : g - t0;
        const int64_t r = x / j.units_max;
        copy_unit(j, r, x - r * j.units_max);
    }
}

// K == 0: the empty sum, through the epilogue (C = beta * C + bias[col], or zeros).
__global__ void fill_epilogue(const KernelParams p)
{
    TileDst d{p.C,     p.ldc,      p.M,     p.N,    false,  true,        nullptr,
              p.c_type, p.epi != 0, p.alpha, p.beta, p.bias, p.bias_type, p.bias_vec != 0};
    const int64_t cols4 = (static_cast<int64_t>(p.N) + 3) / 4;
    const int64_t total = static_cast<int64_t>(p.M) * cols4;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / cols4;
        const int64_t c = (i - r * cols4) * 4;
        store_general(d, r, c, make_float4(0.f, 0.f, 0.f, 0.f));
    }
}

#endif  // TCT_PART == 0

// ---------------------------------------------------------------- host side

template <int CG, int BN, int STAGES>
static cudaLaunchConfig_t launch_config(int grid, cudaStream_t stream, cudaLaunchAttribute *attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = Cfg<CG, BN, STAGES>::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int CG, int BN, int STAGES, bool AT, bool BT, bool BF16>
static cudaError_t launch_variant(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tp,
                                  const CUtensorMap &tc, const KernelParams &p, int grid, cudaStream_t stream)
{
    auto kern = gemm_tcgen05_f32acc<CG, BN, STAGES, AT, BT, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<CG, BN, STAGES>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config<CG, BN, STAGES>(grid, stream, attr);
    // programmatic dependent launch: the prologue may overlap the previous kernel's end
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    // split tiles combined through workspace or reduce-add need room for a part in the stage
    // buffers; stream-K pieces (split_mode 2) need none
    if (p.split_tiles > 0 && p.split_mode != 2 && !Cfg<CG, BN, STAGES>::SPLIT_OK) return cudaErrorInvalidValue;
    if ((p.split_mode == 2 || p.split_mode == 3) && !p.c_tma) return cudaErrorInvalidValue;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tp, tc, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Clusters of this variant that can be resident at once on the current device.
template <int CG, int BN, int STAGES>
static int max_clusters_variant()
{
    auto kern = gemm_tcgen05_f32acc<CG, BN, STAGES, false, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<CG, BN, STAGES>::SMEM_BYTES) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config<CG, BN, STAGES>(2048, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return n;
}

#if TCT_PART == 0
int variant_smem_bytes(int cta_group, int tile_n, int stages)
{
#define TCT_CASE(CG_, BN_, ST_) \
    if (cta_group == CG_ && tile_n == BN_ && stages == ST_) return Cfg<CG_, BN_, ST_>::SMEM_BYTES;
    TCT_VARIANTS(TCT_CASE)
#undef TCT_CASE
    return -1;
}

int variant_max_clusters(int cta_group, int tile_n, int stages)
{
#define TCT_CASE(CG_, BN_, ST_) \
    if (cta_group == CG_ && tile_n == BN_ && stages == ST_) return max_clusters_variant<CG_, BN_, ST_>();
    TCT_VARIANTS(TCT_CASE)
#undef TCT_CASE
    return -1;
}

int variant_split_ok(int cta_group, int tile_n, int stages)
{
#define TCT_CASE(CG_, BN_, ST_) \
    if (cta_group == CG_ && tile_n == BN_ && stages == ST_) return Cfg<CG_, BN_, ST_>::SPLIT_OK ? 1 : 0;
    TCT_VARIANTS(TCT_CASE)
#undef TCT_CASE
    return 0;
}

int variant_exists(int layout, int cta_group, int tile_n, int stages)
{
    if (layout == 0) {
#define TCT_CASE(CG_, BN_, ST_) \
        if (cta_group == CG_ && tile_n == BN_ && stages == ST_) return 1;
        TCT_VARIANTS(TCT_CASE)
#undef TCT_CASE
        return 0;
    }
    if (layout < 0 || layout > 7) return 0;
#define TCT_CASE(CG_, BN_, ST_) \
    if (cta_group == CG_ && tile_n == BN_ && stages == ST_) return 1;
    TCT_VARIANTS_EX(TCT_CASE)
#undef TCT_CASE
    return 0;
}

#endif  // TCT_PART == 0

template <bool AT, bool BT, bool BF16>
static cudaError_t launch_layout(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tp,
                                 const CUtensorMap &tc, const KernelParams &p, int cta_group, int tile_n, int stages,
                                 int grid, cudaStream_t stream)
{
#define TCT_CASE(CG_, BN_, ST_)                             \
    if (cta_group == CG_ && tile_n == BN_ && stages == ST_) \
        return launch_variant<CG_, BN_, ST_, AT, BT, BF16>(ta, tb, tp, tc, p, grid, stream);
    if constexpr (!AT && !BT && !BF16) {
        TCT_VARIANTS(TCT_CASE)
    } else {
        TCT_VARIANTS_EX(TCT_CASE)
    }
#undef TCT_CASE
    return cudaErrorInvalidValue;
}

#if TCT_PART == 1
cudaError_t launch_gemm_part1(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tp,
                              const CUtensorMap &tc, const KernelParams &p, int layout, int cta_group, int tile_n,
                              int stages, int grid, cudaStream_t stream)
{
    switch (layout) {
    case 3: return launch_layout<true, true, false>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    case 4: return launch_layout<false, false, true>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    case 5: return launch_layout<true, false, true>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    case 6: return launch_layout<false, true, true>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    case 7: return launch_layout<true, true, true>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_and_clear_error_part1(unsigned *out)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_error_word, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned));
}
#else
cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tp, const CUtensorMap &tc,
                        const KernelParams &p, int layout, int cta_group, int tile_n, int stages, int grid,
                        cudaStream_t stream)
{
    switch (layout) {
    case 0: return launch_layout<false, false, false>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    case 1: return launch_layout<true, false, false>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    case 2: return launch_layout<false, true, false>(ta, tb, tp, tc, p, cta_group, tile_n, stages, grid, stream);
    default: return launch_gemm_part1(ta, tb, tp, tc, p, layout, cta_group, tile_n, stages, grid, stream);
    }
}

cudaError_t launch_copy_rows(const RowCopy &m0, const RowCopy &m1, cudaStream_t stream, int num_sms)
{
    auto job = [](const RowCopy &m) {
        const int64_t bytes = m.cols * m.esz;
        return CopyJob{static_cast<const uint8_t *>(m.src), m.ld_src * m.esz, static_cast<uint8_t *>(m.dst),
                       m.ld_dst * m.esz, m.src ? m.rows : 0, bytes, m.esz, bytes / 16 + 1};
    };
    if ((m0.src && m0.esz != 2 && m0.esz != 4) || (m1.src && m1.esz != 2 && m1.esz != 4)) return cudaErrorInvalidValue;
    const CopyJob j0 = job(m0);
    const CopyJob j1 = job(m1);
    const int64_t total = j0.rows * j0.units_max + j1.rows * j1.units_max;
    if (total <= 0) return cudaSuccess;
    // enough threads for one unit each, up to 16 blocks of 256 per SM (the grid strides beyond)
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 152) * 16;
    const int64_t blocks = std::min<int64_t>((total + kCopyThreads - 1) / kCopyThreads, cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, copy_rows, j0, j1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_pack2(const void *src0, int64_t ld_src0, void *dst0, int64_t ld_dst0, int64_t rows0, int64_t cols0,
                         const void *src1, int64_t ld_src1, void *dst1, int64_t ld_dst1, int64_t rows1, int64_t cols1,
                         cudaStream_t stream)
{
    return launch_copy_rows(RowCopy{src0, ld_src0, dst0, ld_dst0, rows0, cols0, 2},
                            RowCopy{src1, ld_src1, dst1, ld_dst1, rows1, cols1, 2}, stream, 0);
}

cudaError_t launch_fill_epilogue(const KernelParams &p, int num_sms, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(p.M) * ((static_cast<int64_t>(p.N) + 3) / 4);
    if (total <= 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    fill_epilogue<<<static_cast<int>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t error_word_address(unsigned **out)
{
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_error_word);
    *out = static_cast<unsigned *>(ptr);
    return e;
}

cudaError_t read_and_clear_error(unsigned *out)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(out, g_error_word, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    unsigned other = 0;  // the word of the other object's kernels: the first error recorded wins
    e = read_and_clear_error_part1(&other);
    if (e == cudaSuccess && *out == 0) *out = other;
    return e;
}
#endif  // TCT_PART

}  // namespace tct
