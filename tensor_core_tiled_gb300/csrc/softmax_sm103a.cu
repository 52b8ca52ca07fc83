// softmax_sm103a.cu -- fused row softmax, the second workload of the lecture pages
// ("06_triton_style.py", demo 3: one program reads a row once, keeps it on chip, and writes
// exp(x - max) / sum once -- MN reads and MN writes instead of the 5MN + 2M / 3MN + 2M of
// five separate kernels).  Bandwidth-bound: each input element is read once and each output
// written once, except rows too long for on-chip staging, which are read twice.
//
// Rows whose base and leading dimensions are 16-byte aligned take the staged kernels: a
// producer warp streams rows from HBM into a ring of shared-memory slots with bulk
// asynchronous copies (cp.async.bulk, completion counted on an mbarrier per slot), so that
// tens of kilobytes per SM are in flight with no registers held for them, while eight
// compute warps reduce the staged rows and write the result with 16-byte streaming stores.
//   * N <= 1024: a slot holds several rows; one compute warp per row.
//   * N <= 12288: a slot holds one row (or a 16 KB piece of it); the eight warps share it.
//   * longer rows: a cluster of CTAs splits each row (up to 8 CTAs with 8192-column slices in
//     registers, then up to 16 CTAs with slices of about 20480 columns in shared memory);
//     every CTA reduces its slice to (max, sum), sends the pair to every CTA of the cluster
//     through distributed shared memory (st.async, counted on the receiver's mbarrier), and
//     rescales its slice by exp(max_slice - max_row) / sum_row.
// The team kernels launch as programmatic dependent launches: their barrier set-up may
// overlap the previous kernel on the stream, and X and Y are touched only after waiting for it.
// Rows whose 16 slices each exceed the 112 KB ring are streamed twice by the same cluster
// kernel.  Other layouts take the plain kernels below: a warp per row held in registers, a
// CTA per row staged in shared memory, or two passes over the row.
// exp(-inf) = 0; a row holding a NaN, whose maximum is +inf, or that is all -inf has no
// finite softmax and is written as NaN.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "gemm_internal.h"
#include "ptx_sm103a.cuh"

namespace tct {

namespace {

__host__ __device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kWarpMaxVec = 16;  // float4 per lane in the warp-per-row kernel
constexpr int64_t kSmemMaxCols = 51200;

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_any(int v) { return __any_sync(0xffffffffu, v); }

// Block-wide reductions for kThreads threads (red: kWarps floats of shared memory).
__device__ __forceinline__ float block_max(float v, float *red)
{
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    v = l < kWarps ? red[l] : -INFINITY;
    return warp_max(v);
}

__device__ __forceinline__ float block_sum(float v, float *red)
{
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    v = l < kWarps ? red[l] : 0.0f;
    return warp_sum(v);
}

__device__ __forceinline__ int block_any(int v, int *red)
{
    v = warp_any(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    v = l < kWarps ? red[l] : 0;
    return warp_any(v);
}

// A row's maximum is usable when finite and no element was NaN.
__device__ __forceinline__ bool row_ok(float m, int has_nan) { return !has_nan && isfinite(m); }

template <int VEC>
__global__ void __launch_bounds__(kThreads) softmax_warp_rows(const float *X, float *Y,
                                                              int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                                                              int vec)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarps;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); row < M; row += warps) {
        const float *x = X + row * ldx;
        float v[VEC][4];
        float m = -INFINITY;
        int nan = 0;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const int64_t c = (static_cast<int64_t>(i) * 32 + lane) * 4;
            if (vec && c + 3 < N) {
                const float4 t = __ldcs(reinterpret_cast<const float4 *>(x + c));
                v[i][0] = t.x, v[i][1] = t.y, v[i][2] = t.z, v[i][3] = t.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[i][e] = c + e < N ? __ldcs(x + c + e) : -INFINITY;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                nan |= isnan(v[i][e]);
                m = fmaxf(m, v[i][e]);
            }
        }
        m = warp_max(m);
        nan = warp_any(nan);
        const bool ok = row_ok(m, nan);
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < VEC; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[i][e] = expf(v[i][e] - m);  // padding: exp(-inf) = 0
                s += v[i][e];
            }
        s = warp_sum(s);
        float *y = Y + row * ldy;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const int64_t c = (static_cast<int64_t>(i) * 32 + lane) * 4;
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = ok ? v[i][e] / s : NAN;
            if (vec && c + 3 < N) {
                __stcs(reinterpret_cast<float4 *>(y + c), make_float4(o[0], o[1], o[2], o[3]));
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (c + e < N) __stcs(y + c + e, o[e]);
            }
        }
    }
}

// One CTA per row, the row kept in shared memory (N <= kSmemMaxCols).
__global__ void __launch_bounds__(kThreads) softmax_smem_rows(const float *X, float *Y,
                                                              int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                                                              int vec)
{
    extern __shared__ float srow[];
    __shared__ float redf[kWarps];
    __shared__ int redi[kWarps];
    const int64_t n4 = vec ? N / 4 : 0;  // float4 chunks handled vectorised
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const float *x = X + row * ldx;
        float m = -INFINITY;
        int nan = 0;
        for (int64_t c = threadIdx.x; c < n4; c += kThreads) {
            const float4 t = __ldcs(reinterpret_cast<const float4 *>(x) + c);
            reinterpret_cast<float4 *>(srow)[c] = t;
            nan |= isnan(t.x) | isnan(t.y) | isnan(t.z) | isnan(t.w);
            m = fmaxf(fmaxf(m, fmaxf(t.x, t.y)), fmaxf(t.z, t.w));
        }
        for (int64_t c = n4 * 4 + threadIdx.x; c < N; c += kThreads) {
            const float t = __ldcs(x + c);
            srow[c] = t;
            nan |= isnan(t);
            m = fmaxf(m, t);
        }
        m = block_max(m, redf);
        nan = block_any(nan, redi);
        const bool ok = row_ok(m, nan);
        float s = 0.0f;
        for (int64_t c = threadIdx.x; c < N; c += kThreads) {
            const float e = expf(srow[c] - m);
            srow[c] = e;
            s += e;
        }
        s = block_sum(s, redf);
        float *y = Y + row * ldy;
        for (int64_t c = threadIdx.x; c < n4; c += kThreads) {
            const float4 e = reinterpret_cast<const float4 *>(srow)[c];
            const float4 o = ok ? make_float4(e.x / s, e.y / s, e.z / s, e.w / s) : make_float4(NAN, NAN, NAN, NAN);
            __stcs(reinterpret_cast<float4 *>(y) + c, o);
        }
        for (int64_t c = n4 * 4 + threadIdx.x; c < N; c += kThreads) __stcs(y + c, ok ? srow[c] / s : NAN);
        __syncthreads();  // srow is reused by the next row
    }
}

// One CTA per row, two passes over the row: an online (max, sum), then the output.
__global__ void __launch_bounds__(kThreads) softmax_online_rows(const float *X, float *Y,
                                                                int64_t M, int64_t N, int64_t ldx, int64_t ldy)
{
    __shared__ float redf[kWarps];
    __shared__ float redg[kWarps];
    __shared__ int redi[kWarps];
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const float *x = X + row * ldx;
        float m = -INFINITY, s = 0.0f;
        int nan = 0;
        for (int64_t c = threadIdx.x; c < N; c += kThreads) {
            const float t = x[c];
            nan |= isnan(t);
            if (t == -INFINITY) continue;  // contributes exp(-inf) = 0
            if (t > m) {
                s = s * expf(m - t) + 1.0f;  // rescale the running sum to the new maximum
                m = t;
            } else {
                s += expf(t - m);
            }
        }
        // combine (m, s) over the block: every partial sum rescaled to the row maximum
        const float mb = block_max(m, redf);
        nan = block_any(nan, redi);
        const float part = (m == -INFINITY) ? 0.0f : s * expf(m - mb);
        const float sb = block_sum(part, redg);
        const bool ok = row_ok(mb, nan);
        float *y = Y + row * ldy;
        for (int64_t c = threadIdx.x; c < N; c += kThreads) __stcs(y + c, ok ? expf(x[c] - mb) / sb : NAN);
        __syncthreads();
    }
}


// ---------------------------------------------------------------- staged kernels

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kStagedThreads = kComputeThreads + 32;  // + one producer warp
constexpr int kMaxRing = 32;                          // ring slots (one mbarrier pair each)
constexpr uint32_t kRingBytes = 32 * 1024;            // staging ring per CTA (at least two slots)
constexpr uint32_t kMaxSmemBytes = 200 * 1024;        // dynamic shared memory opt-in of the staged kernels
// Ring of the long-slice cluster kernel: 7 slots, so that a slice of up to 5 slots leaves 2
// for the next row's first chunks (measured on GB300 against 6 slots: 131072-column rows
// 0.75 -> 0.78 of the copy bandwidth, 262144 columns 0.62 -> 0.64; two CTAs still fit per SM).
constexpr uint32_t kLongRingBytes = 112 * 1024;
constexpr int kCtasPerSm = 2;
constexpr uint32_t kHeaderBytes = 1024;               // barriers and reduction scratch
constexpr uint32_t kChunkBytes = 16 * 1024;           // slot size of the CTA kernel for long slices
constexpr int kMaxCluster = 16;

enum SoftmaxWaitSite : unsigned {
    SITE_SM_EMPTY = 16,  // producer waiting for a free slot
    SITE_SM_FULL = 17,   // compute warps waiting for a slot's copy
    SITE_SM_XCHG = 18,   // waiting for the cluster's (max, sum) pairs
    SITE_SM_DRAIN = 19,  // producer waiting for its last copies before exit
};

struct StagedParams {
    const float *X;
    float *Y;
    int64_t M, N, ldx, ldy;
    int64_t slice;          // CTA kernel: columns per cluster rank (multiple of 4)
    int64_t tiles;          // warp kernel: tiles of rows_per_tile rows; CTA kernel: rows
    int32_t rows_per_tile;  // warp kernel
    int32_t ring;           // ring slots in use (<= kMaxRing)
    uint32_t slot_bytes;    // warp kernel: bytes per staged row; CTA kernel: bytes per slot
    int32_t contiguous;     // warp kernel: rows adjacent (ldx == N, N % 4 == 0), one copy per tile
    unsigned *err;
    uint64_t timeout_ns;
};

struct StagedShared {
    uint64_t full[kMaxRing];
    uint64_t empty[kMaxRing];
    uint64_t xchg[2];
    float2 pairs[2][kMaxCluster];  // (slice max, slice sum) of every rank, two rows in turn
    float redm[kComputeWarps];
    float reds[kComputeWarps];
    int abort_flag;
};
static_assert(sizeof(StagedShared) <= kHeaderBytes, "staged kernel header");

__device__ __forceinline__ void staged_timeout(StagedShared &sh, const StagedParams &p, unsigned site)
{
    atomicCAS(p.err, 0u, GEMM_ERR_DEVICE_TIMEOUT_CODE | (site << 8));
    *reinterpret_cast<volatile int *>(&sh.abort_flag) = 1;
    __threadfence_block();
}

// Bounded wait on an mbarrier phase; gives up at the time limit or as soon as another warp
// of this CTA has given up.  On false the caller carries on without waiting again (the
// results are then undefined and the error word says why), so that every warp still
// reaches every barrier of the CTA and the kernel ends.
template <bool kClusterScope>
__device__ __forceinline__ bool staged_wait(uint32_t bar, uint32_t parity, StagedShared &sh, const StagedParams &p,
                                            unsigned site)
{
    auto ready = [&]() { return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (ready()) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spins = 1;; ++spins) {
        if (ready()) return true;
        if ((spins & 15u) == 0u) {
            if (*reinterpret_cast<volatile int *>(&sh.abort_flag)) return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                staged_timeout(sh, p, site);
                return false;
            }
        }
    }
}

// Producer epilogue: waits (bounded, even after an abort) until the copies into the last
// min(issued, ring) slots have landed, so that no copy targets the CTA after it exits.
__device__ __forceinline__ void staged_drain(StagedShared &sh, const StagedParams &p, uint32_t issued)
{
    const uint32_t first = issued > static_cast<uint32_t>(p.ring) ? issued - p.ring : 0u;
    for (uint32_t j = first; j < issued; ++j) {
        const uint32_t s = j % p.ring;
        if (!mbar_wait(smem_u32(&sh.full[s]), (j / p.ring) & 1u, p.timeout_ns)) {
            staged_timeout(sh, p, SITE_SM_DRAIN);
            return;
        }
    }
}

__device__ __forceinline__ void staged_init(StagedShared &sh, const StagedParams &p)
{
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.ring; ++i) {
            mbar_init(smem_u32(&sh.full[i]), 1);
            mbar_init(smem_u32(&sh.empty[i]), kComputeWarps);
        }
        mbar_init(smem_u32(&sh.xchg[0]), 1);
        mbar_init(smem_u32(&sh.xchg[1]), 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
}

__device__ __forceinline__ float max4(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }
// e^d computed as 2^(d log2 e) with the hardware base-2 exponential (ex2.approx: relative
// error about 2^-22 in the result; subnormal results kept).  Rounding d log2 e adds a relative
// error of about |d| u to the result (u = 2^-24), the same order as rounding d = x - max itself.
__device__ __forceinline__ float exp_of(float d)
{
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(d * 1.44269504088896341f));
    return r;
}

// Reductions over a team of TT threads (TT = 8, 16, 32 lanes of one warp, or 2-8 whole
// warps).  Within a warp, xor-shuffles over aligned groups of min(TT, 32) lanes; across the
// warps of a team, each warp publishes its partial in slot `warp` of `red` and, after the
// team's named barrier (1 + team), every lane combines the partials in warp order.
template <int TT>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = (TT < 32 ? TT : 32) / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int TT>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = (TT < 32 ? TT : 32) / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int TT>
__device__ __forceinline__ float team_reduce_max(float m, StagedShared &sh, int team, int warp, int lane)
{
    m = group_max<TT>(m);
    if constexpr (TT > 32) {
        constexpr int T = TT / 32;
        if (lane == 0) sh.redm[warp] = m;
        named_bar_sync(1 + team, TT);
        m = sh.redm[team * T];
#pragma unroll
        for (int w = 1; w < T; ++w) m = fmaxf(m, sh.redm[team * T + w]);
    }
    return m;
}

template <int TT>
__device__ __forceinline__ float team_reduce_sum(float v, StagedShared &sh, int team, int warp, int lane)
{
    v = group_sum<TT>(v);
    if constexpr (TT > 32) {
        constexpr int T = TT / 32;
        if (lane == 0) sh.reds[warp] = v;
        named_bar_sync(1 + team, TT);
        v = sh.reds[team * T];
#pragma unroll
        for (int w = 1; w < T; ++w) v += sh.reds[team * T + w];
    }
    return v;
}

// Scale for a slice whose terms are exp(x - m) (m the slice maximum), given every slice's
// (maximum, sum) pair: exp(m - M) / S with M the row maximum and S the row sum rescaled to
// it.  A NaN sum (the slice held a NaN, or a +inf maximum) or a row with no finite maximum
// gives NaN; a slice that is all -inf gets 0.
__device__ __forceinline__ float slice_scale(const float2 *pairs, uint32_t csize, float m)
{
    float M = -INFINITY;
    for (uint32_t c = 0; c < csize; ++c) M = fmaxf(M, pairs[c].x);
    float S = 0.0f;
    for (uint32_t c = 0; c < csize; ++c) {
        const float2 pr = pairs[c];
        S += pr.y * (pr.x == -INFINITY ? 0.0f : expf(pr.x - M));  // NaN * 0 stays NaN
    }
    if (!isfinite(M)) return NAN;
    return (m == -INFINITY ? 0.0f : expf(m - M)) / S;
}

// Rows (or, in a cluster, row slices) of at most TT * VEC * 4 columns.  The 256 compute
// threads form 256 / TT teams of TT threads; a ring slot holds a tile of rows_per_tile staged
// rows (a multiple of the team count), and team k takes rows k, k + teams, ... of each tile.
// A team reads its row from shared memory into registers once (VEC float4 per thread),
// releases the slot after its last row of the tile, and computes and stores the softmax from
// registers.  Every warp runs the same number of row iterations, so that shuffles always
// have all 32 lanes; a team past the end of the tile runs on -inf fill and stores nothing.
template <int TT, int VEC, bool kCluster>
__global__ void __launch_bounds__(kStagedThreads, kCtasPerSm) softmax_team(const StagedParams p)
{
    constexpr int kTeams = kComputeThreads / TT;
    constexpr int kTeamsPerWarp = TT < 32 ? 32 / TT : 1;
    static_assert(TT == 8 || TT == 16 || TT == 32 || TT == 64 || TT == 128 || TT == 256, "team size");
    static_assert(!kCluster || TT == kComputeThreads, "a cluster row slice is reduced by the whole CTA");
    extern __shared__ __align__(1024) unsigned char smem[];
    StagedShared &sh = *reinterpret_cast<StagedShared *>(smem);
    unsigned char *ring = smem + kHeaderBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    staged_init(sh, p);
    if constexpr (kCluster) cluster_sync_all();  // every CTA's barriers exist before any st.async
    griddep_wait();  // the set-up above touched no global memory; X and Y wait for the previous grid
    const uint32_t rank = kCluster ? cluster_ctarank() : 0u;
    const uint32_t csize = kCluster ? cluster_nctarank() : 1u;
    const int64_t cid = kCluster ? static_cast<int64_t>(cluster_id_x()) : static_cast<int64_t>(blockIdx.x);
    const int64_t ncl = kCluster ? static_cast<int64_t>(cluster_count_x()) : static_cast<int64_t>(gridDim.x);
    const int64_t c0 = static_cast<int64_t>(rank) * p.slice;
    const int64_t len = p.N - c0 > 0 ? lmin(p.slice, p.N - c0) : int64_t(0);
    const int64_t nb = len & ~int64_t(3);
    const int n4 = static_cast<int>(nb >> 2);
    const int64_t R = p.rows_per_tile;
    const uint32_t tile_bytes = static_cast<uint32_t>(R) * p.slot_bytes;

    if (warp == kComputeWarps) {  // producer warp
        uint32_t q = 0;
        for (int64_t t = cid; t < p.tiles; t += ncl, ++q) {
            const uint32_t s = q % p.ring, ph = (q / p.ring) & 1u;
            const int64_t r0 = t * R;
            const int rows = static_cast<int>(lmin(R, p.M - r0));
            bool ok = true;
            if (lane == 0) ok = staged_wait<false>(smem_u32(&sh.empty[s]), ph ^ 1u, sh, p, SITE_SM_EMPTY);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            const uint32_t full = smem_u32(&sh.full[s]);
            const uint32_t dst = smem_u32(ring) + s * tile_bytes;
            if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(rows * nb * 4));
            __syncwarp();
            if (nb > 0) {
                if (p.contiguous) {
                    if (lane == 0) bulk_load(dst, p.X + r0 * p.ldx, static_cast<uint32_t>(rows * nb * 4), full);
                } else {
                    for (int r = lane; r < rows; r += 32)
                        bulk_load(dst + r * p.slot_bytes, p.X + (r0 + r) * p.ldx + c0, static_cast<uint32_t>(nb * 4),
                                  full);
                }
            }
        }
        if (lane == 0) {
            griddep_launch_dependents();  // every row requested: the next grid may start launching
            staged_drain(sh, p, q);
        }
    } else {
        const int team = threadIdx.x / TT;
        const int tt = threadIdx.x % TT;                    // thread index within the team
        const int warp_team0 = warp * kTeamsPerWarp;        // first team of this warp (TT <= 32)
        const int lead = TT <= 32 ? warp_team0 : team;      // team whose rows pace this warp's loop
        const bool has_tail = tt < len - nb;                // columns nb .. len-1 (at most 3): global loads
        uint32_t q = 0, row_ctr = 0;
        for (int64_t t = cid; t < p.tiles; t += ncl, ++q) {
            const uint32_t s = q % p.ring, ph = (q / p.ring) & 1u;
            const int64_t r0 = t * R;
            const int rows = static_cast<int>(lmin(R, p.M - r0));
            staged_wait<false>(smem_u32(&sh.full[s]), ph, sh, p, SITE_SM_FULL);
            const unsigned char *tile = ring + static_cast<size_t>(s) * tile_bytes;
            if (lead >= rows) {  // nothing for this warp in a short last tile
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
            }
            for (int base = 0; lead + base < rows; base += kTeams, ++row_ctr) {
                const int r = team + base;
                const bool live = r < rows;
                const float *xg = p.X + (r0 + r) * p.ldx + c0;
                float *yg = p.Y + (r0 + r) * p.ldy + c0;
                const float4 *x4 = reinterpret_cast<const float4 *>(tile + static_cast<size_t>(r) * p.slot_bytes);
                float4 v[VEC];
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    const int i = tt + k * TT;
                    v[k] = live && i < n4 ? x4[i] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
                if (lead + base + kTeams >= rows) {  // the warp's last rows of this tile are in registers
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
                }
                const float tv = live && has_tail ? xg[nb + tt] : -INFINITY;
                float m = tv;
#pragma unroll
                for (int k = 0; k < VEC; ++k) m = fmaxf(m, max4(v[k]));
                m = team_reduce_max<TT>(m, sh, team, warp, lane);
                // A NaN entry, a +inf maximum or an all -inf row makes a term NaN, hence the sum
                // and every output of the row.  A cluster slice that is all -inf sums to 0.
                const float mu = (kCluster && m == -INFINITY) ? 0.0f : m;
                float sum = 0.0f;
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    float4 &e = v[k];
                    e.x = exp_of(e.x - mu), e.y = exp_of(e.y - mu), e.z = exp_of(e.z - mu), e.w = exp_of(e.w - mu);
                    sum += (e.x + e.y) + (e.z + e.w);
                }
                const float te = exp_of(tv - mu);
                sum = team_reduce_sum<TT>(sum + te, sh, team, warp, lane);

                float f;
                if constexpr (kCluster) {
                    const uint32_t j = row_ctr & 1u;
                    const uint32_t xbar = smem_u32(&sh.xchg[j]);
                    if (tt == 0) {
                        mbar_arrive_expect_tx(xbar, csize * 8u);
                        const uint32_t slot = smem_u32(&sh.pairs[j][rank]);
                        for (uint32_t c = 0; c < csize; ++c)
                            st_async_f32x2(map_to_cta(slot, c), m, sum, map_to_cta(xbar, c));
                    }
                    staged_wait<true>(xbar, (row_ctr >> 1) & 1u, sh, p, SITE_SM_XCHG);
                    f = slice_scale(sh.pairs[j], csize, m);
                } else {
                    f = __frcp_rn(sum);
                }
                if (live) {
                    float4 *y4 = reinterpret_cast<float4 *>(yg);
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        const int i = tt + k * TT;
                        if (i < n4) __stcs(y4 + i, make_float4(v[k].x * f, v[k].y * f, v[k].z * f, v[k].w * f));
                    }
                    if (has_tail) __stcs(yg + nb + tt, te * f);
                }
            }
        }
    }
    if constexpr (kCluster) cluster_sync_all();  // no CTA leaves while a peer may still write to it
}

// Rows longer than 8 * 8192 columns: a cluster of up to 16 CTAs per row, rank r owning columns
// [r * slice, min(N, (r + 1) * slice)), streamed through a ring of 16 KB slots.  When the
// slice fits in the ring (resident mode) it is read once: the (max, sum) pass writes
// exp(x - max) back into the slots and the output pass scales them.  Otherwise (streaming
// mode) the slice is read twice: an online pass keeps a running (max, sum) per thread,
// rescaling the sum whenever its maximum grows, and the output pass recomputes
// exp(x - row max) from the second read.
__global__ void __launch_bounds__(kStagedThreads, kCtasPerSm) softmax_long_slices(const StagedParams p)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    StagedShared &sh = *reinterpret_cast<StagedShared *>(smem);
    unsigned char *ring = smem + kHeaderBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    staged_init(sh, p);
    cluster_sync_all();  // every CTA's barriers exist before any st.async
    const uint32_t rank = cluster_ctarank();
    const uint32_t csize = cluster_nctarank();
    const int64_t cid = cluster_id_x();
    const int64_t ncl = cluster_count_x();
    const int64_t c0 = static_cast<int64_t>(rank) * p.slice;
    const int64_t len = p.N - c0 > 0 ? lmin(p.slice, p.N - c0) : int64_t(0);
    const int64_t nb = len & ~int64_t(3);
    const int64_t n4 = nb >> 2;
    const uint32_t slot_f4 = p.slot_bytes / 16;
    const uint32_t nch = static_cast<uint32_t>((n4 + slot_f4 - 1) / slot_f4);
    const bool resident = nch <= static_cast<uint32_t>(p.ring);
    const uint32_t loads_per_row = resident ? nch : 2 * nch;
    auto chunk_f4 = [&](uint32_t c) { return static_cast<uint32_t>(lmin(slot_f4, n4 - int64_t(c) * slot_f4)); };
    auto slot_ptr = [&](uint32_t j) { return ring + static_cast<size_t>(j % p.ring) * p.slot_bytes; };
    auto wait_full = [&](uint32_t j) { staged_wait<false>(smem_u32(&sh.full[j % p.ring]), (j / p.ring) & 1u, sh, p, SITE_SM_FULL); };
    auto release = [&](uint32_t j) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.empty[j % p.ring]));
    };

    if (warp == kComputeWarps) {  // producer (one lane): the slice once, or twice when streaming
        if (lane == 0) {
            uint32_t q = 0;
            bool ok = true;
            for (int64_t t = cid; ok && t < p.tiles; t += ncl) {
                const float *src = p.X + t * p.ldx + c0;
                for (uint32_t k = 0; k < loads_per_row; ++k, ++q) {
                    const uint32_t c = k < nch ? k : k - nch;
                    const uint32_t s = q % p.ring, ph = (q / p.ring) & 1u;
                    if (!staged_wait<false>(smem_u32(&sh.empty[s]), ph ^ 1u, sh, p, SITE_SM_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t f4 = chunk_f4(c);
                    const uint32_t full = smem_u32(&sh.full[s]);
                    mbar_arrive_expect_tx(full, f4 * 16);
                    bulk_load(smem_u32(ring) + s * p.slot_bytes, src + static_cast<int64_t>(c) * slot_f4 * 4, f4 * 16,
                              full);
                }
            }
            staged_drain(sh, p, q);
        }
    } else {
        const int tid = threadIdx.x;
        uint32_t q = 0, row_ctr = 0;
        for (int64_t t = cid; t < p.tiles; t += ncl, ++row_ctr, q += loads_per_row) {
            const float *xg = p.X + t * p.ldx + c0;
            float *yg = p.Y + t * p.ldy + c0;
            const bool has_tail = tid < len - nb;
            const float tv = has_tail ? xg[nb + tid] : -INFINITY;
            float m = tv, sum = 0.0f;
            if (resident) {
                for (uint32_t c = 0; c < nch; ++c) {
                    wait_full(q + c);
                    const float4 *x4 = reinterpret_cast<const float4 *>(slot_ptr(q + c));
                    const uint32_t f4 = chunk_f4(c);
#pragma unroll 4
                    for (uint32_t i = tid; i < f4; i += kComputeThreads) m = fmaxf(m, max4(x4[i]));
                }
                m = team_reduce_max<kComputeThreads>(m, sh, 0, warp, lane);
                const float mu = m == -INFINITY ? 0.0f : m;  // an all -inf slice sums to 0
                for (uint32_t c = 0; c < nch; ++c) {
                    float4 *x4 = reinterpret_cast<float4 *>(slot_ptr(q + c));
                    const uint32_t f4 = chunk_f4(c);
#pragma unroll 4
                    for (uint32_t i = tid; i < f4; i += kComputeThreads) {
                        float4 v = x4[i];
                        v.x = exp_of(v.x - mu), v.y = exp_of(v.y - mu), v.z = exp_of(v.z - mu), v.w = exp_of(v.w - mu);
                        x4[i] = v;
                        sum += (v.x + v.y) + (v.z + v.w);
                    }
                }
                fence_proxy_async_smem();  // the slots are refilled by bulk copies after release
                sum = team_reduce_sum<kComputeThreads>(sum + exp_of(tv - mu), sh, 0, warp, lane);
            } else {
                // online pass: running (m, sum) per thread, sum relative to m (to 0 while m is -inf)
                sum = exp_of(tv - (m == -INFINITY ? 0.0f : m));
                for (uint32_t c = 0; c < nch; ++c) {
                    wait_full(q + c);
                    const float4 *x4 = reinterpret_cast<const float4 *>(slot_ptr(q + c));
                    const uint32_t f4 = chunk_f4(c);
#pragma unroll 2
                    for (uint32_t i = tid; i < f4; i += kComputeThreads) {
                        const float4 v = x4[i];
                        const float mv = max4(v);
                        if (mv > m) {
                            sum *= m == -INFINITY ? 0.0f : expf(m - mv);  // NaN * 0 stays NaN
                            m = mv;
                        }
                        const float mu = m == -INFINITY ? 0.0f : m;
                        sum += (exp_of(v.x - mu) + exp_of(v.y - mu)) + (exp_of(v.z - mu) + exp_of(v.w - mu));
                    }
                    release(q + c);
                }
                const float mt = m;
                m = team_reduce_max<kComputeThreads>(m, sh, 0, warp, lane);
                sum *= (mt == -INFINITY || m == -INFINITY) ? 1.0f : expf(mt - m);  // to the slice maximum
                sum = team_reduce_sum<kComputeThreads>(sum, sh, 0, warp, lane);
            }

            // (max, sum) of every slice of the row, from every rank of the cluster
            const uint32_t j = row_ctr & 1u;
            const uint32_t xbar = smem_u32(&sh.xchg[j]);
            if (tid == 0) {
                mbar_arrive_expect_tx(xbar, csize * 8u);
                const uint32_t slot = smem_u32(&sh.pairs[j][rank]);
                for (uint32_t r = 0; r < csize; ++r) st_async_f32x2(map_to_cta(slot, r), m, sum, map_to_cta(xbar, r));
            }
            staged_wait<true>(xbar, (row_ctr >> 1) & 1u, sh, p, SITE_SM_XCHG);
            const float f = slice_scale(sh.pairs[j], csize, m);

            float4 *y4 = reinterpret_cast<float4 *>(yg);
            if (resident) {
                for (uint32_t c = 0; c < nch; ++c) {
                    const float4 *x4 = reinterpret_cast<const float4 *>(slot_ptr(q + c));
                    const uint32_t f4 = chunk_f4(c);
                    float4 *yc = y4 + static_cast<int64_t>(c) * slot_f4;
#pragma unroll 4
                    for (uint32_t i = tid; i < f4; i += kComputeThreads) {
                        float4 v = x4[i];
                        v.x *= f, v.y *= f, v.z *= f, v.w *= f;
                        __stcs(yc + i, v);
                    }
                    release(q + c);
                }
                if (has_tail) __stcs(yg + nb + tid, exp_of(tv - (m == -INFINITY ? 0.0f : m)) * f);
            } else {
                // second read: exp(x - m) * f with m the slice maximum, as in resident mode
                const float mu = m == -INFINITY ? 0.0f : m;
                for (uint32_t c = 0; c < nch; ++c) {
                    wait_full(q + nch + c);
                    const float4 *x4 = reinterpret_cast<const float4 *>(slot_ptr(q + nch + c));
                    const uint32_t f4 = chunk_f4(c);
                    float4 *yc = y4 + static_cast<int64_t>(c) * slot_f4;
#pragma unroll 2
                    for (uint32_t i = tid; i < f4; i += kComputeThreads) {
                        const float4 v = x4[i];
                        __stcs(yc + i, make_float4(exp_of(v.x - mu) * f, exp_of(v.y - mu) * f, exp_of(v.z - mu) * f,
                                                   exp_of(v.w - mu) * f));
                    }
                    release(q + nch + c);
                }
                if (has_tail) __stcs(yg + nb + tid, exp_of(tv - mu) * f);
            }
        }
    }
    cluster_sync_all();  // no CTA leaves while a peer may still write to it
}

}  // namespace

namespace {

// Per-device launch state: the staged kernels' shared-memory opt-in, and how many clusters
// of each size fit on the device at once.
struct SoftmaxDevState {
    bool smem_set = false;
    int clusters[2][kMaxCluster + 1] = {};  // [team, long][size]: 0 = not queried, -1 = does not fit
};
constexpr int kMaxDevices = 64;
std::mutex g_sm_mu;
SoftmaxDevState g_sm_dev[kMaxDevices];

using StagedKernel = void (*)(StagedParams);

// Team kernels by row length: (threads per team, float4 per thread) covering up to
// TT * VEC * 4 columns.  Teams grow with the row so that a tile (one row per team) stays
// near 16 KB: a shallow ring of small tiles streams faster than a deep one.
struct TeamVariant {
    int64_t max_cols;
    int team_threads;
    StagedKernel kernel;
};
const TeamVariant kTeamVariants[] = {
    {32, 8, softmax_team<8, 1, false>},       {64, 8, softmax_team<8, 2, false>},
    {128, 8, softmax_team<8, 4, false>},      {256, 16, softmax_team<16, 4, false>},
    {512, 32, softmax_team<32, 4, false>},    {1024, 64, softmax_team<64, 4, false>},
    {2048, 128, softmax_team<128, 4, false>}, {4096, 256, softmax_team<256, 4, false>},
    {8192, 256, softmax_team<256, 8, false>},
};
constexpr int64_t kTeamMaxCols = 8192;  // also the slice length of the cluster team kernel
constexpr int kTeamClusterMax = 8;      // CTAs per row of the cluster team kernel
constexpr int64_t kLongSliceCols = 20480;  // target slice of the long-slice kernel (80 KB)
StagedKernel const kClusterTeam = softmax_team<256, 8, true>;
StagedKernel const kClusterLong = softmax_long_slices;

cudaError_t set_staged_smem()
{
    const int bytes = static_cast<int>(kMaxSmemBytes);
    cudaError_t e = cudaSuccess;
    for (const TeamVariant &v : kTeamVariants)
        if (e == cudaSuccess) e = cudaFuncSetAttribute(v.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    for (StagedKernel k : {kClusterTeam, kClusterLong}) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    return e;
}

// Clusters of `csize` CTAs (smem bytes each) that are co-resident on the current device.
cudaError_t max_clusters(StagedKernel kernel, int csize, size_t smem, int *out)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(csize) * 64u);
    cfg.blockDim = dim3(kStagedThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kernel, &cfg);
}

cudaError_t launch_plain(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy, int num_sms, int vec,
                         cudaStream_t stream)
{
    if (N <= static_cast<int64_t>(kWarpMaxVec) * 128) {
        const int64_t rows_per_block = kWarps;
        int64_t blocks = (M + rows_per_block - 1) / rows_per_block;
        const int64_t cap = static_cast<int64_t>(num_sms) * 8;
        if (blocks > cap) blocks = cap;
        const int nv = static_cast<int>((N + 127) / 128);  // float4 per lane needed
#define TCT_SOFTMAX_WARP(V)                                                                               \
    if (nv <= V) {                                                                                        \
        softmax_warp_rows<V><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(X, Y, M, N, ldx, ldy, vec); \
        return cudaGetLastError();                                                                        \
    }
        TCT_SOFTMAX_WARP(1)
        TCT_SOFTMAX_WARP(2)
        TCT_SOFTMAX_WARP(4)
        TCT_SOFTMAX_WARP(8)
        TCT_SOFTMAX_WARP(16)
#undef TCT_SOFTMAX_WARP
    }
    int64_t blocks = M;
    if (N <= kSmemMaxCols) {
        const size_t smem = static_cast<size_t>(N) * sizeof(float);
        const cudaError_t e =
            cudaFuncSetAttribute(softmax_smem_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_smem_rows, kThreads, smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
        if (blocks > cap) blocks = cap;
        softmax_smem_rows<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(X, Y, M, N, ldx, ldy, vec);
        return cudaGetLastError();
    }
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    softmax_online_rows<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(X, Y, M, N, ldx, ldy);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_rows(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy, int num_sms,
                                unsigned *err, uint64_t timeout_ns, cudaStream_t stream)
{
    if (M <= 0 || N <= 0) return cudaSuccess;
    const int vec = (reinterpret_cast<uintptr_t>(X) % 16 == 0 && reinterpret_cast<uintptr_t>(Y) % 16 == 0 &&
                     ldx % 4 == 0 && ldy % 4 == 0)
                        ? 1
                        : 0;
    if (!vec) return launch_plain(X, Y, M, N, ldx, ldy, num_sms, vec, stream);

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_sm_mu);
    SoftmaxDevState &ds = g_sm_dev[dev];
    if (!ds.smem_set) {
        e = set_staged_smem();
        if (e != cudaSuccess) return e;
        ds.smem_set = true;
    }

    StagedParams p = {};
    p.X = X, p.Y = Y, p.M = M, p.N = N, p.ldx = ldx, p.ldy = ldy;
    p.err = err, p.timeout_ns = timeout_ns;
    // Ring slots hold tiles of R staged rows (slices), R a multiple of the teams per CTA,
    // about 16 KB per tile (at most 128 rows, at least one row per team).
    auto tile_rows = [](uint32_t slot_bytes, int teams) {
        int64_t R = 16384 / slot_bytes;
        R = R > 128 ? 128 : R;
        R = R / teams * teams;
        return R < teams ? int64_t(teams) : R;
    };
    // Slots in the ring: as many tiles as kRingBytes holds, but never fewer than two.
    auto ring_slots = [](uint32_t tile_bytes) {
        const int64_t n = kRingBytes / tile_bytes;
        return static_cast<int32_t>(n < 2 ? 2 : (n > kMaxRing ? kMaxRing : n));
    };
    if (N <= kTeamMaxCols) {
        const TeamVariant *v = kTeamVariants;
        while (v->max_cols < N) ++v;
        p.slice = N;
        p.slot_bytes = static_cast<uint32_t>(((N + 3) & ~int64_t(3)) * 4);
        p.rows_per_tile = static_cast<int32_t>(tile_rows(p.slot_bytes, kComputeThreads / v->team_threads));
        const uint32_t tile_bytes = static_cast<uint32_t>(p.rows_per_tile) * p.slot_bytes;
        p.ring = ring_slots(tile_bytes);
        p.contiguous = (ldx == N && N % 4 == 0) ? 1 : 0;
        p.tiles = (M + p.rows_per_tile - 1) / p.rows_per_tile;
        const size_t smem = kHeaderBytes + static_cast<size_t>(p.ring) * tile_bytes;
        if (smem > kMaxSmemBytes) return cudaErrorInvalidConfiguration;
        const int64_t grid = lmin(p.tiles, static_cast<int64_t>(num_sms) * kCtasPerSm);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kStagedThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // set-up overlaps the previous kernel
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, v->kernel, p);
    }

    // A cluster per row: up to kTeamClusterMax CTAs holding slices of at most kTeamMaxCols
    // columns in registers; longer rows in slices of about kLongSliceCols columns staged in
    // shared memory (at most 5 of the 7 ring slots, so the next row's first slots stream in
    // meanwhile), at most kMaxCluster CTAs.  Measured on GB300: clusters of 7 CTAs stream
    // markedly slower than clusters of 8, so 7 becomes 8.
    const bool team = N <= static_cast<int64_t>(kTeamClusterMax) * kTeamMaxCols;
    int csize = static_cast<int>(team ? (N + kTeamMaxCols - 1) / kTeamMaxCols : (N + kLongSliceCols - 1) / kLongSliceCols);
    if (!team && csize == 7) csize = 8;
    if (csize > kMaxCluster) csize = kMaxCluster;
    p.slice = (((N + csize - 1) / csize) + 3) & ~int64_t(3);
    StagedKernel kernel;
    size_t smem;
    if (team) {
        kernel = kClusterTeam;
        p.slot_bytes = static_cast<uint32_t>(p.slice * 4);
        p.rows_per_tile = static_cast<int32_t>(tile_rows(p.slot_bytes, 1));
        const uint32_t tile_bytes = static_cast<uint32_t>(p.rows_per_tile) * p.slot_bytes;
        p.ring = ring_slots(tile_bytes);
        p.tiles = (M + p.rows_per_tile - 1) / p.rows_per_tile;
        smem = kHeaderBytes + static_cast<size_t>(p.ring) * tile_bytes;
    } else {
        kernel = kClusterLong;
        p.slot_bytes = kChunkBytes;
        p.ring = static_cast<int32_t>(kLongRingBytes / kChunkBytes);  // a slice up to 112 KB is read once
        p.tiles = M;
        smem = kHeaderBytes + static_cast<size_t>(p.ring) * p.slot_bytes;
    }
    if (smem > kMaxSmemBytes) return cudaErrorInvalidConfiguration;
    int &fit = ds.clusters[team ? 0 : 1][csize];
    if (fit == 0) {
        int n = 0;
        // queried at the largest shared-memory size this mode uses, so the count holds for all
        const size_t fit_smem = team ? kHeaderBytes + 2 * (kTeamMaxCols * 4) : kHeaderBytes + kLongRingBytes;
        e = max_clusters(kernel, csize, fit_smem, &n);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        fit = n > 0 ? n : -1;
    }
    if (fit < 0) return launch_plain(X, Y, M, N, ldx, ldy, num_sms, vec, stream);
    const int64_t clusters = lmin(p.tiles, fit);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * csize));
    cfg.blockDim = dim3(kStagedThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // The team kernels' set-up overlaps the previous kernel (measured: 2.4% at 4096 x 16384);
    // the long-slice kernel launches after it (programmatic launch measured 8% slower there).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = team ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace tct
