// api.cu -- the C ABI: argument validation, launch planning, TMA descriptor encoding and
// the stream-ordered launch sequence (optional operand repack, then the GEMM kernel).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "gemm_internal.h"
#include "tile_sched.h"
#include "tensor_core_tiled.h"

namespace {

constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr int kDefaultGroupM = 8;
constexpr int kDefaultTimeoutMs = 2000;
constexpr int kMaxDevices = 64;

// Kernel variants the planner chooses between, with the relative per-tile throughput
// each reached on GB300 with every SM busy (8192^3 and 4096^3, same clocks): the pair
// 256 x 256 tile moves the fewest operand bytes into shared memory per FLOP; the pair
// 256 x 192 tile loads the same stage bytes for three quarters of the MMAs (measured 0.80
// of the 256-column rate at 8192^3, 0.86 at 1792^3) and pays off where it fills a wave
// better (1792^3: 70 tiles on 76 pairs instead of 49); the 128-column tiles are much slower
// per tile and only pay off when they fill SMs that a wider tile would leave idle (skinny
// M or N).  The planner weighs these against wave quantisation.
struct Candidate {
    int cta_group, tile_n, stages;
    double rate;
};
// Time model of one launch (seconds), for choosing between plans.  Per-SM tensor rate at a
// typical loaded clock (8192 FP16 FLOP per clock per SM x 1.9 GHz), HBM copy bandwidth, L2
// bandwidth for the split tiles' parts, and the exposed cost of a split tile's fix-up.
constexpr double kSmFlops = 8192.0 * 1.9e9;
constexpr double kHbmBytesPerSec = 6.5e12;
constexpr double kL2BytesPerSec = 20e12;
constexpr double kL2Bytes = 128.0 * 1024 * 1024;  // about the L2 capacity
// Measured on GB300: the second half's write, its transfer to the owner and the owner's
// store are serial after the halves finish, about two tile epilogues plus a flag handoff.
constexpr double kFixupSec = 12e-6;       // split tile combined through workspace (measured)
constexpr double kFixupReduceSec = 3e-6;  // split tile combined by TMA reduce-add into C
// A tile is only split in two when each half has at least this many k-blocks; a stream-K
// range is at least this long too.
constexpr int64_t kMinSplitIters = 4;
// Exposed cost of one link of a stream-K chain: a piece that ends inside its tile waits for
// the next piece to be in C (its TMA writes complete, then its flag), then adds its own rows
// (128 x tile_n FP32 per CTA) by TMA reduce-add.  Measured on GB300 against whole tiles on
// the same shapes: about 3.5 us per link with 128-column tiles and 5.5 us with 256-column
// tiles (a fixed 1.5 us plus the rows at about 33 GB/s per SM).
constexpr double kLinkFixedSec = 1.5e-6;
constexpr double kLinkBytesPerSecPerSm = 33e9;
// Pieces one tile may be cut into (bounds the chain's length); the planner tries each cap.
// Cap 1 asks for ranges of at least a tile less one k-block, so that no tile has more than two
// pieces: those add into C in either order with no chain (split_mode 3).
constexpr int64_t kStreamKPieceCaps[] = {1, 2, 3, 4, 6};

constexpr Candidate kCandidates[] = {
    {2, 256, 6, 1.00},
    {2, 192, 6, 0.82},
    {1, 256, 4, 0.85},
    {1, 128, 6, 0.70},
    {2, 128, 8, 0.57},
};

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int major = 0;
    int minor = 0;
    int pair_clusters = 0;  // co-resident CTA pairs of the pair kernels (0 = not queried)
    cudaMemPool_t pool = nullptr;  // stream-ordered temporaries (repacks, stream-K partials)
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

gemm_status device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        d.ready = true;
    }
    *out = d;
    if (d.major != 10 || d.minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
    return GEMM_OK;
}

// The library's stream-ordered memory pool on the current device.  It keeps freed memory
// for reuse (release threshold = unlimited), so a temporary of the same size on the next
// call costs no new physical mapping; the memory is returned when the process exits.
gemm_status device_pool(cudaMemPool_t *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.pool) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return GEMM_ERR_CUDA;
        uint64_t keep = UINT64_MAX;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return GEMM_ERR_CUDA;
        }
        d.pool = pool;
    }
    *out = d.pool;
    return GEMM_OK;
}

gemm_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return GEMM_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    *fn = g_encode;
    return GEMM_OK;
}

// 2-D FP16 or BF16 tensor map over a row-major matrix of `rows` x `cols` with leading
// dimension `ld` (elements), boxes of 64 columns x box_rows rows, 128-byte swizzle, zero fill.
gemm_status encode_16bit_2d(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld,
                            uint32_t box_rows, bool bf16)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    gemm_status st = get_encoder(&enc);
    if (st != GEMM_OK) return st;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

bool tma_ok(const void *p, int64_t ld) { return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && (ld % 8 == 0); }

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

gemm_status check_options(const gemm_options *opt)
{
    if (!opt) return GEMM_OK;
    if (opt->fault_inject < 0 || opt->fault_inject > 3) return GEMM_ERR_INVALID_ARG;
    if (opt->stream_k < 0 || opt->stream_k > 3) return GEMM_ERR_INVALID_ARG;
    if (opt->group_m < 0 || opt->group_m > 256) return GEMM_ERR_INVALID_ARG;
    if (opt->tile_n != 0 && opt->tile_n != 128 && opt->tile_n != 192 && opt->tile_n != 256) return GEMM_ERR_INVALID_ARG;
    if (opt->cta_group < 0 || opt->cta_group > 2) return GEMM_ERR_INVALID_ARG;
    if (opt->stages < 0 || opt->max_ctas < 0 || opt->timeout_ms < 0) return GEMM_ERR_INVALID_ARG;
    if (opt->stages != 0) {
        // some compiled variant must match every field that is set
        bool any = false;
        for (int cg = 1; cg <= 2; ++cg)
            for (int tn = 128; tn <= 256; tn += 64) {
                if ((opt->cta_group && opt->cta_group != cg) || (opt->tile_n && opt->tile_n != tn)) continue;
                if (tct::variant_smem_bytes(cg, tn, opt->stages) > 0) any = true;
            }
        if (!any) return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

// Layout bits: 1 = A stored K x M, 2 = B stored N x K, 4 = BF16 operands.
bool a_t(int layout) { return (layout & 1) != 0; }
bool b_t(int layout) { return (layout & 2) != 0; }
bool is_bf16(int layout) { return (layout & 4) != 0; }

int type_bytes(int t) { return t == GEMM_DTYPE_F32 ? 4 : 2; }

gemm_status check_args(const void *A, const void *B, const void *C, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc, int layout = 0, int c_type = GEMM_DTYPE_F32)
{
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_ARG;
    if (lda < (a_t(layout) ? M : K) || ldb < (b_t(layout) ? K : N) || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (lda > kMaxDim * 4 || ldb > kMaxDim * 4 || ldc > kMaxDim * 4) return GEMM_ERR_INVALID_ARG;
    if (M > 0 && N > 0) {
        if (!C || reinterpret_cast<uintptr_t>(C) % type_bytes(c_type) != 0) return GEMM_ERR_INVALID_ARG;
    }
    if (M > 0 && N > 0 && K > 0) {
        if (!A || reinterpret_cast<uintptr_t>(A) % 2 != 0) return GEMM_ERR_INVALID_ARG;
        if (!B || reinterpret_cast<uintptr_t>(B) % 2 != 0) return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

double wave_util(int64_t M, int64_t N, int64_t tm, int64_t tn, int64_t slots, int64_t *tiles_out,
                 int64_t *waves_out)
{
    const int64_t tiles = tct::ceil_div(M, tm) * tct::ceil_div(N, tn);
    const int64_t waves = tct::ceil_div(tiles, slots);
    if (tiles_out) *tiles_out = tiles;
    if (waves_out) *waves_out = waves;
    return static_cast<double>(tiles) / static_cast<double>(waves * slots);
}

// Share of the HBM bandwidth that a fraction `busy` of the units streaming operands reaches.
// Measured on GB300 with the skinny 128 x 16384 x 16384 product: 128 of 152 SMs streaming B
// already draw as much as all 152 (a stream-K plan with every SM busy was not faster), so
// the bandwidth is taken as saturated from 80% of the units on.
double hbm_share(double busy) { return std::min(1.0, busy / 0.8); }

struct Split {
    int64_t units, tiles, waves, dp_tiles, split_tiles;
    int64_t split_kb, parts;  // owner's k-blocks of a split tile; second parts per helper
                              // (stream-K: shortest range; most pieces of one tile)
    double time, eff_waves;
    double compute;  // the compute part of `time` (tile time x effective waves)
    int form;        // 0 whole tiles, 1 two-part split tail, 2 stream-K
    int64_t sk_units;
    bool mem_bound;  // the memory term sets `time`
    double l2_bytes; // operand bytes the tiles' TMA loads move from L2 into shared memory
};

// Work split and modelled time of one variant.  Whole waves of tiles go data-parallel; the
// last, partial wave either runs as whole tiles (a full extra wave of time, "02_gpu_execution
// _model.py" part 5) or has each of its `rest` tiles split into two k-parts: the owner unit
// takes the first split_kb k-blocks, and the units - rest other units ("helpers") each take
// the second parts of p = ceil(rest / helpers) tiles in turn, split_kb balancing the owner's
// split_kb against a helper's p * (kb - split_kb).  p = 1 is the even halving (at most half
// the units in the last wave); larger p needs the reduce-add combination (workspace holds
// one part per helper).  Memory time assumes HBM bandwidth in proportion to busy units.
Split model_split(int64_t M, int64_t N, int64_t K, int cg, int tile_n, int stages, double rate, int64_t units,
                  int want_sk, double fixup_sec, bool reduce_split)
{
    Split sp{};
    const int64_t tile_m = kTileM * cg;
    const int64_t tiles = tct::ceil_div(M, tile_m) * tct::ceil_div(N, tile_n);
    const int64_t kb = std::max<int64_t>(1, tct::ceil_div(K, kTileK));
    units = std::max<int64_t>(1, units);
    const double tile_sec = 2.0 * tile_m * tile_n * static_cast<double>(kb * kTileK) / (cg * kSmFlops * rate);
    const double tile_bytes = 4.0 * tile_m * tile_n;
    const double bytes = 2.0 * M * K + 2.0 * K * N + 4.0 * M * N;
    // whole tiles only, on at most one unit per tile
    const int64_t dp_units = std::min<int64_t>(units, tiles);
    const int64_t waves = tct::ceil_div(tiles, dp_units);
    const double busy = static_cast<double>(dp_units) / units;
    const double t_dp = std::max(waves * tile_sec, bytes / (kHbmBytesPerSec * hbm_share(busy)));
    sp.units = dp_units;
    sp.tiles = tiles;
    sp.waves = waves;
    sp.dp_tiles = tiles;
    sp.split_tiles = 0;
    sp.time = t_dp;
    sp.eff_waves = static_cast<double>(waves);
    sp.compute = waves * tile_sec;
    sp.mem_bound = t_dp > waves * tile_sec;
    sp.l2_bytes = 2.0 * static_cast<double>(tiles) * (tile_m + tile_n) * static_cast<double>(kb * kTileK);
    const int64_t full = tiles / units, rest = tiles - full * units;
    const int64_t helpers = units - rest;
    const int64_t p = helpers > 0 ? tct::ceil_div(rest, helpers) : 0;
    const int64_t kb_o = p > 0 ? tct::ceil_div(p * kb, p + 1) : 0;  // owner part >= a helper's total
    const int64_t min_iters = want_sk == 2 ? 1 : kMinSplitIters;
    const bool can_split = rest > 0 && helpers > 0 && (reduce_split || p == 1) && kb - kb_o >= 1 &&
                           kb_o >= min_iters && want_sk != 1 && tct::variant_split_ok(cg, tile_n, stages);
    if (can_split) {
        const double t_tail = static_cast<double>(std::max(kb_o, p * (kb - kb_o))) / kb;
        const double ew = full + t_tail;
        const double busy_split = static_cast<double>(rest + std::min(helpers, rest)) / units;
        const double t_tail_mem = (full > 0 ? bytes * full / tiles / kHbmBytesPerSec : 0.0) +
                                  bytes * rest / tiles / (kHbmBytesPerSec * hbm_share(busy_split));
        // a helper combines each of its p parts (measured: 9 short parts per helper at 3072^3
        // cost more than the whole extra wave they replace)
        const double t_sp = std::max(ew * tile_sec, t_tail_mem) + fixup_sec * p +
                            2.0 * rest * tile_bytes / kL2BytesPerSec;
        if (want_sk == 2 || t_sp < t_dp) {
            sp.units = units;
            sp.waves = tct::ceil_div(tiles, units);
            sp.dp_tiles = full * units;
            sp.split_tiles = rest;
            sp.split_kb = kb_o;
            sp.parts = p;
            sp.time = t_sp;
            sp.eff_waves = ew;
            sp.compute = ew * tile_sec;
            sp.form = 1;
            sp.mem_bound = t_tail_mem > ew * tile_sec;
        }
    }
    // Stream-K ("02_gpu_execution_model.py" part 5: rather than leave a partial wave's SMs
    // idle, cut the remaining work finer): after dpw whole waves, the k-blocks of the other
    // tiles are shared out in contiguous, balanced ranges over sku units.  The tiles whose
    // k-blocks are shared are the partial wave, or the partial wave and one whole wave
    // before it (longer ranges, fewer pieces per tile).  Each unit's time is dpw tiles plus
    // its range; a tile cut into c pieces adds c - 1 links to the critical path.  Only with
    // the reduce-add combination (plain FP32 epilogue, C TMA-writable).
    if (reduce_split && (want_sk == 0 || want_sk == 3)) {
        bool found = false;
        Split best{};
        const double link_sec = kLinkFixedSec + 4.0 * kTileM * tile_n / kLinkBytesPerSecPerSm;
        for (int64_t d = 0; d <= 1; ++d) {
            const int64_t dpw = full - d;
            if (dpw < 0) continue;
            const int64_t skt = tiles - dpw * units;
            if (skt <= 0) continue;
            const int64_t iters = skt * kb;
            for (const int64_t cap : kStreamKPieceCaps) {
                const int64_t qmin = std::max<int64_t>(want_sk == 3 ? 1 : kMinSplitIters,
                                                       cap == 1 ? kb - 1 : tct::ceil_div(kb, cap));
                const int64_t sku = std::min<int64_t>(units, iters / qmin);
                // Not taken by default when the stream-K tiles outnumber the units: ranges that
                // run across several tiles put the units at scattered k positions, so the
                // k-slices a wave of whole tiles shares through L2 are no longer shared
                // (measured, tiles of two pieces: 4096^3 94.9 against 88.8 us for the two-part
                // split, 4096 x 4096 x 16384 417.7 against 347.5).
                if (sku < 2 || (want_sk != 3 && sku <= skt)) continue;
                const int64_t q = iters / sku, qmax = tct::ceil_div(iters, sku);
                const int64_t pieces = std::min<int64_t>(tct::ceil_div(kb - 1, q) + 1, sku);
                const double ew = dpw + static_cast<double>(qmax) / kb;
                const double busy_sk = static_cast<double>(sku) / units;
                const double t_mem = (dpw > 0 ? bytes * dpw * units / tiles / kHbmBytesPerSec : 0.0) +
                                     bytes * skt / tiles / (kHbmBytesPerSec * hbm_share(busy_sk));
                // at most two pieces per tile: one reduce-add pass, no chain
                const double comb = pieces <= 2 ? fixup_sec : (pieces - 1) * link_sec;
                const double t = std::max(ew * tile_sec, t_mem) + comb;
                if (!found || t < best.time) {
                    found = true;
                    best = sp;
                    best.units = units;
                    best.waves = tct::ceil_div(tiles, units);
                    best.dp_tiles = dpw * units;
                    best.split_tiles = skt;
                    best.split_kb = q;
                    best.parts = pieces;
                    best.time = t;
                    best.eff_waves = ew;
                    best.compute = ew * tile_sec;
                    best.form = 2;
                    best.sk_units = sku;
                    best.mem_bound = t_mem > ew * tile_sec;
                }
            }
        }
        if (found && (want_sk == 3 || best.time < sp.time)) sp = best;
    }
    return sp;
}

// Choice among the compiled variants by modelled time: wave quantisation, the per-tile rate
// of each variant, and HBM time for bandwidth-bound shapes.
// pair_slots: co-resident CTA pairs (from the device, or sms / 2 when planning offline).
// reduce_split: split tiles may be combined by TMA reduce-add into C (plain FP32 epilogue,
// TMA-addressable C), the cheaper combination.
gemm_status make_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int sms, int pair_slots,
                      const gemm_options *opt, const void *A, const void *B, gemm_plan *pl, bool allow_split = true,
                      int layout = 0, bool reduce_split = true)
{
    std::memset(pl, 0, sizeof(*pl));
    const int want_cg = opt ? opt->cta_group : 0;
    const int want_tn = opt ? opt->tile_n : 0;
    const int want_st = opt ? opt->stages : 0;
    const int want_sk = allow_split ? (opt ? opt->stream_k : 0) : 1;
    const int64_t cap = opt && opt->max_ctas > 0 ? opt->max_ctas : 0;
    const Candidate *best = nullptr;
    Split best_sp{};
    for (const Candidate &c : kCandidates) {
        if ((want_cg && want_cg != c.cta_group) || (want_tn && want_tn != c.tile_n)) continue;
        if (!tct::variant_exists(layout, c.cta_group, c.tile_n, want_st ? want_st : c.stages)) continue;
        int64_t units = c.cta_group == 2 ? pair_slots : sms;
        if (cap > 0) units = std::min<int64_t>(units, std::max<int64_t>(1, cap / c.cta_group));
        if (units < 1) continue;
        const int st = want_st ? want_st : c.stages;
        const Split sp = model_split(M, N, K, c.cta_group, c.tile_n, st, c.rate, units, want_sk,
                                     reduce_split ? kFixupReduceSec : kFixupSec, reduce_split);
        if (want_sk == 3 && sp.form != 2) continue;  // stream-K asked for: only plans that use it
        // Within 1% (e.g. every candidate bound by the same HBM time) the one with less compute
        // time wins: it has the most slack (measured: 1-CTA 128x128 tiles stream the skinny
        // 128 x 16384 x 16384 shape 5% faster than CTA-pair 256x256 tiles, half of whose rows
        // are empty).  Between two bandwidth-bound plans within 5%, the one whose tiles move
        // fewer operand bytes from L2 into shared memory wins first (measured at 128 x 16384 x
        // 16384: 1-CTA 128x256 tiles, each split in two k-halves, 4-5% faster than whole
        // 128x128 tiles, which re-read A twice as often); only for operands larger than L2,
        // which stream from HBM.
        const bool tie = best && sp.time <= best_sp.time * 1.01 && best_sp.time <= sp.time * 1.01;
        const bool streaming = 2.0 * (static_cast<double>(M) * K + static_cast<double>(K) * N) > kL2Bytes;
        const bool mem_tie = best && streaming && sp.mem_bound && best_sp.mem_bound && sp.time <= best_sp.time * 1.05 &&
                             best_sp.time <= sp.time * 1.05 &&
                             (sp.l2_bytes < best_sp.l2_bytes * 0.9 || best_sp.l2_bytes < sp.l2_bytes * 0.9);
        if (!best || (mem_tie ? sp.l2_bytes < best_sp.l2_bytes
                              : (tie ? sp.compute < best_sp.compute : sp.time < best_sp.time))) {
            best = &c;
            best_sp = sp;
        }
    }
    if (!best) return GEMM_ERR_INVALID_ARG;
    const int cg = best->cta_group, tile_n = best->tile_n;
    const int stages = want_st ? want_st : best->stages;
    const int smem = tct::variant_smem_bytes(cg, tile_n, stages);
    if (smem < 0) return GEMM_ERR_INVALID_ARG;
    const int tile_m = kTileM * cg;
    pl->tile_m = tile_m;
    pl->tile_n = tile_n;
    pl->tile_k = kTileK;
    pl->stages = stages;
    pl->group_m = opt && opt->group_m ? opt->group_m : kDefaultGroupM;
    // The kernel indexes tiles with 32-bit integers (no allocation on one device holds a C
    // with 2^31 tiles of 128 x 128 or more; such sizes can only be a caller's mistake).
    if (best_sp.tiles >= (int64_t{1} << 31)) return GEMM_ERR_INVALID_ARG;
    pl->grid = static_cast<int32_t>(best_sp.units * cg);
    pl->tiles = best_sp.tiles;
    pl->waves = best_sp.waves;
    pl->wave_efficiency = static_cast<double>(M) * N /
                          (static_cast<double>(best_sp.waves) * best_sp.units * tile_m * tile_n);
    pl->smem_bytes = smem;
    pl->pack_a = (K > 0 && !tma_ok(A, lda)) ? 1 : 0;
    pl->pack_b = (K > 0 && !tma_ok(B, ldb)) ? 1 : 0;
    pl->cta_group = cg;
    pl->units = static_cast<int32_t>(best_sp.units);
    pl->stream_k_tiles = static_cast<int32_t>(best_sp.split_tiles);
    pl->effective_waves = best_sp.eff_waves;
    pl->split_kb = static_cast<int32_t>(best_sp.split_kb);
    pl->split_parts_per_unit = static_cast<int32_t>(best_sp.parts);
    pl->split_form = best_sp.form;
    pl->sk_units = static_cast<int32_t>(best_sp.sk_units);
    if (want_sk == 3 && best_sp.form != 2) return GEMM_ERR_INVALID_ARG;  // stream-K asked for, not possible
    return GEMM_OK;
}

// Kernel parameters for a plan (the caller sets `workspace` when stream-K is used).
// Epilogue fields of the kernel parameters (identity when epi is NULL).
void set_epilogue(tct::KernelParams &p, void *C, int c_type, int64_t ldc, const gemm_epilogue *epi)
{
    p.C = C;
    p.c_type = c_type;
    p.vec_store = (reinterpret_cast<uintptr_t>(C) % (4 * type_bytes(c_type)) == 0 && ldc % 4 == 0) ? 1 : 0;
    p.alpha = epi ? epi->alpha : 1.0f;
    p.beta = epi ? epi->beta : 0.0f;
    p.bias = epi ? epi->bias : nullptr;
    p.bias_type = epi ? epi->bias_type : GEMM_DTYPE_F32;
    p.bias_vec = (p.bias && reinterpret_cast<uintptr_t>(p.bias) % (4 * type_bytes(p.bias_type)) == 0) ? 1 : 0;
    p.epi = (p.alpha != 1.0f || p.beta != 0.0f || p.bias != nullptr) ? 1 : 0;
}

tct::KernelParams make_params(const gemm_plan &pl, float *C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                              int timeout_ms)
{
    tct::KernelParams p;
    set_epilogue(p, C, GEMM_DTYPE_F32, ldc, nullptr);
    p.ldc = ldc;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.num_m = static_cast<int32_t>(tct::ceil_div(M, pl.tile_m));
    p.num_n = static_cast<int32_t>(tct::ceil_div(N, pl.tile_n));
    p.num_kb = static_cast<int32_t>(tct::ceil_div(K, kTileK));
    p.num_tiles = static_cast<int32_t>(pl.tiles);
    p.group_m = pl.group_m;
    p.timeout_ns = static_cast<uint64_t>(timeout_ms) * 1000000ull;
    p.units = pl.units;
    p.dp_tiles = static_cast<int32_t>(pl.tiles - pl.stream_k_tiles);
    p.split_tiles = pl.stream_k_tiles;
    p.split_kb = pl.split_kb;
    p.workspace = nullptr;
    p.flags = nullptr;
    p.fault_inject = 0;
    // stream-K: tiles of at most two pieces add in either order; longer ones chain
    p.split_mode = pl.split_form == 2 ? (pl.split_parts_per_unit <= 2 ? 3 : 2) : 0;
    p.sk_units = pl.split_form == 2 ? pl.sk_units : 0;
    p.b_stream = p.num_m == 1 ? 1 : 0;
    p.a_keep = (p.num_m > 1 && p.num_n > 1 &&
                2.0 * (static_cast<double>(M) * static_cast<double>(K) + static_cast<double>(K) * static_cast<double>(N)) >
                    kL2Bytes)
                   ? 1
                   : 0;
    p.c_tma = 0;
    return p;
}

// Split-tile workspace: one part (the second k-half) per split tile, then one flag per split
// tile and CTA rank.
int64_t split_parts_bytes(const gemm_plan &pl)
{
    if (pl.stream_k_tiles <= 0 || pl.split_form == 2) return 0;
    return static_cast<int64_t>(pl.stream_k_tiles) * pl.tile_m * pl.tile_n * 4;
}

int64_t split_flags_bytes(const gemm_plan &pl)
{
    if (pl.stream_k_tiles <= 0) return 0;
    if (pl.split_form == 2)  // a flag per unit (chains) or per stream-K tile (pairs)
        return round_up(std::max<int64_t>(pl.sk_units, pl.stream_k_tiles) * pl.cta_group * 4, 256);
    return round_up(static_cast<int64_t>(pl.stream_k_tiles) * pl.cta_group * 4, 256);
}

// 2-D FP32 tensor map over the split parts: rows of tile_n floats, boxes of tile_n x 32.
gemm_status encode_parts(CUtensorMap *m, const float *base, int64_t rows, int tile_n)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    gemm_status st = get_encoder(&enc);
    if (st != GEMM_OK) return st;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(tile_n), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(tile_n) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(tile_n), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// 2-D tensor map over C in its own type, for the TMA stores of whole tiles and the TMA
// reduce-add of split tiles: boxes of 128 bytes of a row (32 FP32 or 64 FP16/BF16 columns,
// 128-byte swizzle, the epilogue's staging layout) by 32 rows.
gemm_status encode_c_map(CUtensorMap *m, void *C, int c_type, int64_t M, int64_t N, int64_t ldc)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    gemm_status st = get_encoder(&enc);
    if (st != GEMM_OK) return st;
    const int esz = type_bytes(c_type);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), 32};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = c_type == GEMM_DTYPE_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : c_type == GEMM_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(m, dt, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Whether TMA may write C of type c_type: a 16-byte aligned base and row pitch, and rows of
// whole 16-byte units.  TMA stores and reduce-adds clip a box at the tensor's edge in whole
// 16-byte units of the row (measured on GB300 for FP32: with N = 4q + r, r > 0, columns up
// to 4q + 3 are written), so a row that ends inside a 16-byte unit would have its padding
// written.
bool c_tma_ok(const void *C, int c_type, int64_t N, int64_t ldc)
{
    const int per16 = 16 / type_bytes(c_type);
    return reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % per16 == 0 && N % per16 == 0;
}

// Co-resident CTA pairs on the current device for the pair kernels (queried once).
int device_pair_slots(DeviceInfo *dev)
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return dev->sms / 2;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_dev[d].pair_clusters == 0) {
        const int n = tct::variant_max_clusters(2, 256, 6);
        g_dev[d].pair_clusters = n > 0 ? n : std::max(1, g_dev[d].sms / 2);
    }
    dev->pair_clusters = g_dev[d].pair_clusters;
    return dev->pair_clusters;
}

gemm_status to_status(cudaError_t e) { return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA; }

// The launch sequence for every operand layout (see make_plan for the layout bits).
gemm_status check_epilogue(int c_type, const gemm_epilogue *epi)
{
    if (c_type != GEMM_DTYPE_F16 && c_type != GEMM_DTYPE_BF16 && c_type != GEMM_DTYPE_F32) return GEMM_ERR_INVALID_ARG;
    if (!epi) return GEMM_OK;
    if (epi->reserved != 0) return GEMM_ERR_INVALID_ARG;
    if (epi->bias_type != GEMM_DTYPE_F16 && epi->bias_type != GEMM_DTYPE_BF16 && epi->bias_type != GEMM_DTYPE_F32)
        return GEMM_ERR_INVALID_ARG;
    if (epi->bias && reinterpret_cast<uintptr_t>(epi->bias) % type_bytes(epi->bias_type) != 0)
        return GEMM_ERR_INVALID_ARG;
    if (!std::isfinite(epi->alpha) || !std::isfinite(epi->beta)) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

gemm_status run_gemm(int layout, const void *A, const void *B, void *C, int c_type, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, const gemm_epilogue *epi, void *stream,
                     const gemm_options *opt)
{
    gemm_status st = check_args(A, B, C, M, N, K, lda, ldb, ldc, layout, c_type);
    if (st != GEMM_OK) return st;
    st = check_epilogue(c_type, epi);
    if (st != GEMM_OK) return st;
    st = check_options(opt);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceInfo dev;
    st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        tct::KernelParams p{};
        p.M = static_cast<int32_t>(M);
        p.N = static_cast<int32_t>(N);
        p.ldc = ldc;
        set_epilogue(p, C, c_type, ldc, epi);
        return to_status(tct::launch_fill_epilogue(p, dev.sms, s));
    }

    // When TMA can write C, whole tiles go out by TMA stores, and with the plain FP32
    // epilogue split tiles add into C by TMA reduce-add; otherwise tiles are stored by the
    // epilogue warps, and split tiles combine through workspace.
    const bool plain = !epi || (epi->alpha == 1.0f && epi->beta == 0.0f && !epi->bias);
    const bool c_tma = c_tma_ok(C, c_type, N, ldc);
    const bool reduce_ok = plain && c_type == GEMM_DTYPE_F32 && c_tma;
    gemm_plan pl;
    st = make_plan(M, N, K, lda, ldb, dev.sms, device_pair_slots(&dev), opt, A, B, &pl, true, layout, reduce_ok);
    if (st != GEMM_OK) return st;

    // Stored shapes: A is M x K, or K x M when transposed; B is K x N, or N x K.
    const int64_t a_rows = a_t(layout) ? K : M, a_cols = a_t(layout) ? M : K;
    const int64_t b_rows = b_t(layout) ? N : K, b_cols = b_t(layout) ? K : N;

    // Operands whose rows do not start on 16-byte boundaries are copied first (TMA needs
    // 16-byte aligned bases and row strides); the copy is stream-ordered.  The same
    // stream-ordered block holds the split tiles' parts and flags.
    const void *a_use = A, *b_use = B;
    int64_t lda_use = lda, ldb_use = ldb;
    const int64_t lda_p = round_up(a_cols, 8), ldb_p = round_up(b_cols, 8);
    const int64_t a_bytes = pl.pack_a ? round_up(a_rows * lda_p * 2, 256) : 0;
    const int64_t b_bytes = pl.pack_b ? round_up(b_rows * ldb_p * 2, 256) : 0;
    const int64_t w_bytes = reduce_ok ? 0 : split_parts_bytes(pl), f_bytes = split_flags_bytes(pl);
    void *ws = nullptr;
    if (a_bytes + b_bytes + w_bytes + f_bytes > 0) {
        cudaMemPool_t pool = nullptr;
        st = device_pool(&pool);
        if (st != GEMM_OK) return st;
        if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(a_bytes + b_bytes + w_bytes + f_bytes), pool, s) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
        uint8_t *w = static_cast<uint8_t *>(ws);
        if (pl.pack_a) {
            a_use = w;
            lda_use = lda_p;
        }
        if (pl.pack_b) {
            b_use = w + a_bytes;
            ldb_use = ldb_p;
        }
        cudaError_t e = tct::launch_copy_rows(
            tct::RowCopy{pl.pack_a ? A : nullptr, lda, w, lda_p, a_rows, a_cols, 2},
            tct::RowCopy{pl.pack_b ? B : nullptr, ldb, w + a_bytes, ldb_p, b_rows, b_cols, 2}, s, dev.sms);
        if (e == cudaSuccess && f_bytes)  // the split tiles' flags start lowered
            e = cudaMemsetAsync(w + a_bytes + b_bytes + w_bytes, 0, static_cast<size_t>(f_bytes), s);
        if (e != cudaSuccess) {
            cudaFreeAsync(ws, s);
            return GEMM_ERR_CUDA;
        }
    }

    // TMA boxes: A as M x K -> 64(K) x 128(M); as K x M -> 64(M) x 64(K).  B as K x N ->
    // 64(N) x 64(K); as N x K -> 64(K) x (tile_n / cta_group)(N).
    CUtensorMap ta, tb;
    st = encode_16bit_2d(&ta, a_use, a_rows, a_cols, lda_use, a_t(layout) ? 64 : kTileM, is_bf16(layout));
    if (st == GEMM_OK)
        st = encode_16bit_2d(&tb, b_use, b_rows, b_cols, ldb_use,
                             b_t(layout) ? static_cast<uint32_t>(pl.tile_n / pl.cta_group) : kTileK, is_bf16(layout));
    if (st == GEMM_OK) {
        const int tmo = opt && opt->timeout_ms ? opt->timeout_ms : kDefaultTimeoutMs;
        tct::KernelParams p = make_params(pl, nullptr, M, N, K, ldc, tmo);
        set_epilogue(p, C, c_type, ldc, epi);
        p.fault_inject = opt ? opt->fault_inject : 0;
        CUtensorMap tp, tc;
        std::memset(&tp, 0, sizeof(tp));
        std::memset(&tc, 0, sizeof(tc));
        if (c_tma) {
            p.c_tma = 1;
            st = encode_c_map(&tc, C, c_type, M, N, ldc);
        }
        if (pl.stream_k_tiles > 0 && st == GEMM_OK) {
            uint8_t *w = static_cast<uint8_t *>(ws) + a_bytes + b_bytes;
            p.flags = reinterpret_cast<unsigned int *>(w + w_bytes);
            if (pl.split_form == 2) {
                // stream-K pieces: split_mode 2 from the plan, flags only
            } else if (reduce_ok) {
                p.split_mode = 1;
            } else {
                p.workspace = reinterpret_cast<float *>(w);
                st = encode_parts(&tp, p.workspace, static_cast<int64_t>(pl.stream_k_tiles) * pl.tile_m, pl.tile_n);
            }
        }
        if (st == GEMM_OK)
            st = to_status(tct::launch_gemm(ta, tb, tp, tc, p, layout, pl.cta_group, pl.tile_n, pl.stages, pl.grid, s));
    }
    if (ws) {
        if (cudaFreeAsync(ws, s) != cudaSuccess && st == GEMM_OK) st = GEMM_ERR_CUDA;
    }
    return st;
}

}  // namespace

extern "C" {

gemm_status gemm_f16_f32_ex(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldc, void *stream, const gemm_options *opt)
{
    return run_gemm(0, A, B, C, GEMM_DTYPE_F32, M, N, K, lda, ldb, ldc, nullptr, stream, opt);
}

gemm_status gemm_f32acc(int32_t ab_type, int32_t op_a, int32_t op_b, const void *A, const void *B, float *C,
                        int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void *stream,
                        const gemm_options *opt)
{
    if ((ab_type != GEMM_DTYPE_F16 && ab_type != GEMM_DTYPE_BF16) || (op_a != GEMM_OP_N && op_a != GEMM_OP_T) ||
        (op_b != GEMM_OP_N && op_b != GEMM_OP_T))
        return GEMM_ERR_INVALID_ARG;
    const int layout = (op_a == GEMM_OP_T ? 1 : 0) | (op_b == GEMM_OP_T ? 2 : 0) | (ab_type == GEMM_DTYPE_BF16 ? 4 : 0);
    return run_gemm(layout, A, B, C, GEMM_DTYPE_F32, M, N, K, lda, ldb, ldc, nullptr, stream, opt);
}

gemm_status gemm_ex(int32_t ab_type, int32_t op_a, int32_t op_b, const void *A, const void *B, void *C,
                    int32_t c_type, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                    const gemm_epilogue *epi, void *stream, const gemm_options *opt)
{
    if ((ab_type != GEMM_DTYPE_F16 && ab_type != GEMM_DTYPE_BF16) || (op_a != GEMM_OP_N && op_a != GEMM_OP_T) ||
        (op_b != GEMM_OP_N && op_b != GEMM_OP_T))
        return GEMM_ERR_INVALID_ARG;
    const int layout = (op_a == GEMM_OP_T ? 1 : 0) | (op_b == GEMM_OP_T ? 2 : 0) | (ab_type == GEMM_DTYPE_BF16 ? 4 : 0);
    return run_gemm(layout, A, B, C, c_type, M, N, K, lda, ldb, ldc, epi, stream, opt);
}

gemm_status softmax_rows_f32(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy, void *stream)
{
    if (M < 0 || N < 0 || M > kMaxDim || N > kMaxDim || ldx < N || ldy < N) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!X || !Y || reinterpret_cast<uintptr_t>(X) % 4 || reinterpret_cast<uintptr_t>(Y) % 4) return GEMM_ERR_INVALID_ARG;
    if (X == Y && ldx != ldy) return GEMM_ERR_INVALID_ARG;
    DeviceInfo dev;
    const gemm_status st = device_info(&dev);
    if (st != GEMM_OK) return st;
    unsigned *err = nullptr;
    if (tct::error_word_address(&err) != cudaSuccess) return GEMM_ERR_CUDA;
    return to_status(tct::launch_softmax_rows(X, Y, M, N, ldx, ldy, dev.sms, err,
                                              static_cast<uint64_t>(kDefaultTimeoutMs) * 1000000ull,
                                              static_cast<cudaStream_t>(stream)));
}

gemm_status gemm_f16_f32(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldc, void *stream)
{
    return gemm_f16_f32_ex(A, B, C, M, N, K, lda, ldb, ldc, stream, nullptr);
}

gemm_status gemm_f16_f32_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int32_t num_sms,
                              const gemm_options *opt, gemm_plan *out)
{
    if (!out) return GEMM_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || lda < K || ldb < N)
        return GEMM_ERR_INVALID_ARG;
    gemm_status st = check_options(opt);
    if (st != GEMM_OK) return st;
    int sms = num_sms, pairs = num_sms / 2;
    if (sms <= 0) {
        DeviceInfo dev;
        st = device_info(&dev);
        if (st != GEMM_OK) return st;
        sms = dev.sms;
        pairs = device_pair_slots(&dev);
    }
    // Alignment of the base pointers is unknown here: assume 16-byte aligned bases (and ldc
    // a multiple of 4, so that C is TMA-writable exactly when N is a multiple of 4).
    const void *aligned = reinterpret_cast<const void *>(uintptr_t{256});
    return make_plan(M, N, K, lda, ldb, sms, pairs, opt, aligned, aligned, out, true, 0,
                     c_tma_ok(aligned, GEMM_DTYPE_F32, N, round_up(N, 4)));
}

gemm_status gemm_f16_f32_work_item(int64_t M, int64_t N, int64_t K, int32_t num_sms, const gemm_options *opt,
                                   int32_t unit, int32_t idx, gemm_work *out)
{
    if (!out || num_sms <= 0 || unit < 0 || idx < 0) return GEMM_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_ARG;
    gemm_status st = check_options(opt);
    if (st != GEMM_OK) return st;
    const void *aligned = reinterpret_cast<const void *>(uintptr_t{256});
    gemm_plan pl;
    st = make_plan(M, N, K, K, N, num_sms, num_sms / 2, opt, aligned, aligned, &pl);
    if (st != GEMM_OK) return st;
    if (unit >= pl.units) return GEMM_ERR_INVALID_ARG;
    const tct::KernelParams p = make_params(pl, nullptr, M, N, K, N, kDefaultTimeoutMs);
    tct::WorkItem w;
    if (!tct::work_item(p, unit, idx, w)) return GEMM_ERR_INVALID_ARG;
    out->tile = w.tile;
    out->kb0 = w.kb0;
    out->kb1 = w.kb1;
    out->mode = w.mode;
    out->part = w.part;
    return GEMM_OK;
}

gemm_status gemm_tile_coord(int64_t t, int64_t num_m, int64_t num_n, int32_t group_m, int64_t *tile_row,
                            int64_t *tile_col)
{
    if (num_m <= 0 || num_n <= 0 || group_m <= 0 || t < 0 || !tile_row || !tile_col) return GEMM_ERR_INVALID_ARG;
    if (num_m > kMaxDim || num_n > kMaxDim || num_m * num_n > kMaxDim || t >= num_m * num_n)
        return GEMM_ERR_INVALID_ARG;
    const tct::TileCoord c = tct::tile_coord(static_cast<int32_t>(t), static_cast<int32_t>(num_m),
                                             static_cast<int32_t>(num_n), group_m);
    *tile_row = c.m;
    *tile_col = c.n;
    return GEMM_OK;
}

gemm_status gemm_wave_model(int64_t M, int64_t N, int64_t tile_m, int64_t tile_n, int64_t slots, int64_t *tiles,
                            int64_t *waves, double *utilization)
{
    if (M <= 0 || N <= 0 || tile_m <= 0 || tile_n <= 0 || slots <= 0) return GEMM_ERR_INVALID_ARG;
    const double u = wave_util(M, N, tile_m, tile_n, slots, tiles, waves);
    if (utilization) *utilization = u;
    return GEMM_OK;
}

gemm_status gemm_f16_f32_get_error(void)
{
    unsigned w = 0;
    if (tct::read_and_clear_error(&w) != cudaSuccess) return GEMM_ERR_CUDA;
    if (w == 0) return GEMM_OK;
    return static_cast<gemm_status>(w & 0xffu);
}

const char *gemm_status_string(int status)
{
    switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103, GB300)";
    case GEMM_ERR_CUDA: return "CUDA runtime or driver error";
    case GEMM_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
    }
}

const char *gemm_version(void) { return "tensor_core_tiled 0.1 sm_103a"; }

}  // extern "C"

// ---------------------------------------------------------------- allocation-free variant
//
// Some callers cannot call cudaMalloc: their device memory belongs to another allocator (a
// framework's caching pool, or a server that reserves the whole GPU when it starts), so a
// fresh driver allocation in the middle of a run can fail or stall, or their calling
// context (an operator/plugin interface that hands over only input and output buffers)
// forbids touching the CUDA allocator.  gemm_f16_f32_noalloc serves them: the only
// scratch the GEMM path can need -- the 16-byte-aligned copy of operands whose rows are
// not aligned for TMA -- lives in this fixed, library-owned device array instead of a
// cudaMallocAsync block.
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device, looked up once per device.
// In host code the array's name is only a host-side stand-in, so kernels must be given
// this address, never the symbol itself.
gemm_status noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GEMM_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status gemm_f16_f32_noalloc(const void *A, const void *B, float *C, int64_t M, int64_t N,
                                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void *stream)
{
    gemm_status st = check_args(A, B, C, M, N, K, lda, ldb, ldc);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    // Scratch needed for the repacked operands, checked against the fixed array first.
    const bool pack_a = K > 0 && !tma_ok(A, lda);
    const bool pack_b = K > 0 && !tma_ok(B, ldb);
    // Each size is compared with the limit before it is formed, so that no product or sum
    // can wrap around for the largest dimensions check_args accepts.
    constexpr int64_t kLimit = static_cast<int64_t>(GEMM_NOALLOC_SCRATCH_BYTES);
    const int64_t lda_p = round_up(K, 8), ldb_p = round_up(N, 8);
    if (pack_a && M > kLimit / (2 * lda_p)) return GEMM_ERR_INVALID_ARG;
    if (pack_b && K > kLimit / (2 * ldb_p)) return GEMM_ERR_INVALID_ARG;
    const int64_t a_bytes = pack_a ? round_up(M * lda_p * 2, 256) : 0;
    const int64_t b_bytes = pack_b ? round_up(K * ldb_p * 2, 256) : 0;
    if (a_bytes > kLimit || b_bytes > kLimit - a_bytes) return GEMM_ERR_INVALID_ARG;

    DeviceInfo dev;
    st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        tct::KernelParams p{};
        p.M = static_cast<int32_t>(M);
        p.N = static_cast<int32_t>(N);
        p.ldc = ldc;
        set_epilogue(p, C, GEMM_DTYPE_F32, ldc, nullptr);
        return to_status(tct::launch_fill_epilogue(p, dev.sms, s));
    }

    gemm_plan pl;
    st = make_plan(M, N, K, lda, ldb, dev.sms, device_pair_slots(&dev), nullptr, A, B, &pl,
                   /*allow_split=*/false);
    if (st != GEMM_OK) return st;

    const void *a_use = A, *b_use = B;
    int64_t lda_use = lda, ldb_use = ldb;
    if (pack_a || pack_b) {
        void *scratch = nullptr;
        st = noalloc_scratch(&scratch);
        if (st != GEMM_OK) return st;
        uint8_t *w = static_cast<uint8_t *>(scratch);
        // Every element the GEMM reads is written here first; nothing needs clearing.
        if (tct::launch_pack2(pack_a ? A : nullptr, lda, w, lda_p, M, K, pack_b ? B : nullptr, ldb, w + a_bytes,
                              ldb_p, K, N, s) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (pack_a) {
            a_use = w;
            lda_use = lda_p;
        }
        if (pack_b) {
            b_use = w + a_bytes;
            ldb_use = ldb_p;
        }
    }

    CUtensorMap ta, tb;
    st = encode_16bit_2d(&ta, a_use, M, K, lda_use, kTileM, false);
    if (st == GEMM_OK) st = encode_16bit_2d(&tb, b_use, K, N, ldb_use, kTileK, false);
    if (st != GEMM_OK) return st;
    tct::KernelParams p = make_params(pl, C, M, N, K, ldc, kDefaultTimeoutMs);
    CUtensorMap tp, tc;  // no split tiles on this path; the C map, for TMA stores, when C allows it
    std::memset(&tp, 0, sizeof(tp));
    std::memset(&tc, 0, sizeof(tc));
    if (c_tma_ok(C, GEMM_DTYPE_F32, N, ldc)) {
        p.c_tma = 1;
        st = encode_c_map(&tc, C, GEMM_DTYPE_F32, M, N, ldc);
        if (st != GEMM_OK) return st;
    }
    return to_status(tct::launch_gemm(ta, tb, tp, tc, p, 0, pl.cta_group, pl.tile_n, pl.stages, pl.grid, s));
}

// ---------------------------------------------------------------- host-buffer pipelines

namespace {

constexpr int kHostChunks = 8;        // row blocks of the host-buffer softmax
constexpr int kHostGemmBlocks = 4;    // row blocks of A and column blocks of B in the host GEMM
constexpr int64_t kHostChunkAlign = 256;  // GEMM blocks: whole CTA-pair tiles

// Per-device copy streams and events of the host-buffer calls.  One call at a time enqueues
// on them (the mutex); waits already enqueued keep the event state of their own call, so the
// events are reused by the next call.
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kHostChunks] = {}, out[kHostChunks] = {};
    cudaEvent_t a_in[kHostGemmBlocks] = {}, b_in[kHostGemmBlocks] = {};
    cudaEvent_t c_out[kHostGemmBlocks * kHostGemmBlocks] = {};
};
std::mutex g_host_mu;
HostPipe g_host[kMaxDevices];

gemm_status host_pipe(HostPipe **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    HostPipe &h = g_host[dev];
    if (!h.ready) {
        const unsigned ef = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.start, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.done, ef) == cudaSuccess;
        for (int i = 0; ok && i < kHostChunks; ++i)
            ok = cudaEventCreateWithFlags(&h.in[i], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.out[i], ef) == cudaSuccess;
        for (int i = 0; ok && i < kHostGemmBlocks; ++i)
            ok = cudaEventCreateWithFlags(&h.a_in[i], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.b_in[i], ef) == cudaSuccess;
        for (int i = 0; ok && i < kHostGemmBlocks * kHostGemmBlocks; ++i)
            ok = cudaEventCreateWithFlags(&h.c_out[i], ef) == cudaSuccess;
        if (!ok) return GEMM_ERR_CUDA;
        h.ready = true;
    }
    *out = &h;
    return GEMM_OK;
}

// Row blocks of a host-buffer call: ceil(M / kHostChunks) rounded up to `align`.
int64_t host_chunk_rows(int64_t M, int64_t align)
{
    return std::max<int64_t>(align, round_up((M + kHostChunks - 1) / kHostChunks, align));
}

// Ends a host-buffer call: the caller's stream waits for both copy streams, then releases the
// device temporary (also on the error path, so nothing in flight loses its memory).
gemm_status host_finish(HostPipe *hp, cudaStream_t s, void *ws, gemm_status result)
{
    bool ok = cudaEventRecord(hp->done, hp->d2h) == cudaSuccess && cudaStreamWaitEvent(s, hp->done, 0) == cudaSuccess &&
              cudaEventRecord(hp->start, hp->h2d) == cudaSuccess && cudaStreamWaitEvent(s, hp->start, 0) == cudaSuccess;
    ok = cudaFreeAsync(ws, s) == cudaSuccess && ok;
    return result != GEMM_OK ? result : (ok ? GEMM_OK : GEMM_ERR_CUDA);
}

#define TCT_CUDA_OK(x)                                                 \
    do {                                                               \
        if ((x) != cudaSuccess) return host_finish(hp, s, ws, GEMM_ERR_CUDA); \
    } while (0)

}  // namespace

extern "C" gemm_status gemm_f16_f32_host(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                                         int64_t lda, int64_t ldb, int64_t ldc, void *stream)
{
    gemm_status st = check_args(A, B, C, M, N, K, lda, ldb, ldc, 0, GEMM_DTYPE_F32);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceInfo dev;
    st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaMemPool_t pool = nullptr;
    st = device_pool(&pool);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostPipe *hp = nullptr;
    st = host_pipe(&hp);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // Device copies with 16-byte row pitches, so that the GEMM reads them in place.
    const int64_t ka = round_up(std::max<int64_t>(K, 1), 8), nb = round_up(N, 8), nc = round_up(N, 4);
    const size_t a_bytes = static_cast<size_t>(M * ka * 2), b_bytes = static_cast<size_t>(K * nb * 2);
    const size_t c_bytes = static_cast<size_t>(M * nc * 4);
    const size_t a_off = round_up(static_cast<int64_t>(b_bytes), 256);
    const size_t c_off = a_off + round_up(static_cast<int64_t>(a_bytes), 256);
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, c_off + c_bytes, pool, s) != cudaSuccess) return GEMM_ERR_CUDA;
    char *base = static_cast<char *>(ws);
    auto *dB = reinterpret_cast<uint16_t *>(base);
    auto *dA = reinterpret_cast<uint16_t *>(base + a_off);
    auto *dC = reinterpret_cast<float *>(base + c_off);

    // Blocks: up to kHostGemmBlocks row blocks of A and column blocks of B, on whole-tile
    // boundaries.  The copy stream sends them interleaved along the diagonal (A0, B0, B1, A1,
    // A2, B2, ...); as soon as the inputs of block C(i, j) are on the device its product runs
    // on the caller's stream and its rows go back on the second copy stream, so the
    // device-to-host copies start after the first A and B blocks, not after all of B.
    const int64_t rb = round_up(tct::ceil_div(M, kHostGemmBlocks), kHostChunkAlign);
    const int64_t cb = round_up(tct::ceil_div(N, kHostGemmBlocks), kHostChunkAlign);
    const int P = static_cast<int>(tct::ceil_div(M, rb)), Q = static_cast<int>(tct::ceil_div(N, cb));
    TCT_CUDA_OK(cudaEventRecord(hp->start, s));
    TCT_CUDA_OK(cudaStreamWaitEvent(hp->h2d, hp->start, 0));
    TCT_CUDA_OK(cudaStreamWaitEvent(hp->d2h, hp->start, 0));
    auto send_a = [&](int i) {
        const int64_t r0 = i * rb, mr = std::min(rb, M - r0);
        if (K > 0 && cudaMemcpy2DAsync(dA + r0 * ka, ka * 2, static_cast<const uint16_t *>(A) + r0 * lda, lda * 2,
                                       K * 2, mr, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess)
            return false;
        return cudaEventRecord(hp->a_in[i], hp->h2d) == cudaSuccess;
    };
    auto send_b = [&](int j) {
        const int64_t c0 = j * cb, nw = std::min(cb, N - c0);
        if (K > 0 && cudaMemcpy2DAsync(dB + c0, nb * 2, static_cast<const uint16_t *>(B) + c0, ldb * 2, nw * 2, K,
                                       cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess)
            return false;
        return cudaEventRecord(hp->b_in[j], hp->h2d) == cudaSuccess;
    };
    auto block = [&](int i, int j) {
        const int64_t r0 = i * rb, mr = std::min(rb, M - r0), c0 = j * cb, nw = std::min(cb, N - c0);
        if (cudaStreamWaitEvent(s, hp->a_in[i], 0) != cudaSuccess || cudaStreamWaitEvent(s, hp->b_in[j], 0) != cudaSuccess)
            return GEMM_ERR_CUDA;
        const gemm_status g =
            run_gemm(0, dA + r0 * ka, dB + c0, dC + r0 * nc + c0, GEMM_DTYPE_F32, mr, nw, K, ka, nb, nc, nullptr, s, nullptr);
        if (g != GEMM_OK) return g;
        cudaEvent_t done = hp->c_out[i * kHostGemmBlocks + j];
        if (cudaEventRecord(done, s) != cudaSuccess || cudaStreamWaitEvent(hp->d2h, done, 0) != cudaSuccess ||
            cudaMemcpy2DAsync(C + r0 * ldc + c0, ldc * 4, dC + r0 * nc + c0, nc * 4, nw * 4, mr, cudaMemcpyDeviceToHost,
                              hp->d2h) != cudaSuccess)
            return GEMM_ERR_CUDA;
        return GEMM_OK;
    };
    auto row_blocks = [&](int t) {  // row t against the earlier column blocks
        for (int j = 0; j < std::min(t, Q); ++j)
            if (t < P && (st = block(t, j)) != GEMM_OK) return false;
        return true;
    };
    auto col_blocks = [&](int t) {  // column t against the earlier row blocks
        for (int i = 0; i < std::min(t, P); ++i)
            if (t < Q && (st = block(i, t)) != GEMM_OK) return false;
        return true;
    };
    for (int t = 0; t < std::max(P, Q); ++t) {
        // A_t then B_t on even steps, B_t then A_t on odd ones; the blocks go on the caller's
        // stream in the order their inputs arrive (a block whose inputs are in never queues
        // behind one still waiting for its row or column), then the diagonal block.
        const bool a_first = (t % 2) == 0;
        if (a_first && t < P && !send_a(t)) return host_finish(hp, s, ws, GEMM_ERR_CUDA);
        if (!a_first && t < Q && !send_b(t)) return host_finish(hp, s, ws, GEMM_ERR_CUDA);
        if (!(a_first ? row_blocks(t) : col_blocks(t))) return host_finish(hp, s, ws, st);
        if (a_first && t < Q && !send_b(t)) return host_finish(hp, s, ws, GEMM_ERR_CUDA);
        if (!a_first && t < P && !send_a(t)) return host_finish(hp, s, ws, GEMM_ERR_CUDA);
        if (!(a_first ? col_blocks(t) : row_blocks(t))) return host_finish(hp, s, ws, st);
        if (t < P && t < Q && (st = block(t, t)) != GEMM_OK) return host_finish(hp, s, ws, st);
    }
    return host_finish(hp, s, ws, GEMM_OK);
}

extern "C" gemm_status softmax_rows_f32_host(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                                             void *stream)
{
    if (M < 0 || N < 0 || M > kMaxDim || N > kMaxDim || ldx < N || ldy < N) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!X || !Y || reinterpret_cast<uintptr_t>(X) % 4 || reinterpret_cast<uintptr_t>(Y) % 4) return GEMM_ERR_INVALID_ARG;
    if (X == Y && ldx != ldy) return GEMM_ERR_INVALID_ARG;
    DeviceInfo dev;
    gemm_status st = device_info(&dev);
    if (st != GEMM_OK) return st;
    cudaMemPool_t pool = nullptr;
    st = device_pool(&pool);
    if (st != GEMM_OK) return st;
    unsigned *err = nullptr;
    if (tct::error_word_address(&err) != cudaSuccess) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostPipe *hp = nullptr;
    st = host_pipe(&hp);
    if (st != GEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // One device matrix with 16-byte row pitches, softmaxed in place block by block.
    const int64_t nd = round_up(N, 4);
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(M * nd * 4), pool, s) != cudaSuccess) return GEMM_ERR_CUDA;
    float *dX = static_cast<float *>(ws);
    TCT_CUDA_OK(cudaEventRecord(hp->start, s));
    TCT_CUDA_OK(cudaStreamWaitEvent(hp->h2d, hp->start, 0));
    TCT_CUDA_OK(cudaStreamWaitEvent(hp->d2h, hp->start, 0));
    const int64_t rows = host_chunk_rows(M, 1);
    const uint64_t timeout_ns = static_cast<uint64_t>(kDefaultTimeoutMs) * 1000000ull;
    int j = 0;
    for (int64_t r0 = 0; r0 < M; r0 += rows, ++j) {
        const int64_t mr = std::min(rows, M - r0);
        TCT_CUDA_OK(cudaMemcpy2DAsync(dX + r0 * nd, nd * 4, X + r0 * ldx, ldx * 4, N * 4, mr, cudaMemcpyHostToDevice,
                                      hp->h2d));
        TCT_CUDA_OK(cudaEventRecord(hp->in[j], hp->h2d));
        TCT_CUDA_OK(cudaStreamWaitEvent(s, hp->in[j], 0));
        TCT_CUDA_OK(tct::launch_softmax_rows(dX + r0 * nd, dX + r0 * nd, mr, N, nd, nd, dev.sms, err, timeout_ns, s));
        TCT_CUDA_OK(cudaEventRecord(hp->out[j], s));
        TCT_CUDA_OK(cudaStreamWaitEvent(hp->d2h, hp->out[j], 0));
        TCT_CUDA_OK(cudaMemcpy2DAsync(Y + r0 * ldy, ldy * 4, dX + r0 * nd, nd * 4, N * 4, mr, cudaMemcpyDeviceToHost,
                                      hp->d2h));
    }
    return host_finish(hp, s, ws, GEMM_OK);
}
