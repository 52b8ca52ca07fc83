// softmax_sm103a.cu -- fused row softmax, the second workload of the lecture pages
// ("06_triton_style.py", demo 3: one program reads a row once, keeps it on chip, and writes
// exp(x - max) / sum once -- MN reads and MN writes instead of the 5MN + 2M / 3MN + 2M of
// five separate kernels).  Bandwidth-bound: every variant reads each input once and writes
// each output once, except rows too long for shared memory, which are read twice.
//
//   * N <= 2048: one warp per row, the row held in registers (up to 16 float4 per lane).
//   * N <= 51200: one 256-thread CTA per row, the row staged in shared memory.
//   * longer rows: one CTA per row, an online pass for (max, sum) -- the running sum is
//     rescaled whenever the running maximum grows -- then a second pass that writes.
// Rows are walked by a persistent grid.  exp(-inf) = 0; a row holding a NaN, whose maximum
// is +inf, or that is all -inf has no finite softmax and is written as NaN.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "gemm_internal.h"

namespace tct {

namespace {

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

}  // namespace

cudaError_t launch_softmax_rows(const float *X, float *Y, int64_t M, int64_t N, int64_t ldx, int64_t ldy, int num_sms,
                                cudaStream_t stream)
{
    if (M <= 0 || N <= 0) return cudaSuccess;
    const int vec = (reinterpret_cast<uintptr_t>(X) % 16 == 0 && reinterpret_cast<uintptr_t>(Y) % 16 == 0 &&
                     ldx % 4 == 0 && ldy % 4 == 0)
                        ? 1
                        : 0;
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

}  // namespace tct
