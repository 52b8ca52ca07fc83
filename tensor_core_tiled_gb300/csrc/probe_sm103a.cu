// probe_sm103a.cu -- measures the dense FP16 tensor rate of one SM per clock.
//
// The roofline of the GEMM's main loop is the tensor core's rate, SMs x (FLOP per SM per
// clock) x SM clock.  This probe measures the per-clock factor on the device itself rather
// than taking it from a data sheet: every SM runs one CTA whose single issuing thread queues
// n back-to-back tcgen05.mma.kind::f16 instructions (M = 128, N = 256, K = 16, FP32
// accumulation in tensor memory; operands in shared memory in the same 128-byte-swizzled
// layouts the GEMM's k-blocks use), then waits for their completion through an mbarrier.
// The SM clock counter (clock64) read before the first issue and after the completion gives
// the cycles; FLOP = n x 2 x 128 x 256 x 16.  Operands are zeros: the rate per clock does
// not depend on the values (only the power drawn does).  The wait is bounded in wall time.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "ptx_sm103a.cuh"
#include "tensor_core_tiled.h"

namespace tct {
namespace {

constexpr int kProbeM = 128, kProbeN = 256, kProbeK = 16;
constexpr int kProbeA = kProbeM * 64 * 2;   // one 128 x 64 K-major FP16 tile (16 KB)
constexpr int kProbeB = 64 * kProbeN * 2;   // four 64 x 64 N-major FP16 boxes (32 KB)
// More than half of an SM's shared memory, so that no SM holds two probe CTAs.
constexpr int kProbeSmem = 120 * 1024;
constexpr int kProbeMaxCtas = 1024;

__device__ unsigned long long g_probe_cycles[kProbeMaxCtas];
__device__ unsigned int g_probe_status;

__global__ void __launch_bounds__(128, 1) tensor_rate_probe(int n_mma, uint64_t limit_ns)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + kProbeA;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + kProbeB);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 1);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (kProbeA + kProbeB) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kProbeN);
        tmem_relinquish();
    }
    fence_proxy_async_smem();  // the zeros (generic writes) before the tensor core reads them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = idesc_f32acc(kProbeM, kProbeN, false, true, false);
        const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
        const unsigned long long t0 = clock64();
        for (int i = 0; i < n_mma; ++i) {
            const int kk = i & 3;  // the four 16-deep steps of one 64-deep k-block, cycled
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_base + kk * 2048, 64 * 64 * 2, 1024);
            tc_mma_f16(tmem, adesc, bdesc, idesc, i > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(bar));
        const bool ok = mbar_wait(smem_u32(bar), 0, limit_ns);
        const unsigned long long t1 = clock64();
        g_probe_cycles[blockIdx.x] = ok ? t1 - t0 : 0ull;
        if (!ok) atomicExch(&g_probe_status, 1u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kProbeN);
}

}  // namespace
}  // namespace tct

extern "C" gemm_status gemm_tensor_rate_probe(int32_t n_mma, void *stream, double *flop_per_clk_sm,
                                              double *min_flop_per_clk_sm, double *max_flop_per_clk_sm)
{
    if (n_mma < 1 || n_mma > (1 << 22) || !flop_per_clk_sm) return GEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
    if (sms < 1 || sms > tct::kProbeMaxCtas) return GEMM_ERR_UNSUPPORTED_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned zero = 0;
    if (cudaFuncSetAttribute(tct::tensor_rate_probe, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tct::kProbeSmem) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(tct::g_probe_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    tct::tensor_rate_probe<<<sms, 128, tct::kProbeSmem, s>>>(n_mma, 2000000000ull);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    std::vector<unsigned long long> cycles(static_cast<size_t>(sms));
    unsigned status = 0;
    if (cudaMemcpyFromSymbolAsync(cycles.data(), tct::g_probe_cycles, sizeof(unsigned long long) * sms, 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&status, tct::g_probe_status, sizeof(status), 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (status != 0) return GEMM_ERR_DEVICE_TIMEOUT;
    const double flop = static_cast<double>(n_mma) * 2.0 * tct::kProbeM * tct::kProbeN * tct::kProbeK;
    std::vector<double> rate(static_cast<size_t>(sms));
    for (int i = 0; i < sms; ++i) {
        if (cycles[i] == 0) return GEMM_ERR_DEVICE_TIMEOUT;
        rate[i] = flop / static_cast<double>(cycles[i]);
    }
    std::sort(rate.begin(), rate.end());
    *flop_per_clk_sm = rate[rate.size() / 2];
    if (min_flop_per_clk_sm) *min_flop_per_clk_sm = rate.front();
    if (max_flop_per_clk_sm) *max_flop_per_clk_sm = rate.back();
    return GEMM_OK;
}
