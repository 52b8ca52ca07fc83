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
    float *C;
    int64_t ldc;
    int32_t M, N, K;
    int32_t num_m, num_n, num_kb, num_tiles;
    int32_t group_m;
    int32_t vec_store;  // 1 when C is 16-byte aligned and ldc % 4 == 0
    uint64_t timeout_ns;
};

// Compiled (cta_group, tile_n, stages) variants of the main kernel.  cta_group 1: 128 x
// tile_n tiles, one CTA each; per stage 16 KB of A + tile_n * 128 B of B.  cta_group 2:
// 256 x tile_n tiles on a CTA pair; per CTA and stage 16 KB of A + tile_n * 64 B of B.
// The epilogue staging takes 16 KB more.
#define TCT_VARIANTS(X) \
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

int variant_smem_bytes(int cta_group, int tile_n, int stages);

// Co-resident clusters of the variant on the current device (-1 if the query fails).
int variant_max_clusters(int cta_group, int tile_n, int stages);

cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const KernelParams &p, int cta_group,
                        int tile_n, int stages, int grid, cudaStream_t stream);

cudaError_t launch_pack(const void *src, int64_t ld_src, void *dst, int64_t ld_dst, int64_t rows,
                        int64_t cols, int num_sms, cudaStream_t stream);

cudaError_t launch_fill_zero(float *C, int64_t ldc, int64_t rows, int64_t cols, int num_sms,
                             cudaStream_t stream);

cudaError_t read_and_clear_error(unsigned *out);

}  // namespace tct
