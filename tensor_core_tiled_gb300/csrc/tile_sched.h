// tile_sched.h -- tile scheduler shared by the host planner and the device kernel.
//
// Launch order with grouping ("06_triton_style.py", matmul_kernel and demo 2): linear
// tile indices are cut into groups of `group_m` tile rows spanning every tile column;
// inside a group the index walks down the rows first, then across the columns, so the
// tiles that run at the same time touch a squarer patch of A-rows and B-columns and share
// them through L2.  group_m = 1 is plain row-major order.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TCT_HD __host__ __device__ __forceinline__
#else
#define TCT_HD inline
#endif

namespace tct {

struct TileCoord {
    int32_t m;  // tile row
    int32_t n;  // tile column
};

TCT_HD TileCoord tile_coord(int32_t t, int32_t num_m, int32_t num_n, int32_t group_m)
{
    const int32_t per_group = group_m * num_n;
    const int32_t group = t / per_group;
    const int32_t first_m = group * group_m;
    const int32_t rows_left = num_m - first_m;
    const int32_t group_rows = rows_left < group_m ? rows_left : group_m;
    const int32_t r = t - group * per_group;
    TileCoord c;
    c.m = first_m + r % group_rows;
    c.n = r / group_rows;
    return c;
}

TCT_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace tct
