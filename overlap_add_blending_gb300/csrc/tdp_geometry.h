// Tile geometry shared by the host planner and the kernels of libtdp.
// Pure integer arithmetic on a tdp_plan_t; no CUDA runtime calls.
#ifndef TDP_GEOMETRY_H_
#define TDP_GEOMETRY_H_

#include <stdint.h>

#include "tdp.h"

#if defined(__CUDACC__)
#define TDP_HD __host__ __device__ __forceinline__
#else
#define TDP_HD inline
#endif

namespace tdp {

TDP_HD int tile_size(const tdp_plan_t& p, int d, int i) { return p.end[d][i] - p.start[d][i]; }

// (i_f, i_h, i_w) of tile t; tiles are numbered frames-major.
TDP_HD void tile_coords(const tdp_plan_t& p, int t, int& i_f, int& i_h, int& i_w) {
    i_w = t % p.num_tiles[2];
    const int r = t / p.num_tiles[2];
    i_h = r % p.num_tiles[1];
    i_f = r / p.num_tiles[1];
}

// Sum of f*h*w volumes of all tiles numbered before (i_f, i_h, i_w).  With
// per-axis prefix sums P_d and totals S_d this is
//   P_f(i_f) S_h S_w + s_f(i_f) (P_h(i_h) S_w + s_h(i_h) P_w(i_w)).
TDP_HD int64_t tile_prefix_volume(const tdp_plan_t& p, int i_f, int i_h, int i_w) {
    const int64_t SH = p.prefix[1][p.num_tiles[1]];
    const int64_t SW = p.prefix[2][p.num_tiles[2]];
    const int64_t sf = tile_size(p, 0, i_f);
    const int64_t sh = tile_size(p, 1, i_h);
    return (int64_t)p.prefix[0][i_f] * SH * SW + sf * ((int64_t)p.prefix[1][i_h] * SW + sh * p.prefix[2][i_w]);
}

TDP_HD int64_t total_volume(const tdp_plan_t& p) {
    return (int64_t)p.prefix[0][p.num_tiles[0]] * p.prefix[1][p.num_tiles[1]] * p.prefix[2][p.num_tiles[2]];
}

// Tiles covering index x of axis d form the contiguous range [lo, hi]:
// starts are i * stride and ends never decrease.
TDP_HD void axis_cover(const tdp_plan_t& p, int d, int x, int& lo, int& hi) {
    const int n = p.num_tiles[d];
    int h = x / p.stride[d];
    if (h > n - 1) h = n - 1;
    int l = h;
    while (l > 0 && p.end[d][l - 1] > x) --l;
    lo = l;
    hi = h;
}

// Tiles of axis d that intersect [x0, x1): the contiguous range [lo, hi].
TDP_HD void axis_range_cover(const tdp_plan_t& p, int d, int x0, int x1, int& lo, int& hi) {
    int a, b;
    axis_cover(p, d, x0, lo, a);
    axis_cover(p, d, x1 - 1, b, hi);
    (void)a;
    (void)b;
}

#if defined(__CUDACC__)
// 1-D trapezoid of tile i on axis d at coordinate x (x inside the tile):
// rising ramp min(1, (x-a+1)/(o+1)) except on the first tile, falling ramp
// min(1, (e-x)/(o+1)) except on the last, multiplied.  IEEE fp32 division.
__device__ __forceinline__ float axis_weight(const tdp_plan_t& p, int d, int i, int x) {
    const float o1 = static_cast<float>(p.overlap[d] + 1);
    float up = 1.0f, dn = 1.0f;
    if (i > 0) up = fminf(1.0f, static_cast<float>(x - p.start[d][i] + 1) / o1);
    if (i < p.num_tiles[d] - 1) dn = fminf(1.0f, static_cast<float>(p.end[d][i] - x) / o1);
    return __fmul_rn(up, dn);
}
#endif

}  // namespace tdp

#endif  // TDP_GEOMETRY_H_
