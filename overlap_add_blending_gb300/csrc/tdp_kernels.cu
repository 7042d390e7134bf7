// Device side of libtdp (sm_103a): tile extract, trapezoid overlap-add,
// window sum, per-tile positions and conditioning-token selection.
//
// Data movement design (all paths are HBM-bound; nothing here is a dense
// contraction, so there are no tensor-core paths):
//   * One CTA owns one (b, c, frame, row-band) box of the LATENT.  Both
//     regions it moves are contiguous spans in global memory: the band of
//     full latent rows, and -- for every tile covering that box -- the run
//     of whole tile rows that falls inside the band (tile rows are packed
//     back to back).  Each span is staged into shared memory with one bulk
//     TMA copy (cp.async.bulk, 16-byte aligned body, mbarrier completion)
//     plus plain loads for its last partial 16 bytes.
//   * Extract writes the packed tile spans; blend reads them and writes the
//     latent band.  Blend is ordered by output: each output element is the
//     register sum of its <= 8 (under the guard) contributions, so there is
//     no zero-fill pass and no atomics.
//   * Shared memory is read with consecutive threads on consecutive
//     elements (conflict-free) and global memory is written with 32-bit
//     stores of element pairs (full 128-byte warp transactions).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>

#include "tdp.h"
#include "tdp_geometry.h"

namespace cg = cooperative_groups;

namespace tdp {
bool plan_is_valid(const tdp_plan_t* p);
}

namespace {

constexpr int kThreads = 256;
constexpr int kCluster = 8;                  // CTAs cooperating on one tile's token reduction
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;  // give up on staged copies after 200 ms
constexpr uint32_t kErrExtractWait = 1u;
constexpr uint32_t kErrBlendWait = 2u;
constexpr int kExtractSmemBudget = 48 * 1024;
constexpr int kBlendSmemBudget = 48 * 1024;

__device__ unsigned int g_device_error = 0;

thread_local int t_last_cuda_error = 0;

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Poll phase 0 of `bar` until it completes or kWaitNs of wall time pass.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar) {
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, 0)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// Bounded wait for the CTA's staged copies.  Returns true (uniformly over
// the CTA) when they have landed.  On a timeout the CTA records `code` in
// the diagnostic word, waits once more (bounded) so that no copy is still
// writing into its shared memory, and the caller returns without working.
__device__ bool mbar_wait_or_flag(uint64_t* bar, uint32_t code) {
    bool ok = mbar_wait_bounded(bar);
    const bool any_fail = __syncthreads_or(!ok);
    if (any_fail) {
        if (threadIdx.x == 0) atomicOr(&g_device_error, code);
        if (!ok) mbar_wait_bounded(bar);
        return false;
    }
    return true;
}

// ------------------------------------------------------------------ element helpers
__device__ __forceinline__ float load_f(const float* p, int i) { return p[i]; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p, int i) {
    const uint16_t bits = reinterpret_cast<const uint16_t*>(p)[i];
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
}
__device__ __forceinline__ uint16_t to_bits(__nv_bfloat16 v) { return __bfloat16_as_ushort(v); }

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

// ------------------------------------------------------------------ block / warp scans
__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Exclusive block scan of v; *total gets the block sum.  Uses 33 ints of `sh`.
__device__ int block_excl_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int incl = warp_incl_scan(v);
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nw ? sh[lane] : 0;
        const int wi = warp_incl_scan(w);
        if (lane < nw) sh[lane] = wi - w;
        if (lane == nw - 1) sh[32] = wi;
    }
    __syncthreads();
    const int r = sh[warp] + incl - v;
    *total = sh[32];
    __syncthreads();
    return r;
}

// =================================================================== K1: extract
struct ExtractSlot {
    long long dst;  // element index of the span in the packed tiles
    int src;        // shared-memory element index of (first row, column 0) of the tile
    int rows;       // tile rows inside the band
    int sw;         // tile width
    int pad;
};

struct ExtractArgs {
    const void* latent;
    void* tiles;
    int BC;          // B * C
    int band_rows;
    int nbands;
    int data_off;    // byte offset of the staged band in shared memory
};

template <typename E>
__device__ __forceinline__ void extract_copy_slot(const ExtractSlot& sl, const E* __restrict__ band,
                                                  E* __restrict__ tiles, int W) {
    const int len = sl.rows * sl.sw;
    E* dst = tiles + sl.dst;
    if constexpr (sizeof(E) == 2) {
        // Element pairs -> 32-bit stores; an odd span start leaves one head element.
        const int head = static_cast<int>(sl.dst & 1);
        const int npairs = (len - head) >> 1;
        if (threadIdx.x == 0 && head && len > 0) dst[0] = band[sl.src];
        if (threadIdx.x == blockDim.x - 1 && ((len - head) & 1)) {
            const int e = len - 1, row = e / sl.sw, x = e - row * sl.sw;
            dst[e] = band[sl.src + row * W + x];
        }
        int e0 = head + 2 * static_cast<int>(threadIdx.x);
        int row = e0 / sl.sw, x = e0 - row * sl.sw;
        const int step = 2 * static_cast<int>(blockDim.x);
        const int dq = step / sl.sw, dr = step - dq * sl.sw;
        uint32_t* dst32 = reinterpret_cast<uint32_t*>(dst + head);
        for (int j = threadIdx.x; j < npairs; j += blockDim.x) {
            const uint32_t lo = band[sl.src + row * W + x];
            int x1 = x + 1, row1 = row;
            if (x1 == sl.sw) { x1 = 0; ++row1; }
            const uint32_t hi = band[sl.src + row1 * W + x1];
            dst32[j] = lo | (hi << 16);
            x += dr;
            row += dq;
            if (x >= sl.sw) { x -= sl.sw; ++row; }
        }
    } else {
        int row = static_cast<int>(threadIdx.x) / sl.sw, x = static_cast<int>(threadIdx.x) - row * sl.sw;
        const int step = static_cast<int>(blockDim.x);
        const int dq = step / sl.sw, dr = step - dq * sl.sw;
        for (int j = threadIdx.x; j < len; j += blockDim.x) {
            dst[j] = band[sl.src + row * W + x];
            x += dr;
            row += dq;
            if (x >= sl.sw) { x -= sl.sw; ++row; }
        }
    }
}

template <typename E>
__global__ void __launch_bounds__(kThreads) extract_kernel(const __grid_constant__ tdp_plan_t p,
                                                           const ExtractArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    ExtractSlot* slots = reinterpret_cast<ExtractSlot*>(smem + 16);
    E* band = reinterpret_cast<E*>(smem + a.data_off);
    const E* latent = static_cast<const E*>(a.latent);
    E* tiles = static_cast<E*>(a.tiles);

    const int F = p.dims[0], H = p.dims[1], W = p.dims[2];
    int cta = blockIdx.x;
    const int bi = cta % a.nbands;
    cta /= a.nbands;
    const int f = cta % F;
    const int bc = cta / F;
    const int hb0 = bi * a.band_rows, hb1 = min(H, hb0 + a.band_rows);

    // The band [hb0, hb1) x [0, W) of plane (bc, f) is one contiguous span.
    const long long span0 = ((long long)bc * F + f) * H * W + (long long)hb0 * W;
    const int span_len = (hb1 - hb0) * W;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(latent + span0);
    const uintptr_t g1 = reinterpret_cast<uintptr_t>(latent + span0 + span_len);
    const uintptr_t lo = g0 & ~uintptr_t(15), mid = g1 & ~uintptr_t(15);
    const int shift = static_cast<int>((g0 - lo) / sizeof(E));
    const uint32_t bulk = mid > lo ? static_cast<uint32_t>(mid - lo) : 0u;

    if (threadIdx.x == 0) mbar_init(bar, 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, bulk);
        if (bulk) bulk_copy_g2s(band, reinterpret_cast<const void*>(lo), bulk, bar);
    }
    // Partial last 16 bytes: plain loads.
    {
        const int t0 = mid > g0 ? static_cast<int>((mid - g0) / sizeof(E)) : 0;
        for (int e = t0 + threadIdx.x; e < span_len; e += blockDim.x) band[shift + e] = latent[span0 + e];
    }
    // One slot per (covering frame tile, row tile meeting the band, column tile).
    int if_lo, if_hi, ih_lo, ih_hi;
    tdp::axis_cover(p, 0, f, if_lo, if_hi);
    tdp::axis_range_cover(p, 1, hb0, hb1, ih_lo, ih_hi);
    const int nw = p.num_tiles[2], NH = ih_hi - ih_lo + 1;
    const int nslots = (if_hi - if_lo + 1) * NH * nw;
    for (int s = threadIdx.x; s < nslots; s += blockDim.x) {
        const int iw = s % nw, jh = (s / nw) % NH, i_f = if_lo + s / (nw * NH), i_h = ih_lo + jh;
        const int sf = tdp::tile_size(p, 0, i_f), sh = tdp::tile_size(p, 1, i_h), sw = tdp::tile_size(p, 2, iw);
        const int r0 = max(p.start[1][i_h], hb0), r1 = min(p.end[1][i_h], hb1);
        const long long tile0 = (long long)a.BC * tdp::tile_prefix_volume(p, i_f, i_h, iw);
        ExtractSlot sl;
        sl.dst = tile0 + (((long long)bc * sf + (f - p.start[0][i_f])) * sh + (r0 - p.start[1][i_h])) * sw;
        sl.src = shift + (r0 - hb0) * W + p.start[2][iw];
        sl.rows = r1 - r0;
        sl.sw = sw;
        sl.pad = 0;
        slots[s] = sl;
    }
    __syncthreads();
    if (!mbar_wait_or_flag(bar, kErrExtractWait)) return;
    for (int s = 0; s < nslots; ++s) extract_copy_slot<E>(slots[s], band, tiles, W);
}

// =================================================================== K2: blend
struct Cov {
    int i;
    float w;
};

struct StageSlot {       // one staged run of tile rows
    long long src;       // element index in the packed tiles
    int len;             // elements
    int smem_off;        // byte offset inside the data region
};

struct BlendArgs {
    const void* tiles;
    void* out;
    int BC;
    int band_rows;
    int nbands;
    // shared-memory layout (bytes); computed on the host by blend_layout()
    int off_fcov, off_hcnt, off_hcov, off_wcnt, off_wcov, off_wtile, off_slotbase, off_stage, off_data;
    int kf, kh, kw;
};

struct BlendLayout {
    int off_fcov, off_hcnt, off_hcov, off_wcnt, off_wcov, off_wtile, off_slotbase, off_stage, off_data;
};

__host__ __device__ inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

BlendLayout blend_layout(int kf, int kh, int kw, int band_rows, int W, int nw, int max_slots) {
    BlendLayout L;
    int o = 16;  // mbarrier
    L.off_fcov = o; o = round_up(o + kf * (int)sizeof(Cov), 16);
    L.off_hcnt = o; o = round_up(o + band_rows * 4, 16);
    L.off_hcov = o; o = round_up(o + band_rows * kh * (int)sizeof(Cov), 16);
    L.off_wcnt = o; o = round_up(o + W * 4, 16);
    L.off_wcov = o; o = round_up(o + W * kw * (int)sizeof(Cov), 16);
    L.off_wtile = o; o = round_up(o + nw * 8, 16);
    L.off_slotbase = o; o = round_up(o + max_slots * 4, 16);
    L.off_stage = o; o = round_up(o + max_slots * (int)sizeof(StageSlot), 16);
    L.off_data = o;
    return L;
}

__device__ __forceinline__ void store_out(float* out, long long i, const float (&v)[1]) { out[i] = v[0]; }
__device__ __forceinline__ void store_out(__nv_bfloat16* out, long long i, const float (&v)[1]) {
    out[i] = __float2bfloat16_rn(v[0]);
}
__device__ __forceinline__ void store_out(__nv_bfloat16* out, long long i, const float (&v)[2]) {
    const uint32_t lo = to_bits(__float2bfloat16_rn(v[0]));
    const uint32_t hi = to_bits(__float2bfloat16_rn(v[1]));
    *reinterpret_cast<uint32_t*>(out + i) = lo | (hi << 16);
}
__device__ __forceinline__ void store_out(float* out, long long i, const float (&v)[2]) {
    *reinterpret_cast<float2*>(out + i) = make_float2(v[0], v[1]);
}

// U = output columns per thread item (2 when a pair store is aligned).
template <typename Tin, typename Tout, int U>
__global__ void __launch_bounds__(kThreads) blend_kernel(const __grid_constant__ tdp_plan_t p, const BlendArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    Cov* fcov = reinterpret_cast<Cov*>(smem + a.off_fcov);
    int* hcnt = reinterpret_cast<int*>(smem + a.off_hcnt);
    Cov* hcov = reinterpret_cast<Cov*>(smem + a.off_hcov);
    int* wcnt = reinterpret_cast<int*>(smem + a.off_wcnt);
    Cov* wcov = reinterpret_cast<Cov*>(smem + a.off_wcov);
    int2* wtile = reinterpret_cast<int2*>(smem + a.off_wtile);  // (start, size) per column tile
    int* slotbase = reinterpret_cast<int*>(smem + a.off_slotbase);
    StageSlot* stage = reinterpret_cast<StageSlot*>(smem + a.off_stage);
    unsigned char* data = smem + a.off_data;
    const Tin* tiles = static_cast<const Tin*>(a.tiles);
    Tout* out = static_cast<Tout*>(a.out);

    const int F = p.dims[0], H = p.dims[1], W = p.dims[2];
    int cta = blockIdx.x;
    const int bi = cta % a.nbands;
    cta /= a.nbands;
    const int f = cta % F;
    const int bc = cta / F;
    const int hb0 = bi * a.band_rows, hb1 = min(H, hb0 + a.band_rows);
    const int rows = hb1 - hb0;

    int if_lo, if_hi, ih_lo, ih_hi;
    tdp::axis_cover(p, 0, f, if_lo, if_hi);
    tdp::axis_range_cover(p, 1, hb0, hb1, ih_lo, ih_hi);
    const int nw = p.num_tiles[2], NH = ih_hi - ih_lo + 1, NF = if_hi - if_lo + 1;
    const int nslots = NF * NH * nw;

    if (threadIdx.x == 0) mbar_init(bar, 1);
    __syncthreads();

    if (threadIdx.x < 32) {
        // Warp 0: locate each slot's run of tile rows, lay the runs out in
        // shared memory (exclusive scan of their padded sizes), then issue
        // one bulk copy per run plus plain loads for its partial tail.
        const int lane = threadIdx.x;
        int carry = 0;
        for (int s0 = 0; s0 < nslots; s0 += 32) {
            const int s = s0 + lane;
            int padded = 0;
            StageSlot st;
            int r0 = 0, sw = 1;
            if (s < nslots) {
                const int iw = s % nw, jh = (s / nw) % NH, i_f = if_lo + s / (nw * NH), i_h = ih_lo + jh;
                const int sf = tdp::tile_size(p, 0, i_f), sh = tdp::tile_size(p, 1, i_h);
                sw = tdp::tile_size(p, 2, iw);
                r0 = max(p.start[1][i_h], hb0);
                const int r1 = min(p.end[1][i_h], hb1);
                const long long tile0 = (long long)a.BC * tdp::tile_prefix_volume(p, i_f, i_h, iw);
                st.src = tile0 + (((long long)bc * sf + (f - p.start[0][i_f])) * sh + (r0 - p.start[1][i_h])) * sw;
                st.len = (r1 - r0) * sw;
                padded = round_up(st.len * (int)sizeof(Tin), 16) + 16;
            }
            const int incl = warp_incl_scan(padded);
            if (s < nslots) {
                st.smem_off = carry + incl - padded;
                stage[s] = st;
                const uintptr_t g0 = reinterpret_cast<uintptr_t>(tiles + st.src);
                const uintptr_t lo = g0 & ~uintptr_t(15);
                // shared element index of (row r0, column 0) of this slot, minus r0*sw
                slotbase[s] = (st.smem_off + static_cast<int>(g0 - lo)) / (int)sizeof(Tin) - r0 * sw;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        // Total bytes the bulk copies will deliver.
        uint32_t mine = 0;
        for (int s = lane; s < nslots; s += 32) {
            const StageSlot st = stage[s];
            const uintptr_t g0 = reinterpret_cast<uintptr_t>(tiles + st.src);
            const uintptr_t g1 = reinterpret_cast<uintptr_t>(tiles + st.src + st.len);
            const uintptr_t lo = g0 & ~uintptr_t(15), mid = g1 & ~uintptr_t(15);
            if (mid > lo) mine += static_cast<uint32_t>(mid - lo);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
        if (lane == 0) mbar_arrive_expect_tx(bar, mine);
        __syncwarp();
        for (int s = lane; s < nslots; s += 32) {
            const StageSlot st = stage[s];
            const uintptr_t g0 = reinterpret_cast<uintptr_t>(tiles + st.src);
            const uintptr_t g1 = reinterpret_cast<uintptr_t>(tiles + st.src + st.len);
            const uintptr_t lo = g0 & ~uintptr_t(15), mid = g1 & ~uintptr_t(15);
            if (mid > lo) bulk_copy_g2s(data + st.smem_off, reinterpret_cast<const void*>(lo),
                                        static_cast<uint32_t>(mid - lo), bar);
            Tin* dst = reinterpret_cast<Tin*>(data + st.smem_off + (g0 - lo));
            const int t0 = mid > g0 ? static_cast<int>((mid - g0) / sizeof(Tin)) : 0;
            for (int e = t0; e < st.len; ++e) dst[e] = tiles[st.src + e];
        }
    } else {
        // Warps 1..: weight tables (ascending tile order on every axis).
        const int t = threadIdx.x - 32, nt = blockDim.x - 32;
        if (t == 0) {
            for (int i = if_lo; i <= if_hi; ++i) fcov[i - if_lo] = Cov{i, axis_weight(p, 0, i, f)};
        }
        for (int r = t; r < rows; r += nt) {
            int lo, hi;
            tdp::axis_cover(p, 1, hb0 + r, lo, hi);
            hcnt[r] = hi - lo + 1;
            for (int i = lo; i <= hi; ++i) hcov[r * a.kh + (i - lo)] = Cov{i, axis_weight(p, 1, i, hb0 + r)};
        }
        for (int c = t; c < W; c += nt) {
            int lo, hi;
            tdp::axis_cover(p, 2, c, lo, hi);
            wcnt[c] = hi - lo + 1;
            for (int i = lo; i <= hi; ++i) wcov[c * a.kw + (i - lo)] = Cov{i, axis_weight(p, 2, i, c)};
        }
        for (int i = t; i < nw; i += nt) wtile[i] = make_int2(p.start[2][i], tdp::tile_size(p, 2, i));
    }
    __syncthreads();
    if (!mbar_wait_or_flag(bar, kErrBlendWait)) return;

    const Tin* sdata = reinterpret_cast<const Tin*>(data);
    const int ncu = W / U;
    const long long out0 = ((long long)bc * F + f) * H * W + (long long)hb0 * W;
    const int items = rows * ncu;
    int r = static_cast<int>(threadIdx.x) / ncu, cu = static_cast<int>(threadIdx.x) - r * ncu;
    const int dq = static_cast<int>(blockDim.x) / ncu, dr = static_cast<int>(blockDim.x) - dq * ncu;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
        const int h = hb0 + r;
        float acc[U];
#pragma unroll
        for (int v = 0; v < U; ++v) acc[v] = 0.0f;
        const int hc = hcnt[r];
        for (int fa = 0; fa < NF; ++fa) {
            const float wf = fcov[fa].w;
            for (int k = 0; k < hc; ++k) {
                const Cov hk = hcov[r * a.kh + k];
                const float wfh = __fmul_rn(wf, hk.w);
                const int sbase = (fa * NH + (hk.i - ih_lo)) * nw;
#pragma unroll
                for (int v = 0; v < U; ++v) {
                    const int col = cu * U + v;
                    const int wc = wcnt[col];
                    for (int q = 0; q < wc; ++q) {
                        const Cov wq = wcov[col * a.kw + q];
                        const int2 wt = wtile[wq.i];
                        const int idx = slotbase[sbase + wq.i] + h * wt.y + (col - wt.x);
                        acc[v] = fmaf(__fmul_rn(wfh, wq.w), load_f(sdata, idx), acc[v]);
                    }
                }
            }
        }
        store_out(out, out0 + (long long)r * W + cu * U, acc);
        cu += dr;
        r += dq;
        if (cu >= ncu) { cu -= ncu; ++r; }
    }
}

// =================================================================== K3: window sum
__global__ void __launch_bounds__(kThreads) window_sum_kernel(const __grid_constant__ tdp_plan_t p,
                                                              float* max_abs_dev, float* sum_out) {
    const int F = p.dims[0], H = p.dims[1], W = p.dims[2];
    const long long N = (long long)F * H * W;
    float worst = 0.0f;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < N;
         idx += (long long)gridDim.x * blockDim.x) {
        const int w = static_cast<int>(idx % W);
        const long long fh = idx / W;
        const int h = static_cast<int>(fh % H), f = static_cast<int>(fh / H);
        int f0, f1, h0, h1, w0, w1;
        tdp::axis_cover(p, 0, f, f0, f1);
        tdp::axis_cover(p, 1, h, h0, h1);
        tdp::axis_cover(p, 2, w, w0, w1);
        // Same weights, products and summation order as the blend kernel
        // (products rounded on their own: never contracted into the sum).
        float S = 0.0f;
        for (int i = f0; i <= f1; ++i) {
            const float wf = axis_weight(p, 0, i, f);
            for (int j = h0; j <= h1; ++j) {
                const float wfh = __fmul_rn(wf, axis_weight(p, 1, j, h));
                for (int k = w0; k <= w1; ++k) S = __fadd_rn(S, __fmul_rn(wfh, axis_weight(p, 2, k, w)));
            }
        }
        if (sum_out) sum_out[idx] = S;
        worst = fmaxf(worst, fabsf(S - 1.0f));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, o));
    // Non-negative floats order like their bit patterns.
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(max_abs_dev), __float_as_uint(worst));
}

// =================================================================== K4 / K5: tokens
struct TileTokens {
    int f0, h0, w0, sf, sh, sw, n;
    long long prefix;  // sum of token counts of earlier tiles
};

__device__ __forceinline__ TileTokens tile_tokens(const tdp_plan_t& p, int t) {
    int i_f, i_h, i_w;
    tdp::tile_coords(p, t, i_f, i_h, i_w);
    TileTokens tt;
    tt.f0 = p.start[0][i_f];
    tt.h0 = p.start[1][i_h];
    tt.w0 = p.start[2][i_w];
    tt.sf = tdp::tile_size(p, 0, i_f);
    tt.sh = tdp::tile_size(p, 1, i_h);
    tt.sw = tdp::tile_size(p, 2, i_w);
    tt.n = tt.sf * tt.sh * tt.sw;
    tt.prefix = tdp::tile_prefix_volume(p, i_f, i_h, i_w);
    return tt;
}

// Global token index of tile-local token j.
__device__ __forceinline__ int global_token(const tdp_plan_t& p, const TileTokens& tt, int j) {
    const int x = j % tt.sw;
    const int r = j / tt.sw;
    const int y = r % tt.sh, k = r / tt.sh;
    return ((tt.f0 + k) * p.dims[1] + tt.h0 + y) * p.dims[2] + tt.w0 + x;
}

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Cluster-wide [min start, max end) of tile t's generated tokens, per axis.
// Each CTA of the cluster reduces a chunk of the tile's tokens; the chunks
// are combined through distributed shared memory.  ext_sh: 6 ints of this
// CTA's shared memory.  Leaves the result in ext[6]; a final cluster.sync
// by the caller must follow before any CTA exits.
__device__ void tile_extent_cluster(const tdp_plan_t& p, const TileTokens& tt, const int* gen, int b, long long N,
                                    int* ext_sh, int ext[6]) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int csize = static_cast<int>(cluster.num_blocks());
    if (threadIdx.x < 3) { ext_sh[2 * threadIdx.x] = INT_MAX; ext_sh[2 * threadIdx.x + 1] = INT_MIN; }
    __syncthreads();
    const int chunk = (tt.n + csize - 1) / csize;
    const int j0 = rank * chunk, j1 = min(tt.n, j0 + chunk);
    int mn[3] = {INT_MAX, INT_MAX, INT_MAX}, mx[3] = {INT_MIN, INT_MIN, INT_MIN};
    for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
        const long long n = global_token(p, tt, j);
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int2 v = *reinterpret_cast<const int2*>(gen + (((long long)b * 3 + d) * N + n) * 2);
            mn[d] = min(mn[d], v.x);
            mx[d] = max(mx[d], v.y);
        }
    }
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        mn[d] = warp_min(mn[d]);
        mx[d] = warp_max(mx[d]);
    }
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            atomicMin(&ext_sh[2 * d], mn[d]);
            atomicMax(&ext_sh[2 * d + 1], mx[d]);
        }
    }
    cluster.sync();
#pragma unroll
    for (int d = 0; d < 3; ++d) { ext[2 * d] = INT_MAX; ext[2 * d + 1] = INT_MIN; }
    for (int r = 0; r < csize; ++r) {
        const int* peer = cluster.map_shared_rank(ext_sh, r);
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            ext[2 * d] = min(ext[2 * d], peer[2 * d]);
            ext[2 * d + 1] = max(ext[2 * d + 1], peer[2 * d + 1]);
        }
    }
}

struct PositionsArgs {
    const int* gen;
    int* tile_pos;
    int* offsets;
    int B;
    int normalize;
};

__global__ void __launch_bounds__(kThreads) positions_kernel(const __grid_constant__ tdp_plan_t p,
                                                             const PositionsArgs a) {
    __shared__ int ext_sh[6];
    cg::cluster_group cluster = cg::this_cluster();
    const int tb = blockIdx.x / kCluster;
    const int t = tb / a.B, b = tb % a.B;
    const long long N = (long long)p.dims[0] * p.dims[1] * p.dims[2];
    const TileTokens tt = tile_tokens(p, t);
    int ext[6];
    tile_extent_cluster(p, tt, a.gen, b, N, ext_sh, ext);
    cluster.sync();  // every CTA has read its peers' partials
    const int rank = static_cast<int>(cluster.block_rank());
    if (rank == 0 && threadIdx.x < 3) a.offsets[((long long)t * a.B + b) * 3 + threadIdx.x] = ext[2 * threadIdx.x];
    const int chunk = (tt.n + kCluster - 1) / kCluster;
    const int j0 = rank * chunk, j1 = min(tt.n, j0 + chunk);
    int* dst = a.tile_pos + tt.prefix * 6 * a.B;
    for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
        const long long n = global_token(p, tt, j);
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            int2 v = *reinterpret_cast<const int2*>(a.gen + (((long long)b * 3 + d) * N + n) * 2);
            if (a.normalize) { v.x -= ext[2 * d]; v.y -= ext[2 * d]; }
            *reinterpret_cast<int2*>(dst + (((long long)b * 3 + d) * tt.n + j) * 2) = v;
        }
    }
}

struct CondArgs {
    const int* gen;
    const int* cond;
    int* extent;
    unsigned char* keep;
    int* kept_idx;
    int* num_kept;
    int* tile_cond;
    int B, M, normalize;
};

__device__ __forceinline__ bool cond_keep(const int* cond, int b, int M, int m, const int ext[6]) {
    const int2 t = *reinterpret_cast<const int2*>(cond + (((long long)b * 3 + 0) * M + m) * 2);
    if (t.x < 0) return true;  // negative time start: a reference token, kept everywhere
    bool ok = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        const int2 v = *reinterpret_cast<const int2*>(cond + (((long long)b * 3 + d) * M + m) * 2);
        ok = ok && (v.x < ext[2 * d + 1]) && (v.y > ext[2 * d]);
    }
    return ok;
}

__global__ void __launch_bounds__(kThreads) cond_kernel(const __grid_constant__ tdp_plan_t p, const CondArgs a) {
    __shared__ int ext_sh[6];
    __shared__ int scan_sh[33];
    __shared__ int kept_sh;
    cg::cluster_group cluster = cg::this_cluster();
    const int tb = blockIdx.x / kCluster;
    const int t = tb / a.B, b = tb % a.B;
    const long long N = (long long)p.dims[0] * p.dims[1] * p.dims[2];
    const TileTokens tt = tile_tokens(p, t);
    int ext[6];
    tile_extent_cluster(p, tt, a.gen, b, N, ext_sh, ext);
    const int rank = static_cast<int>(cluster.block_rank());
    if (rank == 0 && threadIdx.x < 6) a.extent[((long long)t * a.B + b) * 6 + threadIdx.x] = ext[threadIdx.x];

    const long long row = (long long)t * a.B + b;  // (t, b) row of keep / kept_idx
    const int chunk = (a.M + kCluster - 1) / kCluster;
    const int m0 = min(a.M, rank * chunk), m1 = min(a.M, m0 + chunk);
    // Pass 1: keep flags and this CTA's kept count.
    int mine = 0;
    for (int m = m0 + threadIdx.x; m < m1; m += blockDim.x) {
        const bool k = cond_keep(a.cond, b, a.M, m, ext);
        a.keep[row * a.M + m] = k ? 1 : 0;
        mine += k;
    }
    int total_cta;
    block_excl_scan(mine, scan_sh, &total_cta);
    if (threadIdx.x == 0) kept_sh = total_cta;
    cluster.sync();  // kept counts visible cluster-wide (also ends the extent reads)
    int before = 0, total = 0;
    for (int r = 0; r < kCluster; ++r) {
        const int c = *cluster.map_shared_rank(&kept_sh, r);
        if (r < rank) before += c;
        total += c;
    }
    // Pass 2: compacted indices and shifted positions, original order.
    if (a.kept_idx || a.tile_cond) {
        int base = before;
        for (int m00 = m0; m00 < m1; m00 += blockDim.x) {
            const int m = m00 + threadIdx.x;
            const bool k = (m < m1) && cond_keep(a.cond, b, a.M, m, ext);
            int round_total;
            const int pos = base + block_excl_scan(k ? 1 : 0, scan_sh, &round_total);
            if (k) {
                if (a.kept_idx) a.kept_idx[row * a.M + pos] = m;
                if (a.tile_cond) {
#pragma unroll
                    for (int d = 0; d < 3; ++d) {
                        int2 v = *reinterpret_cast<const int2*>(a.cond + (((long long)b * 3 + d) * a.M + m) * 2);
                        if (a.normalize) { v.x -= ext[2 * d]; v.y -= ext[2 * d]; }
                        *reinterpret_cast<int2*>(a.tile_cond + ((row * 3 + d) * a.M + pos) * 2) = v;
                    }
                }
            }
            base += round_total;
        }
        // Fill the slots after the last kept token: -1 indices, zero positions.
        const int fill = a.M - total;
        const int fchunk = (fill + kCluster - 1) / kCluster;
        const int q0 = total + min(fill, rank * fchunk), q1 = total + min(fill, (rank + 1) * fchunk);
        for (int q = q0 + threadIdx.x; q < q1; q += blockDim.x) {
            if (a.kept_idx) a.kept_idx[row * a.M + q] = -1;
            if (a.tile_cond) {
#pragma unroll
                for (int d = 0; d < 3; ++d)
                    *reinterpret_cast<int2*>(a.tile_cond + ((row * 3 + d) * a.M + q) * 2) = make_int2(0, 0);
            }
        }
    }
    if (rank == 0 && threadIdx.x == 0 && a.num_kept) a.num_kept[row] = total;
    cluster.sync();  // peers finished reading kept_sh
}

__global__ void __launch_bounds__(kThreads) cond_count_kernel(const unsigned char* keep, int T, int BM,
                                                              int* count, float* weight) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BM) return;
    int c = 0;
    for (int t = 0; t < T; ++t) c += keep[(long long)t * BM + i];
    count[i] = c;
    weight[i] = c ? 1.0f / static_cast<float>(c) : 0.0f;
}

// =================================================================== host helpers
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tdp_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TDP_OK;
    t_last_cuda_error = static_cast<int>(e);
    return TDP_ERR_CUDA;
}

int dtype_size(tdp_dtype d) { return d == TDP_F32 ? 4 : (d == TDP_BF16 ? 2 : 0); }

// Largest number of slots any (frame, band) box can have, for a band height.
int max_slots_for(const tdp_plan_t& p, int band_rows, int nbands) {
    int best = 0, nh_max = 0;
    for (int bi = 0; bi < nbands; ++bi) {
        int lo, hi;
        const int hb0 = bi * band_rows, hb1 = std::min(p.dims[1], hb0 + band_rows);
        tdp::axis_range_cover(p, 1, hb0, hb1, lo, hi);
        nh_max = std::max(nh_max, hi - lo + 1);
    }
    best = p.max_cover[0] * nh_max * p.num_tiles[2];
    return best;
}

int extract_smem(const tdp_plan_t& p, int band_rows, int esz, int* data_off) {
    const int nbands = (p.dims[1] + band_rows - 1) / band_rows;
    const int slots = max_slots_for(p, band_rows, nbands);
    *data_off = round_up(16 + slots * (int)sizeof(ExtractSlot), 16);
    const long long bytes = (long long)*data_off + round_up(band_rows * p.dims[2] * esz, 16) + 16;
    return bytes > INT_MAX ? INT_MAX : static_cast<int>(bytes);
}

// Exact shared-memory need of the blend for a band height: tables plus the
// largest sum of padded staged runs over all (frame, band) boxes.
int blend_smem(const tdp_plan_t& p, int band_rows, int esz, BlendLayout* L) {
    const int H = p.dims[1], W = p.dims[2], nw = p.num_tiles[2];
    const int nbands = (H + band_rows - 1) / band_rows;
    const int slots = max_slots_for(p, band_rows, nbands);
    *L = blend_layout(p.max_cover[0], p.max_cover[1], p.max_cover[2], band_rows, W, nw, slots);
    long long worst = 0;
    for (int f = 0; f < p.dims[0]; ++f) {
        int flo, fhi;
        tdp::axis_cover(p, 0, f, flo, fhi);
        for (int bi = 0; bi < nbands; ++bi) {
            const int hb0 = bi * band_rows, hb1 = std::min(H, hb0 + band_rows);
            int hlo, hhi;
            tdp::axis_range_cover(p, 1, hb0, hb1, hlo, hhi);
            long long sum = 0;
            for (int i_h = hlo; i_h <= hhi; ++i_h) {
                const int rows = std::min(p.end[1][i_h], hb1) - std::max(p.start[1][i_h], hb0);
                for (int iw = 0; iw < nw; ++iw)
                    sum += round_up(rows * tdp::tile_size(p, 2, iw) * esz, 16) + 16;
            }
            worst = std::max(worst, sum * (fhi - flo + 1));
        }
    }
    const long long bytes = L->off_data + worst;
    return bytes > INT_MAX ? INT_MAX : static_cast<int>(bytes);
}

template <typename K>
tdp_status set_smem(K kernel, int bytes) {
    if (bytes <= 48 * 1024) return TDP_OK;
    return cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
}

template <typename K, typename... Args>
tdp_status launch_cluster(K kernel, long long blocks, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, args...));
}

template <typename Tin, typename Tout>
tdp_status launch_blend(const tdp_plan_t& p, int BC, const void* tiles, void* out, cudaStream_t stream) {
    int band_rows = p.dims[1], smem = 0;
    BlendLayout L;
    for (;;) {
        smem = blend_smem(p, band_rows, (int)sizeof(Tin), &L);
        if (smem <= kBlendSmemBudget || band_rows == 1) break;
        band_rows = std::max(1, band_rows / 2);
    }
    if (smem > 200 * 1024) return TDP_ERR_UNSUPPORTED;
    const int nbands = (p.dims[1] + band_rows - 1) / band_rows;
    const long long blocks = (long long)BC * p.dims[0] * nbands;
    if (blocks > INT_MAX) return TDP_ERR_INVALID_ARG;
    BlendArgs a;
    a.tiles = tiles;
    a.out = out;
    a.BC = BC;
    a.band_rows = band_rows;
    a.nbands = nbands;
    a.off_fcov = L.off_fcov;
    a.off_hcnt = L.off_hcnt;
    a.off_hcov = L.off_hcov;
    a.off_wcnt = L.off_wcnt;
    a.off_wcov = L.off_wcov;
    a.off_wtile = L.off_wtile;
    a.off_slotbase = L.off_slotbase;
    a.off_stage = L.off_stage;
    a.off_data = L.off_data;
    a.kf = p.max_cover[0];
    a.kh = p.max_cover[1];
    a.kw = p.max_cover[2];
    // Pair stores need every output row to start on a 4-byte (bf16) or
    // 8-byte (fp32) boundary: W even.
    tdp_status st;
    if (p.dims[2] % 2 == 0) {
        if ((st = set_smem(blend_kernel<Tin, Tout, 2>, smem)) != TDP_OK) return st;
        blend_kernel<Tin, Tout, 2><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(p, a);
    } else {
        if ((st = set_smem(blend_kernel<Tin, Tout, 1>, smem)) != TDP_OK) return st;
        blend_kernel<Tin, Tout, 1><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(p, a);
    }
    return cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

tdp_status tdp_extract(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype, const void* latent,
                       void* tiles, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || C < 0) return TDP_ERR_INVALID_ARG;
    const int esz = dtype_size(dtype);
    if (!esz) return TDP_ERR_INVALID_ARG;
    if (B == 0 || C == 0) return TDP_OK;
    if (!latent || !tiles) return TDP_ERR_INVALID_ARG;
    if (!aligned16(latent) || !aligned16(tiles)) return TDP_ERR_ALIGNMENT;
    const tdp_plan_t& p = *plan;
    int band_rows = p.dims[1], data_off = 0, smem = 0;
    for (;;) {
        smem = extract_smem(p, band_rows, esz, &data_off);
        if (smem <= kExtractSmemBudget || band_rows == 1) break;
        band_rows = std::max(1, band_rows / 2);
    }
    if (smem > 200 * 1024) return TDP_ERR_UNSUPPORTED;
    const int nbands = (p.dims[1] + band_rows - 1) / band_rows;
    const long long blocks = (long long)B * C * p.dims[0] * nbands;
    if (blocks > INT_MAX || (long long)B * C > INT_MAX) return TDP_ERR_INVALID_ARG;
    ExtractArgs a{latent, tiles, B * C, band_rows, nbands, data_off};
    tdp_status st;
    if (esz == 2) {
        if ((st = set_smem(extract_kernel<uint16_t>, smem)) != TDP_OK) return st;
        extract_kernel<uint16_t><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(p, a);
    } else {
        if ((st = set_smem(extract_kernel<uint32_t>, smem)) != TDP_OK) return st;
        extract_kernel<uint32_t><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(p, a);
    }
    return cuda_status(cudaGetLastError());
}

tdp_status tdp_blend(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype in_dtype, const void* tiles,
                     tdp_dtype out_dtype, void* out, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || C < 0) return TDP_ERR_INVALID_ARG;
    if (!dtype_size(in_dtype) || !dtype_size(out_dtype)) return TDP_ERR_INVALID_ARG;
    if (B == 0 || C == 0) return TDP_OK;
    if (!tiles || !out) return TDP_ERR_INVALID_ARG;
    if (!aligned16(tiles) || !aligned16(out)) return TDP_ERR_ALIGNMENT;
    if ((long long)B * C > INT_MAX) return TDP_ERR_INVALID_ARG;
    const int BC = B * C;
    if (in_dtype == TDP_BF16 && out_dtype == TDP_BF16)
        return launch_blend<__nv_bfloat16, __nv_bfloat16>(*plan, BC, tiles, out, stream);
    if (in_dtype == TDP_BF16 && out_dtype == TDP_F32)
        return launch_blend<__nv_bfloat16, float>(*plan, BC, tiles, out, stream);
    if (in_dtype == TDP_F32 && out_dtype == TDP_BF16)
        return launch_blend<float, __nv_bfloat16>(*plan, BC, tiles, out, stream);
    return launch_blend<float, float>(*plan, BC, tiles, out, stream);
}

tdp_status tdp_window_sum(const tdp_plan_t* plan, float* max_abs_dev, float* sum_out, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || !max_abs_dev) return TDP_ERR_INVALID_ARG;
    if (!aligned16(max_abs_dev) || (sum_out && !aligned16(sum_out))) return TDP_ERR_ALIGNMENT;
    tdp_status st = cuda_status(cudaMemsetAsync(max_abs_dev, 0, sizeof(float), stream));
    if (st != TDP_OK) return st;
    const long long N = (long long)plan->dims[0] * plan->dims[1] * plan->dims[2];
    const long long blocks = std::min<long long>((N + kThreads - 1) / kThreads, 152LL * 8);
    window_sum_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(*plan, max_abs_dev, sum_out);
    return cuda_status(cudaGetLastError());
}

tdp_status tdp_positions(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos, int32_t normalize,
                         int32_t* tile_pos, int32_t* offsets, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0) return TDP_ERR_INVALID_ARG;
    if (B == 0) return TDP_OK;
    if (!gen_pos || !tile_pos || !offsets) return TDP_ERR_INVALID_ARG;
    if (!aligned16(gen_pos) || !aligned16(tile_pos) || !aligned16(offsets)) return TDP_ERR_ALIGNMENT;
    const long long blocks = (long long)kCluster * plan->total_tiles * B;
    if (blocks > INT_MAX) return TDP_ERR_INVALID_ARG;
    PositionsArgs a{gen_pos, tile_pos, offsets, B, normalize ? 1 : 0};
    return launch_cluster(positions_kernel, blocks, stream, *plan, a);
}

tdp_status tdp_cond_select(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos, int32_t M,
                           const int32_t* cond_pos, int32_t normalize, int32_t* tile_extent, uint8_t* keep,
                           int32_t* count, float* weight, int32_t* kept_idx, int32_t* num_kept,
                           int32_t* tile_cond_pos, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || M < 0) return TDP_ERR_INVALID_ARG;
    if (B == 0) return TDP_OK;
    if (!gen_pos || !tile_extent) return TDP_ERR_INVALID_ARG;
    if (M > 0 && (!cond_pos || !keep || !count || !weight)) return TDP_ERR_INVALID_ARG;
    const void* ptrs[] = {gen_pos, tile_extent, cond_pos, keep, count, weight, kept_idx, num_kept, tile_cond_pos};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return TDP_ERR_ALIGNMENT;
    const long long blocks = (long long)kCluster * plan->total_tiles * B;
    if (blocks > INT_MAX || (long long)B * M > INT_MAX) return TDP_ERR_INVALID_ARG;
    CondArgs a{gen_pos, cond_pos, tile_extent, keep, kept_idx, num_kept, tile_cond_pos, B, M, normalize ? 1 : 0};
    tdp_status st = launch_cluster(cond_kernel, blocks, stream, *plan, a);
    if (st != TDP_OK || M == 0) return st;
    const int BM = B * M;
    cond_count_kernel<<<(BM + kThreads - 1) / kThreads, kThreads, 0, stream>>>(keep, plan->total_tiles, BM, count,
                                                                              weight);
    return cuda_status(cudaGetLastError());
}

tdp_status tdp_device_error(uint32_t* code, int32_t clear) {
    if (!code) return TDP_ERR_INVALID_ARG;
    unsigned int v = 0;
    tdp_status st = cuda_status(cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)));
    if (st != TDP_OK) return st;
    *code = v;
    if (clear && v) {
        const unsigned int zero = 0;
        st = cuda_status(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)));
    }
    return st;
}

int32_t tdp_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"
