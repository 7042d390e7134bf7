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
#include <vector>

#include "tdp.h"
#include "tdp_geometry.h"

namespace cg = cooperative_groups;

namespace tdp {
bool plan_is_valid(const tdp_plan_t* p);
}

namespace {

constexpr int kThreads = 256;
constexpr int kCluster = 8;                  // CTAs cooperating on one tile's token reduction
constexpr uint64_t kWaitNs = 1000ull * 1000 * 1000;  // give up on staged copies after 1 s
constexpr uint32_t kSuspendHintNs = 20000;           // a polling thread sleeps up to 20 us per try
constexpr uint32_t kBackoffNs = 200;                 // sleep between polls of a waiter off the critical path
// Bits of the device error word (tdp_device_error).
constexpr uint32_t kErrExtractWait = 1u;   // an extract kernel gave up waiting for its staged copies
constexpr uint32_t kErrBlendWait = 2u;     // a blend kernel gave up waiting
constexpr uint32_t kErrDrain = 4u;         // copies still in flight after a give-up did not land in time
constexpr uint32_t kErrIndex = 8u;         // (debug builds) an index check failed; the access was skipped

// Debug builds (TDP_DEBUG_CHECKS=1) check the global and shared indices of
// the hot kernels' accesses; release builds compile the checks away.
#ifndef TDP_DEBUG_CHECKS
#define TDP_DEBUG_CHECKS 0
#endif
constexpr bool kDebugChecks = TDP_DEBUG_CHECKS != 0;
constexpr int kExtractStages = 3;               // staged bands per extract CTA (2 in flight)
constexpr int kExtractSmemBudget = 64 * 1024;   // staged bands + slot table
constexpr int kBlendSmemBudget = 64 * 1024;     // ring of staged tile rows + tables (3 CTAs per SM)
constexpr int kBlendQueue = 4;                  // blend items staged ahead at most (the header holds 4 ring offsets)
constexpr int kMaxOrdered = 256;                // column units ordered on the host
constexpr int kBlendTabBudget = 6 * 1024;       // shared bytes for the per-CTA axis entries
constexpr int kBlendConsumers = 256;            // blend threads that compute (8 warps)
constexpr int kBlendThreads = kBlendConsumers + 32;   // + one producer warp

__device__ unsigned int g_device_error = 0;
// Scratch of tdp_extract_and_tokens_no_alloc (the partial token extents and
// arrival counters of one call): 64 KiB, one instance per device.
static __device__ __align__(256) int g_token_scratch[16384];

// Debug builds: records a failed index check (kErrIndex) and tells the
// caller to skip the access.  Release builds: always false, no code.
__device__ __forceinline__ bool index_bad(bool bad) {
    if constexpr (kDebugChecks) {
        if (bad) {
            atomicOr(&g_device_error, kErrIndex);
            return true;
        }
    }
    return false;
}

// Debug builds: a byte range outside [lo, hi) of some buffer.
__device__ __forceinline__ bool range_bad(const void* p, long long bytes, const void* lo, long long size) {
    if constexpr (kDebugChecks) {
        const char* a = static_cast<const char*>(p);
        const char* b = static_cast<const char*>(lo);
        return index_bad(bytes < 0 || a < b || a + bytes > b + size);
    }
    return false;
}

thread_local int t_last_cuda_error = 0;

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// After the last mbar_init of a CTA (once: each fence costs hundreds of
// cycles): makes the initialised barriers visible to the async proxy.
__device__ __forceinline__ void mbar_init_done() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}


__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The same copy for data read once: its lines go first when L2 needs room
// (evict_first policy), so that data a later kernel reads stays longer.
__device__ __forceinline__ void bulk_copy_g2s_once(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Poll phase `parity` of `bar` until it completes or kWaitNs of wall time pass.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// As mbar_wait_bounded, for a waiter off the critical path (a producer
// waiting for buffer space): it sleeps between polls so that it does not
// take issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        __nanosleep(kBackoffNs);
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// CTA-wide wait for a staged phase: thread 0 polls while the other warps sit
// in the hardware barrier (they take no issue slots).  The barrier also
// publishes everything the CTA wrote to shared memory before it.  Returns
// false, uniformly, if the copies did not land within kWaitNs.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity) {
    bool ok = true;
    if (threadIdx.x == 0) ok = mbar_wait_bounded(bar, parity);
    return !__syncthreads_or(!ok);
}

// Programmatic dependent launch.  Every kernel here is launched so that it
// may start while the previous kernel in the stream finishes; it lets its
// own dependents start early, and waits for the previous kernel to complete
// (and its memory to be visible) before the first global access that kernel
// could have produced or could still be reading.  Launched without the
// attribute, the wait returns at once.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// The plan is a __grid_constant__ kernel parameter; indexed reads of it with
// a different index in each lane are serialised by the constant cache, so
// every kernel first copies it into shared memory and reads that copy.
__device__ __forceinline__ void load_plan(tdp_plan_t* dst, const tdp_plan_t& src) {
    const int* from = reinterpret_cast<const int*>(&src);
    int* to = reinterpret_cast<int*>(dst);
    for (int i = threadIdx.x; i < static_cast<int>(sizeof(tdp_plan_t) / 4); i += blockDim.x) to[i] = from[i];
}

// ------------------------------------------------------------------ element helpers

using tdp::axis_weight;

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

// Thread groups that run a CTA-wide step: the whole CTA (barrier 0), or
// the first NT threads, whole warps, of a warp-specialised CTA (named
// barrier 1, which the remaining warps never use).  Threads of a group are
// threadIdx.x in [0, size()).
struct CtaGroup {
    __device__ static int size() { return static_cast<int>(blockDim.x); }
    __device__ static void sync() { __syncthreads(); }
};
template <int NT>
struct WarpsGroup {
    static_assert(NT % 32 == 0 && NT <= 1024, "whole warps");
    __device__ static constexpr int size() { return NT; }
    __device__ static void sync() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }
};

// Exclusive scan of v over the group; *total gets the group sum.  Uses 33
// ints of `sh`.
template <class G>
__device__ int group_excl_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = G::size() >> 5;
    const int incl = warp_incl_scan(v);
    if (lane == 31) sh[warp] = incl;
    G::sync();
    if (warp == 0) {
        const int w = lane < nw ? sh[lane] : 0;
        const int wi = warp_incl_scan(w);
        if (lane < nw) sh[lane] = wi - w;
        if (lane == nw - 1) sh[32] = wi;
    }
    G::sync();
    const int r = sh[warp] + incl - v;
    *total = sh[32];
    G::sync();
    return r;
}

// Exclusive block scan of v; *total gets the block sum.  Uses 33 ints of `sh`.
__device__ int block_excl_scan(int v, int* sh, int* total) { return group_excl_scan<CtaGroup>(v, sh, total); }

// =================================================================== staging
// A contiguous span [g0, g1) of a global buffer staged into shared memory:
// one bulk copy of the 16-byte chunks it touches, except that a chunk
// reaching past the buffer's last full 16 bytes (`limit`) is not copied in
// bulk -- those last elements are loaded one by one.  The shared region
// needs round_up(span bytes, 16) + 16 bytes.
struct SpanCopy {
    uintptr_t lo;    // first byte copied in bulk (16-byte aligned)
    uint32_t bulk;   // bytes copied in bulk (multiple of 16, may be 0)
    int shift;       // elements between the region start and g0
    int tail0;       // first span element not covered by the bulk copy
};

template <typename E>
__device__ __forceinline__ SpanCopy plan_span(const E* base, long long first, int len, uintptr_t limit) {
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(base + first);
    const uintptr_t g1 = reinterpret_cast<uintptr_t>(base + first + len);
    SpanCopy c;
    c.lo = g0 & ~uintptr_t(15);
    uintptr_t hi = (g1 + 15) & ~uintptr_t(15);
    if (hi > limit) hi = g1 & ~uintptr_t(15);
    c.bulk = hi > c.lo ? static_cast<uint32_t>(hi - c.lo) : 0u;
    c.shift = static_cast<int>((g0 - c.lo) / sizeof(E));
    c.tail0 = hi >= g1 ? len : (hi > g0 ? static_cast<int>((hi - g0) / sizeof(E)) : 0);
    return c;
}

// ------------------------------------------------------------------ element conversions
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ------------------------------------------------------------------ shared loads by address
// 32-bit shared-window byte addresses keep the hot loops' address math to
// one add per access.  Each load names memory as clobbered: without that,
// the compiler may treat the asm as touching no memory and move it across
// ordinary C++ stores to shared memory (tables a thread writes and then
// reads back), which volatile alone does not forbid.
extern __shared__ __align__(16) unsigned char tdp_dynamic_smem[];   // the CTA's dynamic shared memory

// Debug builds: a shared-window byte range outside the CTA's dynamic shared
// memory (every table and stage the kernels read by address lives there).
__device__ __forceinline__ bool smem_addr_bad(uint32_t addr, uint32_t bytes) {
    if constexpr (kDebugChecks) {
        uint32_t size;
        asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
        const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(tdp_dynamic_smem));
        return index_bad(addr < base || addr + bytes > base + size);
    }
    return false;
}

__device__ __forceinline__ int lds_s32(uint32_t addr) {
    if (smem_addr_bad(addr, 4)) return 0;
    int v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    if (smem_addr_bad(addr, 4)) return 0.0f;
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    if (smem_addr_bad(addr, 2)) return 0u;
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}
// One staged element as fp32 (bf16 is widened exactly).
__device__ __forceinline__ float lds_elem(uint32_t addr, const __nv_bfloat16*) {
    return __uint_as_float(lds_u16(addr) << 16);
}
__device__ __forceinline__ float lds_elem(uint32_t addr, const float*) { return lds_f32(addr); }
// A staged element as fp32, or +0 where the tile does not reach the column:
// a byte permute of the bf16 bits into the upper half (selector 0x1044) or
// of zeros (0x4444); fp32 elements use a select.
__device__ __forceinline__ float lds_masked(uint32_t addr, uint32_t sel, bool, const __nv_bfloat16*) {
    return __uint_as_float(__byte_perm(lds_u16(addr), 0u, sel));
}
__device__ __forceinline__ float lds_masked(uint32_t addr, uint32_t, bool in, const float*) {
    const float x = lds_f32(addr);
    return in ? x : 0.0f;
}

// =================================================================== work split
// Items are numbered (frame, band) major, then b * C + c, and every CTA of a
// persistent kernel takes one contiguous range of them: consecutive items
// share their frame and band, so the geometry built for one serves the
// next, and ranges differ in length by at most one item (the first
// n mod G ranges are one longer).
__device__ __forceinline__ void cta_item_range(int n_items, int& first, int& last) {
    const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    const int q = n_items / G, r = n_items - q * G;
    first = b * q + min(b, r);
    last = first + q + (b < r ? 1 : 0);
}

// Items of one (frame, band) group cost alike, but groups do not: a frame
// covered by two frame tiles stages and blends twice the tile rows.  The
// host tabulates, per group, the elements one item moves (the band's latent
// rows, plus the tile rows of every covering (frame tile, row tile, column
// tile)), and a CTA then takes the contiguous item range holding its equal
// share of the total.  groups == 0: equal item counts (cta_item_range).
constexpr int kCostGroups = 64;

struct ItemCosts {
    int groups;
    long long cum[kCostGroups + 1];   // B*C times the cost of one item of every group before g
};

// First item of CTA b's share: the first item whose cost-so-far reaches
// b / G of the total.
__device__ __forceinline__ int cost_share_start(const ItemCosts& ic, int BC, int n_items, int G, int b) {
    if (b >= G) return n_items;
    const long long target = (long long)b * ic.cum[ic.groups] / G;
    int g = 0;
    while (g + 1 < ic.groups && ic.cum[g + 1] <= target) ++g;
    const long long per = (ic.cum[g + 1] - ic.cum[g]) / BC;
    const long long j = (target - ic.cum[g] + per - 1) / per;
    return g * BC + static_cast<int>(j < BC ? j : BC);
}

__device__ __forceinline__ void cta_cost_range(const ItemCosts& ic, int BC, int n_items, int& first, int& last) {
    if (ic.groups == 0) return cta_item_range(n_items, first, last);
    const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    first = cost_share_start(ic, BC, n_items, G, b);
    last = cost_share_start(ic, BC, n_items, G, b + 1);
}

struct FrameBand {
    int f, hb0, hb1;
};

__device__ __forceinline__ FrameBand frame_band(const tdp_plan_t& p, int fb, int band_rows, int nbands) {
    FrameBand x;
    x.f = fb / nbands;
    x.hb0 = (fb - x.f * nbands) * band_rows;
    x.hb1 = min(p.dims[1], x.hb0 + band_rows);
    return x;
}

// Walks (fb, bc) = divmod(item, BC) without dividing per step.
struct ItemCursor {
    int fb, bc, BC;
    __device__ __forceinline__ void init(int item, int BC_) {
        BC = BC_;
        fb = item / BC;
        bc = item - fb * BC;
    }
    __device__ __forceinline__ void next() {
        if (++bc == BC) { bc = 0; ++fb; }
    }
};

// =================================================================== K1: extract
struct ExtractSlot {
    long long dst0;  // packed-tile element index of the slot's first element for b*C + c = 0
    long long vol;   // elements per (b, c) of the slot's tile: dst = dst0 + (b*C + c) * vol
    int src;         // band element index of (first row, column 0), before the staging shift
    int rows;        // tile rows inside the band
    int sw;          // tile width
    float inv_sw;    // 1 / sw, for the lanes' start (exact for the small numerators used)
};

struct ExtractArgs {
    const void* latent;
    void* tiles;
    long long latent_numel;
    long long tiles_numel;
    int BC;          // B * C
    int band_rows;
    int nbands;
    int n_items;     // F * nbands * B * C
    int off_slots;   // byte offsets in shared memory
    int off_data;    // stage s starts at off_data + s * stage_bytes
    int stage_bytes;
};

// floor(e / sw) for 0 <= e < 4096 via the rounded reciprocal: (e + 1/2) / sw
// is at least 1/(2 sw) away from an integer, far more than the error.
__device__ __forceinline__ int small_div(int e, float inv_sw) {
    return __float2int_rz((static_cast<float>(e) + 0.5f) * inv_sw);
}

// One warp copies one slot: the slot's rows (sw elements each, W apart in
// the staged band) are written back to back into the packed tile.  Lanes
// walk the output in steps of 64 elements (32 lanes x 2) for 2-byte types,
// 32 elements for 4-byte types, tracking the source index incrementally.
template <typename E>
__device__ __forceinline__ void extract_copy_slot_warp(E* __restrict__ dst, const E* __restrict__ src,
                                                       const ExtractSlot& e, int W, int lane, const E* tiles_lo,
                                                       long long tiles_n) {
    // (debug builds) every store of the slot stays inside the tile buffer
    auto bad = [&](const void* q, int bytes) { return range_bad(q, bytes, tiles_lo, tiles_n * (long long)sizeof(E)); };
    const int sw = e.sw;
    const int len = e.rows * sw;
    const int wrap = W - sw;
    if constexpr (sizeof(E) == 2) {
        const int head = static_cast<int>((reinterpret_cast<uintptr_t>(dst) >> 1) & 1);  // odd start
        const int body = len - head;
        const int npairs = body >> 1;
        if (lane == 0 && head && !bad(dst, 2)) dst[0] = src[0];
        if (lane == 31 && (body & 1)) {
            const int last = len - 1, row = last / sw;
            if (!bad(dst + last, 2)) dst[last] = src[row * W + (last - row * sw)];
        }
        const int e0 = head + 2 * lane;
        const int r0 = small_div(e0, e.inv_sw);
        int x = e0 - r0 * sw;
        const int dq = small_div(64, e.inv_sw), dr = 64 - dq * sw;
        // shared byte address of the pair's first element, and its steps
        uint32_t sa = smem_u32(src) + 2u * static_cast<uint32_t>(r0 * W + x);
        const uint32_t sstep = 2u * static_cast<uint32_t>(dq * W + dr), swrap = 2u * static_cast<uint32_t>(wrap);
        uint32_t* dp = reinterpret_cast<uint32_t*>(dst + head) + lane;
        const int nit = npairs > lane ? (npairs - lane + 31) >> 5 : 0;
        // one pass step on (x, sa), and one pair's word (its second element
        // may open the next row)
        auto advance = [&](int& xx, uint32_t& aa) {
            xx += dr;
            aa += sstep;
            if (xx >= sw) { xx -= sw; aa += swrap; }
        };
        auto pair = [&](int xx, uint32_t aa) {
            return lds_u16(aa) | (lds_u16(aa + (xx + 1 < sw ? 2u : 2u + swrap)) << 16);
        };
        int it = 0;
        // four passes per trip, positions stepped explicitly so that the
        // eight loads are in flight together (the loop itself stays rolled)
#pragma unroll 1
        for (; it + 3 < nit; it += 4) {
            int x1 = x, x2, x3;
            uint32_t a1 = sa, a2, a3;
            advance(x1, a1);
            x2 = x1; a2 = a1;
            advance(x2, a2);
            x3 = x2; a3 = a2;
            advance(x3, a3);
            const uint32_t w0 = pair(x, sa), w1 = pair(x1, a1), w2 = pair(x2, a2), w3 = pair(x3, a3);
            if (kDebugChecks && (bad(dp, 4) || bad(dp + 96, 4))) return;
            dp[0] = w0;
            dp[32] = w1;
            dp[64] = w2;
            dp[96] = w3;
            dp += 128;
            x = x3;
            sa = a3;
            advance(x, sa);
        }
#pragma unroll 1
        for (; it < nit; ++it) {
            if (bad(dp, 4)) return;
            *dp = pair(x, sa);
            dp += 32;
            advance(x, sa);
        }
    } else {
        const int r0 = small_div(lane, e.inv_sw);
        int x = lane - r0 * sw;
        int a = r0 * W + x;
        const int dq = small_div(32, e.inv_sw), dr = 32 - dq * sw;
        const int step = dq * W + dr;
#pragma unroll 4
        for (int j = lane; j < len; j += 32) {
            if (bad(dst + j, 4) || index_bad(a < 0)) return;
            dst[j] = src[a];
            x += dr;
            a += step;
            if (x >= sw) { x -= sw; a += wrap; }
        }
    }
}

// Persistent: each CTA walks its item range; an item is one (frame, row
// band, b, c) box of the latent, staged as one contiguous span.  A ring of
// `stages` shared-memory stages: thread 0 keeps the next stages - 1 items'
// bulk copies in flight while the CTA writes out the current one.
template <typename E>
__global__ void __launch_bounds__(kThreads, 5) extract_kernel(const __grid_constant__ tdp_plan_t pg,
                                                           const ExtractArgs a) {
    __shared__ tdp_plan_t p;
    pdl_launch_dependents();
    load_plan(&p, pg);
    __syncthreads();
    pdl_wait();   // latent (read) and tiles (written) may belong to the previous kernel
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    ExtractSlot* slots = reinterpret_cast<ExtractSlot*>(smem + a.off_slots);
    E* stage0 = reinterpret_cast<E*>(smem + a.off_data);
    const int stage_elems = a.stage_bytes / static_cast<int>(sizeof(E));
    constexpr int S = kExtractStages;
    const E* latent = static_cast<const E*>(a.latent);
    E* tiles = static_cast<E*>(a.tiles);
    const int F = p.dims[0], H = p.dims[1], W = p.dims[2], nw = p.num_tiles[2];
    const uintptr_t limit = reinterpret_cast<uintptr_t>(latent + a.latent_numel) & ~uintptr_t(15);

    int first, last;
    cta_item_range(a.n_items, first, last);
    if (first >= last) return;
    // thread 0 stages ahead with its own cursor
    ItemCursor ahead;
    ahead.init(first, a.BC);
    auto issue = [&](int s) {  // thread 0: stage the item under `ahead` into stage s
        const FrameBand x = frame_band(p, ahead.fb, a.band_rows, a.nbands);
        const long long span0 = ((long long)ahead.bc * F + x.f) * H * W + (long long)x.hb0 * W;
        const int len = (x.hb1 - x.hb0) * W;
        const SpanCopy cp = plan_span(latent, span0, len, limit);
        E* band = stage0 + s * stage_elems;
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar[s], cp.bulk);
        if (cp.bulk) bulk_copy_g2s(band, reinterpret_cast<const void*>(cp.lo), cp.bulk, &bar[s]);
        for (int e = cp.tail0; e < len; ++e) band[cp.shift + e] = latent[span0 + e];
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        mbar_init_done();
        for (int s = 0; s < S - 1 && first + s < last; ++s) {
            issue(s);
            ahead.next();
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    ItemCursor cur;
    cur.init(first, a.BC);
    int cached_fb = -1, nslots = 0, band_len = 0, f = 0, hb0 = 0;
    for (int k = 0, item = first, s = 0; item < last; ++k, ++item, cur.next(), s = (s + 1 == S ? 0 : s + 1)) {
        // stage (k - 1) mod S was freed by the barrier ending item k - 1
        if (threadIdx.x == 0 && item + S - 1 < last) {
            issue(s == 0 ? S - 1 : s - 1);
            ahead.next();
        }
        if (cur.fb != cached_fb) {
            // One slot per (covering frame tile, row tile meeting the band, column tile).
            const FrameBand x = frame_band(p, cur.fb, a.band_rows, a.nbands);
            f = x.f;
            hb0 = x.hb0;
            band_len = (x.hb1 - x.hb0) * W;
            int if_lo, if_hi, ih_lo, ih_hi;
            tdp::axis_cover(p, 0, x.f, if_lo, if_hi);
            tdp::axis_range_cover(p, 1, x.hb0, x.hb1, ih_lo, ih_hi);
            const int NH = ih_hi - ih_lo + 1;
            nslots = (if_hi - if_lo + 1) * NH * nw;
            for (int sl = threadIdx.x; sl < nslots; sl += blockDim.x) {
                const int iw = sl % nw, jh = (sl / nw) % NH, i_f = if_lo + sl / (nw * NH), i_h = ih_lo + jh;
                const int sf = tdp::tile_size(p, 0, i_f), sh = tdp::tile_size(p, 1, i_h), sw = tdp::tile_size(p, 2, iw);
                const int r0 = max(p.start[1][i_h], x.hb0), r1 = min(p.end[1][i_h], x.hb1);
                ExtractSlot e;
                e.vol = (long long)sf * sh * sw;
                e.dst0 = (long long)a.BC * tdp::tile_prefix_volume(p, i_f, i_h, iw) +
                         ((long long)(x.f - p.start[0][i_f]) * sh + (r0 - p.start[1][i_h])) * sw;
                e.src = (r0 - x.hb0) * W + p.start[2][iw];
                e.rows = r1 - r0;
                e.sw = sw;
                e.inv_sw = 1.0f / static_cast<float>(sw);
                slots[sl] = e;
            }
            cached_fb = cur.fb;
        }
        const long long span0 = ((long long)cur.bc * F + f) * H * W + (long long)hb0 * W;
        const int shift = plan_span(latent, span0, band_len, limit).shift;
        if (!cta_wait(&bar[s], (k / S) & 1)) {
            if (threadIdx.x == 0) {  // let every issued copy land before the CTA exits
                atomicOr(&g_device_error, kErrExtractWait);
                for (int j = k; j < k + S && first + j < last; ++j)
                    if (!mbar_wait_bounded(&bar[j % S], (j / S) & 1)) atomicOr(&g_device_error, kErrDrain);
            }
            return;
        }
        const E* band = stage0 + s * stage_elems + shift;
        for (int sl = warp; sl < nslots; sl += nwarps) {
            const ExtractSlot e = slots[sl];
            extract_copy_slot_warp<E>(tiles + e.dst0 + (long long)cur.bc * e.vol, band + e.src, e, W, lane, tiles,
                                      a.tiles_numel);
        }
        __syncthreads();  // stage s is free again; the slot table may be rebuilt
    }
}

// =================================================================== K2: blend
struct Cov {
    int i;
    float w;
};

struct StageSlot {      // one run of tile rows of a (frame, band) box, in bytes
    long long src0;     // offset in the packed tiles for b*C + c = 0
    long long vol;      // per (b, c) of the tile: offset = src0 + (b*C + c) * vol
    int len;            // bytes of the run
    int smem_off;       // offset inside an item's staged data
    int r0sw;           // first row of the run times the tile row
    int pad;
};

struct BlendArgs {
    const void* tiles;
    void* out;
    long long tiles_numel;
    int BC;
    int band_rows;
    int nbands;
    int n_items;
    // shared-memory layout (bytes), computed on the host; slotbase and data
    // have one copy per stage
    int off_a, off_b, off_c, off_d, off_e, off_stage, off_slotbase, off_data;
    int max_slots, data_bytes;
    int kf, kh, kw;
    int off_tab;   // fast kernel: axis entries (F + H + W of them), or -1: computed on demand
    // fast kernel: column units (U output columns each) in the order the
    // consumer threads take them -- fewest column tiles first -- when there
    // are at most kMaxOrdered units; otherwise the identity order
    int ordered;
    uint16_t order[kMaxOrdered];
    ItemCosts costs;   // fast kernel: the item split
};

__host__ __device__ inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

struct BlendBox {
    int f, hb0, hb1, rows, if_lo, if_hi, ih_lo, ih_hi, NF, NH, nslots;
};

__device__ __forceinline__ BlendBox blend_box(const tdp_plan_t& p, const BlendArgs& a, int fb) {
    BlendBox c;
    const FrameBand x = frame_band(p, fb, a.band_rows, a.nbands);
    c.f = x.f;
    c.hb0 = x.hb0;
    c.hb1 = x.hb1;
    c.rows = c.hb1 - c.hb0;
    tdp::axis_cover(p, 0, c.f, c.if_lo, c.if_hi);
    tdp::axis_range_cover(p, 1, c.hb0, c.hb1, c.ih_lo, c.ih_hi);
    c.NF = c.if_hi - c.if_lo + 1;
    c.NH = c.ih_hi - c.ih_lo + 1;
    c.nslots = c.NF * c.NH * p.num_tiles[2];
    return c;
}

// Warp 0: the staged runs of one (frame, band) box -- one per (covering
// frame tile, row tile meeting the band, column tile) -- and their layout
// in a stage's data region (exclusive scan of padded sizes).
template <typename Tin>
__device__ int blend_build_stage_table(const tdp_plan_t& p, const BlendArgs& a, const BlendBox& c,
                                       StageSlot* table) {
    const int lane = threadIdx.x & 31, nw = p.num_tiles[2];
    int carry = 0;
    for (int s0 = 0; s0 < c.nslots; s0 += 32) {
        const int s = s0 + lane;
        int padded = 0;
        StageSlot st;
        if (s < c.nslots) {
            const int iw = s % nw, jh = (s / nw) % c.NH, i_f = c.if_lo + s / (nw * c.NH), i_h = c.ih_lo + jh;
            const int sf = tdp::tile_size(p, 0, i_f), sh = tdp::tile_size(p, 1, i_h), sw = tdp::tile_size(p, 2, iw);
            const int r0 = max(p.start[1][i_h], c.hb0), r1 = min(p.end[1][i_h], c.hb1);
            constexpr int esz = static_cast<int>(sizeof(Tin));
            st.vol = (long long)sf * sh * sw * esz;
            st.src0 = ((long long)a.BC * tdp::tile_prefix_volume(p, i_f, i_h, iw) +
                       ((long long)(c.f - p.start[0][i_f]) * sh + (r0 - p.start[1][i_h])) * sw) * esz;
            st.len = (r1 - r0) * sw * esz;
            st.r0sw = r0 * sw * esz;
            st.pad = 0;
            padded = round_up(st.len, 16) + 16;
        }
        const int incl = warp_incl_scan(padded);
        if (s < c.nslots) {
            st.smem_off = carry + incl - padded;
            table[s] = st;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    return carry;   // bytes of one staged item
}

// One warp: stage item (box table, b*C + c) at byte `pos` of the data
// region.  Each lane takes runs s = lane, lane + 32, ...: it records the
// byte offset in the data region of the run's (row 0, column 0), loads
// with plain copies the part of a run in the buffer's last partial 16
// bytes, arrives on the barrier with its bulk bytes (the arrival releases
// those writes; the barrier counts 32 arrivals) and then issues its bulk
// copies.
template <typename Tin>
__device__ void blend_stage_item(const Tin* tiles, uintptr_t limit, const StageSlot* table, int nslots, int bc,
                                 int* slotbase, unsigned char* data, int pos, uint64_t* bar) {
    const int lane = threadIdx.x & 31;
    const uintptr_t base = reinterpret_cast<uintptr_t>(tiles);
    uint32_t bytes = 0;
    for (int s = lane; s < nslots; s += 32) {
        const StageSlot st = table[s];
        const uintptr_t g0 = base + st.src0 + (uintptr_t)bc * st.vol, g1 = g0 + st.len;
        const uintptr_t lo = g0 & ~uintptr_t(15);
        uintptr_t hi = (g1 + 15) & ~uintptr_t(15);
        if (hi > limit) {   // the tail past the last 16-byte boundary: plain copies
            hi = g1 & ~uintptr_t(15);
            const uintptr_t t0 = hi > g0 ? hi : g0;
            Tin* dst = reinterpret_cast<Tin*>(data + pos + st.smem_off + (t0 - lo));
            const Tin* src = reinterpret_cast<const Tin*>(t0);
            for (int e = 0; e < static_cast<int>((g1 - t0) / sizeof(Tin)); ++e) dst[e] = src[e];
        }
        bytes += hi > lo ? static_cast<uint32_t>(hi - lo) : 0u;
        slotbase[s] = pos + st.smem_off + static_cast<int>(g0 - lo) - st.r0sw;
    }
    fence_proxy_async();
    mbar_arrive_expect_tx(bar, bytes);
    for (int s = lane; s < nslots; s += 32) {
        const StageSlot st = table[s];
        const uintptr_t g0 = base + st.src0 + (uintptr_t)bc * st.vol, g1 = g0 + st.len;
        const uintptr_t lo = g0 & ~uintptr_t(15);
        uintptr_t hi = (g1 + 15) & ~uintptr_t(15);
        if (hi > limit) hi = g1 & ~uintptr_t(15);
        if (hi > lo)
            bulk_copy_g2s(data + pos + st.smem_off, reinterpret_cast<const void*>(lo), static_cast<uint32_t>(hi - lo), bar);
    }
}

// A thread's column tiles ("terms") for its output columns c .. c+U-1: the
// tiles covering any of them, each with the columns' offset into the tile
// row, the tile width, and per column the weight r_w and whether the tile
// reaches it.  Terms past the count are copies of the last one with no
// column reached (weight 0, value masked to 0), so every thread runs the
// same KT terms.
template <int U, int KT>
struct Terms {
    int n;                 // column tiles touching the columns (<= KT)
    int iw[KT], xo[KT], sw[KT];
    float w[KT][U];
    bool in[KT][U];
    uint32_t sel[KT][U];   // byte-permute selector: bf16 -> fp32 bits, or +0 where the tile does not reach
};

template <int U, int KT>
__device__ __forceinline__ void load_terms(const tdp_plan_t& p, int c, int W, Terms<U, KT>& t) {
    int lo, hi;
    tdp::axis_cover(p, 2, c, lo, hi);
#pragma unroll
    for (int v = 1; v < U; ++v) {
        if (c + v < W) {
            int l2, h2;
            tdp::axis_cover(p, 2, c + v, l2, h2);
            lo = min(lo, l2);
            hi = max(hi, h2);
        }
    }
    t.n = hi - lo + 1;
#pragma unroll
    for (int q = 0; q < KT; ++q) {
        const bool real = lo + q <= hi;
        const int i = min(lo + q, hi);
        const int w0 = p.start[2][i], w1 = p.end[2][i];
        t.iw[q] = i;
        t.sw[q] = w1 - w0;
        t.xo[q] = c - w0;
#pragma unroll
        for (int v = 0; v < U; ++v) {
            const bool in = real && c + v >= w0 && c + v < w1;
            t.in[q][v] = in;
            t.sel[q][v] = in ? 0x1044u : 0x4444u;
            t.w[q][v] = in ? axis_weight(p, 2, i, c + v) : 0.0f;
        }
    }
}


// Covering tiles of one index of an axis (at most two in the fast blend):
// the first one, their count, and their weights r(x).
struct AxisEnt {
    uint8_t lo, n, pad0, pad1;
    float w[2];
};

__device__ __forceinline__ AxisEnt axis_ent(const tdp_plan_t& p, int d, int x) {
    int lo, hi;
    tdp::axis_cover(p, d, x, lo, hi);
    AxisEnt e;
    e.lo = static_cast<uint8_t>(lo);
    e.n = static_cast<uint8_t>(hi - lo + 1);
    e.pad0 = e.pad1 = 0;
    e.w[0] = axis_weight(p, d, lo, x);
    e.w[1] = hi > lo ? axis_weight(p, d, lo + 1, x) : 0.0f;
    return e;
}

// The three axes' entries, tabulated once per CTA in shared memory (frames,
// then rows, then columns) when they fit; otherwise computed on demand.
struct AxisTabs {
    const AxisEnt* tab;   // nullptr: compute
    int hbase, wbase;
    __device__ __forceinline__ AxisEnt get(const tdp_plan_t& p, int d, int x) const {
        if (tab) return tab[(d == 0 ? 0 : (d == 1 ? hbase : wbase)) + x];
        return axis_ent(p, d, x);
    }
};

// load_terms from the column entries (same values: the entries hold the
// same axis_weight results).
template <int U, int KT>
__device__ __forceinline__ void load_terms_tab(const tdp_plan_t& p, const AxisTabs& at, int c, int W, Terms<U, KT>& t) {
    AxisEnt e[U];
#pragma unroll
    for (int v = 0; v < U; ++v) e[v] = at.get(p, 2, c + v < W ? c + v : c);
    int lo = e[0].lo, hi = e[0].lo + e[0].n - 1;
#pragma unroll
    for (int v = 1; v < U; ++v) {
        if (c + v < W) {
            lo = min(lo, static_cast<int>(e[v].lo));
            hi = max(hi, e[v].lo + e[v].n - 1);
        }
    }
    t.n = hi - lo + 1;
#pragma unroll
    for (int q = 0; q < KT; ++q) {
        const bool real = lo + q <= hi;
        const int i = min(lo + q, hi);
        const int w0 = p.start[2][i], w1 = p.end[2][i];
        t.iw[q] = i;
        t.sw[q] = w1 - w0;
        t.xo[q] = c - w0;
#pragma unroll
        for (int v = 0; v < U; ++v) {
            const bool in = real && c + v < W && c + v >= w0 && c + v < w1;
            t.in[q][v] = in;
            t.sel[q][v] = in ? 0x1044u : 0x4444u;
            t.w[q][v] = in ? e[v].w[i - e[v].lo] : 0.0f;
        }
    }
}

template <int U>
__device__ __forceinline__ void store_cols(float* out, long long i, const float (&v)[U]) {
    if constexpr (U == 2) *reinterpret_cast<float2*>(out + i) = make_float2(v[0], v[1]);
    else out[i] = v[0];
}
template <int U>
__device__ __forceinline__ void store_cols(__nv_bfloat16* out, long long i, const float (&v)[U]) {
    if constexpr (U == 2) {
        uint32_t b;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(v[1]), "f"(v[0]));
        *reinterpret_cast<uint32_t*>(out + i) = b;
    } else {
        out[i] = __float2bfloat16_rn(v[0]);
    }
}

// Band rows [r0, r1) of one (frame, band) box that share their list of
// (frame tile, row tile) pairs, in (frame tile, row tile) order.
struct __align__(16) Run {
    int r0, r1;
    int nc;             // pairs (1, 2 or 4)
    int ones;           // nc == 1 and r_f * r_h is exactly 1 on every row
    int slot0b[4];      // per pair: byte offset of its column tile 0's entry in the run-base table
};

// Band rows [r, r1) of run R for one thread's U columns with its first KTW
// column terms: per pair, inner = sum over terms of r_w * value, then
// acc = fma(w_fh, inner, acc) (acc = inner when every weight is 1:
// fma(1, inner, +0) is inner, which is never -0).  Shared addresses of
// every (pair, term) live in registers for the whole run.
template <int NC, int KTW, bool ONES, typename Tin, typename Tout, int U, int KT>
__device__ __forceinline__ void blend_run(const Run& R, int r, int r1, uint32_t sdata, uint32_t sbase, uint32_t wrow,
                                          int KC, const Terms<U, KT>& tm, const int (&colb)[KT],
                                          const int (&swb)[KT], const int (&iwb)[KT], int hb0, Tout* dcol, int W) {
    constexpr int esz = static_cast<int>(sizeof(Tin));
    uint32_t ea[NC][KTW];
#pragma unroll
    for (int kk = 0; kk < NC; ++kk)
#pragma unroll
        for (int q = 0; q < KTW; ++q)
            ea[kk][q] = sdata + lds_s32(sbase + R.slot0b[kk] + iwb[q]) + (hb0 + r) * swb[q] + colb[q];
    uint32_t wa = wrow + 4 * KC * r;
    Tout* dst = dcol + (long long)r * W;
    // One output row, `s` rows past the current pointers.
    auto row = [&](int s) {
        float acc[U];
#pragma unroll
        for (int v = 0; v < U; ++v) acc[v] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < NC; ++kk) {
            float inner[U];
#pragma unroll
            for (int v = 0; v < U; ++v) inner[v] = 0.0f;
#pragma unroll
            for (int q = 0; q < KTW; ++q)
#pragma unroll
                for (int v = 0; v < U; ++v) {
                    const float x = lds_masked(ea[kk][q] + s * swb[q] + v * esz, tm.sel[q][v], tm.in[q][v],
                                               static_cast<const Tin*>(nullptr));
                    inner[v] = fmaf(tm.w[q][v], x, inner[v]);
                }
            if constexpr (ONES) {
#pragma unroll
                for (int v = 0; v < U; ++v) acc[v] = inner[v];
            } else {
                const float wfh = lds_f32(wa + 4 * (s * KC + kk));
#pragma unroll
                for (int v = 0; v < U; ++v) acc[v] = fmaf(wfh, inner[v], acc[v]);
            }
        }
        store_cols<U>(dst, (long long)s * W, acc);
    };
    // Two rows per pass, written out (the loop itself stays rolled: an
    // unrolled form of the one-row loop gave wrong shared addresses on its
    // second iteration in some builds, found by the row-band parity test).
#pragma unroll 1
    for (; r + 1 < r1; r += 2) {
        row(0);
        row(1);
#pragma unroll
        for (int kk = 0; kk < NC; ++kk)
#pragma unroll
            for (int q = 0; q < KTW; ++q) ea[kk][q] += 2 * swb[q];
        wa += 8 * KC;
        dst += 2LL * W;
    }
    if (r < r1) row(0);
}

// A run of rows whose value is one tile's elements unchanged (one pair
// with w_fh = 1 and, on every column of every thread of the warp, one
// column tile with r_w = 1): the elements are copied.  The arithmetic path
// gives the same values except that it turns -0 into +0.
template <int U>
__device__ __forceinline__ void copy_row(uint32_t ea, __nv_bfloat16* dst) {
    if constexpr (U == 2) *reinterpret_cast<uint32_t*>(dst) = lds_u16(ea) | (lds_u16(ea + 2) << 16);
    else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(lds_u16(ea));
}
template <int U>
__device__ __forceinline__ void copy_row(uint32_t ea, float* dst) {
    if constexpr (U == 2) *reinterpret_cast<float2*>(dst) = make_float2(lds_f32(ea), lds_f32(ea + 4));
    else *dst = lds_f32(ea);
}
template <int U, typename T>
__device__ __forceinline__ void copy_run(const Run& R, int r, int r1, uint32_t sdata, uint32_t sbase, int colb,
                                         int swb, int iwb, int hb0, T* dcol, int W) {
    uint32_t ea = sdata + lds_s32(sbase + R.slot0b[0] + iwb) + (hb0 + r) * swb + colb;
    T* dst = dcol + (long long)r * W;
#pragma unroll 1
    for (; r < r1; ++r) {
        copy_row<U>(ea, dst);
        ea += swb;
        dst += W;
    }
}

// Blend for plans where at most two tiles cover any index on every axis
// (always the case under the guard: a tile holds at least twice the
// overlap, so tiles i and i+2 never meet).
//
// Persistent over a contiguous range of (frame, band, b, c) items, with
// one producer warp and kBlendConsumers consumer threads.  The producer
// keeps up to kBlendQueue items' tile rows in flight in a ring of shared
// memory (items differ in size: frames covered by two frame tiles stage
// twice the rows); per queue entry a "full" barrier completes when the
// item's bulk copies land and an "empty" barrier when every consumer warp
// is done with it.  A consumer thread owns U adjacent output columns for
// the whole run (U = 2, or 1 when W is odd) and KT column-tile terms for
// them.  The band's rows are split into runs that share their (frame tile,
// row tile) pairs, and into one contiguous block per row group, balanced
// by pair count.  Per pair and column the thread forms inner = sum over
// column tiles of r_w * value, then acc = fma(w_fh, inner, acc): the window
// product r_f r_h r_w grouped as w_fh * (r_w * value), in fp32, summed in
// the order (frame tile, row tile, column tile).
template <typename Tin, typename Tout, int U, int KT>
__global__ void __launch_bounds__(kBlendThreads, 3) blend_fast_kernel(const __grid_constant__ tdp_plan_t pg,
                                                                   const BlendArgs a) {
    __shared__ tdp_plan_t p;
    pdl_launch_dependents();
    load_plan(&p, pg);
    __syncthreads();
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);                  // [kBlendQueue]
    uint64_t* empty = full + kBlendQueue;                                // [kBlendQueue]
    uint64_t* csync = empty + kBlendQueue;                               // consumers only
    int* hdr = reinterpret_cast<int*>(smem + a.off_a);                   // run count, row-group bounds
    int* qstart = hdr + 12;                                              // [kBlendQueue] ring offsets
    Run* runs = reinterpret_cast<Run*>(smem + a.off_a + 64);
    float* wts = reinterpret_cast<float*>(smem + a.off_b);
    StageSlot* table = reinterpret_cast<StageSlot*>(smem + a.off_stage);
    int* slotbase0 = reinterpret_cast<int*>(smem + a.off_slotbase);
    unsigned char* data0 = smem + a.off_data;
    const Tin* tiles = static_cast<const Tin*>(a.tiles);
    Tout* out = static_cast<Tout*>(a.out);
    const int F = p.dims[0], H = p.dims[1], W = p.dims[2], nw = p.num_tiles[2];
    const int KC = a.kf * a.kh;
    const int max_slots = a.max_slots, ring = a.data_bytes;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kConsumerWarps = kBlendConsumers / 32;
    static_assert(kBlendQueue <= 4 && kConsumerWarps <= 8, "shared header: 12 ints of run count and row-group bounds, 4 ring offsets");

    int first, last;
    cta_cost_range(a.costs, a.BC, a.n_items, first, last);
    if (first >= last) return;
    const int n = last - first;
    if (threadIdx.x == 0) {
        for (int q = 0; q < kBlendQueue; ++q) {
            mbar_init(&full[q], 32);
            mbar_init(&empty[q], kConsumerWarps);
        }
        mbar_init(csync, kBlendConsumers);
        mbar_init_done();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---- producer.  Item k (k = item - first) uses queue entry
        // k mod kBlendQueue; items sit in the ring in order, item k at
        // qstart[k mod kBlendQueue]; kfree items are known released.
        const uintptr_t limit = reinterpret_cast<uintptr_t>(tiles + a.tiles_numel) & ~uintptr_t(15);
        int table_fb = -1, table_n = 0, table_bytes = 0, head = 0, kfree = 0;
        bool ok = true;
        ItemCursor ahead;
        ahead.init(first, a.BC);
        auto release = [&]() -> bool {   // wait for the oldest staged item to be released
            const bool r = mbar_wait_backoff(&empty[kfree % kBlendQueue], (kfree / kBlendQueue) & 1);
            ++kfree;
            return r;
        };
        int kst = 0;
        pdl_wait();   // the tiles may come from the previous kernel
        for (; kst < n && ok; ++kst, ahead.next()) {
            if (ahead.fb != table_fb) {
                const BlendBox cn = blend_box(p, a, ahead.fb);
                table_bytes = blend_build_stage_table<Tin>(p, a, cn, table);
                table_fb = ahead.fb;
                table_n = cn.nslots;
            }
            while (ok && kfree < kst - kBlendQueue + 1) ok = release();   // queue entry free
            int pos = 0;
            for (;;) {                                                     // ring room
                if (!ok) break;
                if (kfree == kst) { pos = 0; break; }                      // ring empty
                const int tail = qstart[kfree % kBlendQueue];
                if (head > tail) {
                    if (head + table_bytes <= ring) { pos = head; break; }
                    if (table_bytes <= tail) { pos = 0; break; }
                } else if (head < tail && head + table_bytes <= tail) {
                    pos = head;
                    break;
                }
                ok = release();
            }
            if (!ok) break;
            const int q = kst % kBlendQueue;
            if (lane == 0) qstart[q] = pos;
            __syncwarp();
            blend_stage_item(tiles, limit, table, table_n, ahead.bc, slotbase0 + q * max_slots, data0, pos, &full[q]);
            head = pos + table_bytes;
        }
        if (!ok) {
            // a consumer stopped: let every issued copy land, then leave
            if (lane == 0) atomicOr(&g_device_error, kErrBlendWait);
            for (int j = kfree; j < kst; ++j)
                if (!mbar_wait_bounded(&full[j % kBlendQueue], (j / kBlendQueue) & 1) && lane == 0)
                    atomicOr(&g_device_error, kErrDrain);
        }
        return;
    }

    // ---- consumers.  They meet (every thread arrives, then waits, bounded)
    // on `csync`; a wait that runs out stops the consumer, and the others
    // then run out too, since it never arrives again.
    uint32_t cphase = 0;
    auto consumer_sync = [&]() -> bool {
        mbar_arrive(csync);
        const bool r = mbar_wait_bounded(csync, cphase & 1);
        ++cphase;
        return r;
    };
    // A row group is the column units rounded up to whole
    // warps, so a warp stays on one row.  Column units are sorted by how
    // many column tiles they touch (fewest first) so that whole warps share
    // one term count.
    const int ncu = (W + U - 1) / U;
    const int per_row = min(round_up(ncu, 32), kBlendConsumers);
    const int RG = kBlendConsumers / per_row;   // 1 .. 8
    const int rg = static_cast<int>(threadIdx.x) / per_row;
    const int cu0 = static_cast<int>(threadIdx.x) - rg * per_row;
    const int ncu_mine = (rg < RG && cu0 < ncu) ? (ncu - cu0 + per_row - 1) / per_row : 0;
    auto unit_of = [&](int i) -> int { return a.ordered ? static_cast<int>(a.order[i]) : i; };
    AxisTabs at;
    at.tab = a.off_tab >= 0 ? reinterpret_cast<const AxisEnt*>(smem + a.off_tab) : nullptr;
    at.hbase = F;
    at.wbase = F + H;
    if (at.tab) {
        AxisEnt* tab = reinterpret_cast<AxisEnt*>(smem + a.off_tab);
        for (int i = threadIdx.x; i < F + H + W; i += kBlendConsumers)
            tab[i] = i < F ? axis_ent(p, 0, i) : (i < F + H ? axis_ent(p, 1, i - F) : axis_ent(p, 2, i - F - H));
        if (!consumer_sync()) return (void)atomicOr(&g_device_error, kErrBlendWait);
    }
    Terms<U, KT> tm;
    tm.n = 0;
    bool lane_copy = false;
    if (ncu_mine == 1) {
        load_terms_tab<U, KT>(p, at, unit_of(cu0) * U, W, tm);
        lane_copy = tm.n == 1 && sizeof(Tin) == sizeof(Tout);
#pragma unroll
        for (int v = 0; v < U; ++v) lane_copy = lane_copy && tm.in[0][v] && tm.w[0][v] == 1.0f;
    }
    // warp-uniform: term count (idle lanes count 0), and whether every
    // working lane may copy; wide rows take the general path
    const int kt_warp = __reduce_max_sync(0xffffffffu, ncu_mine > 1 ? KT : (ncu_mine == 1 ? tm.n : 0));
    const bool warp_copy = __all_sync(0xffffffffu, ncu_mine == 0 || (ncu_mine == 1 && lane_copy)) &&
                           __any_sync(0xffffffffu, ncu_mine == 1);

    ItemCursor cur;
    cur.init(first, a.BC);
    int box_fb = -1;
    BlendBox c{};
    int nruns = 0, rb0 = 0, rb1 = 0;
    pdl_wait();   // the previous kernel may still read `out`
    for (int k = 0; k < n; ++k, cur.next()) {
        if (cur.fb != box_fb) {
            // new (frame, band): rebuild the row tables once every consumer
            // is done with the old ones
            c = blend_box(p, a, cur.fb);
            box_fb = cur.fb;
            if (!consumer_sync()) return (void)atomicOr(&g_device_error, kErrBlendWait);
            // w_fh = r_f * r_h per band row and pair (frame tile major), one
            // row per thread
            {
                const AxisEnt ef = at.get(p, 0, c.f);   // ef.lo == c.if_lo, ef.n == c.NF
                for (int r = threadIdx.x; r < c.rows; r += kBlendConsumers) {
                    const AxisEnt eh = at.get(p, 1, c.hb0 + r);
                    int m = 0;
                    for (int fa = 0; fa < c.NF; ++fa)
                        for (int j = 0; j < eh.n; ++j) wts[r * KC + m++] = __fmul_rn(ef.w[fa], eh.w[j]);
                }
            }
            // runs: the rows between consecutive starts and ends of the row
            // tiles meeting the band (where the covering tiles change)
            if (threadIdx.x == 0) {
                const int nh = p.num_tiles[1];
                int lo, hi;
                tdp::axis_cover(p, 1, c.hb0, lo, hi);
                int h = c.hb0, nr = 0;
                while (h < c.hb1) {
                    int nxt = min(p.end[1][lo], c.hb1);
                    if (hi + 1 < nh) nxt = min(nxt, p.start[1][hi + 1]);
                    Run& R = runs[nr++];
                    R.r0 = h - c.hb0;
                    R.r1 = nxt - c.hb0;
                    R.nc = c.NF * (hi - lo + 1);
                    R.ones = 0;
                    int m = 0;
                    for (int fa = 0; fa < c.NF; ++fa)
                        for (int ih = lo; ih <= hi; ++ih) R.slot0b[m++] = 4 * (fa * c.NH + ih - c.ih_lo) * nw;
                    for (; m < 4; ++m) R.slot0b[m] = 0;
                    if (p.end[1][lo] == nxt) ++lo;
                    if (hi + 1 < nh && p.start[1][hi + 1] == nxt) ++hi;
                    h = nxt;
                }
                hdr[0] = nr;
            }
            if (!consumer_sync()) return (void)atomicOr(&g_device_error, kErrBlendWait);
            if (warp == 0) {
                const int nr = hdr[0];
                // a one-pair run is all ones when w_fh is 1 on its first and
                // last rows: r_h is a rising ramp times a falling one, each at
                // most 1, so it is 1 in between too
                for (int i = lane; i < nr; i += 32) {
                    Run& R = runs[i];
                    R.ones = R.nc == 1 && wts[R.r0 * KC] == 1.0f && wts[(R.r1 - 1) * KC] == 1.0f;
                }
                // row-group blocks: contiguous rows, split where the running
                // pair count crosses g / RG of the band's total (RG and nc are
                // powers of two)
                if (lane < RG) {
                    int b = lane == 0 ? 0 : c.rows;
                    if (lane > 0) {
                        int total = 0;
                        for (int i = 0; i < nr; ++i) total += runs[i].nc * (runs[i].r1 - runs[i].r0);
                        const int target = (total * lane + (RG >> 1)) >> (__ffs(RG) - 1);
                        int acc = 0;
                        for (int i = 0; i < nr; ++i) {
                            const int nc = runs[i].nc, len = runs[i].r1 - runs[i].r0;
                            if (acc + nc * len >= target) {
                                b = runs[i].r0 + min(len, max(0, (target - acc + nc - 1) >> (__ffs(nc) - 1)));
                                break;
                            }
                            acc += nc * len;
                        }
                    }
                    hdr[1 + lane] = b;
                }
                if (lane == 0) hdr[1 + RG] = c.rows;
            }
            if (!consumer_sync()) return (void)atomicOr(&g_device_error, kErrBlendWait);
            nruns = hdr[0];
            rb0 = rg < RG ? hdr[1 + rg] : 0;
            rb1 = rg < RG ? hdr[2 + rg] : 0;
        }
        const int q = k % kBlendQueue;
        if (!mbar_wait_bounded(&full[q], (k / kBlendQueue) & 1)) {
            if (lane == 0) atomicOr(&g_device_error, kErrBlendWait);
            return;   // no further releases: the producer gives up and drains its copies
        }
        const uint32_t sdata = smem_u32(data0);
        const uint32_t sbase = smem_u32(slotbase0 + q * max_slots);
        const uint32_t wrow = smem_u32(wts);
        constexpr int esz = static_cast<int>(sizeof(Tin));
        Tout* const out_band = out + ((long long)cur.bc * F + c.f) * H * W + (long long)c.hb0 * W;
        for (int m = 0; m < ncu_mine; ++m) {
            const int cu = unit_of(cu0 + m * per_row);
            if (ncu_mine > 1) load_terms_tab<U, KT>(p, at, cu * U, W, tm);
            // per term: byte offsets of the columns in the tile row, of one
            // tile row, and of the term's entry in the run-base table
            int colb[KT], swb[KT], iwb[KT];
#pragma unroll
            for (int t = 0; t < KT; ++t) {
                colb[t] = tm.xo[t] * esz;
                swb[t] = tm.sw[t] * esz;
                iwb[t] = 4 * tm.iw[t];
            }
            Tout* const dcol = out_band + cu * U;
            for (int ri = 0; ri < nruns; ++ri) {
                const Run R = runs[ri];
                const int r = max(R.r0, rb0), r1 = min(R.r1, rb1);
                if (r >= r1) continue;
                if constexpr (kDebugChecks) {
                    // the run's stores are affine in the row: its first and last row bound them all
                    const long long out_bytes = (long long)a.BC * F * H * W * (long long)sizeof(Tout);
                    if (range_bad(dcol + (long long)r * W, U * (int)sizeof(Tout), out, out_bytes) ||
                        range_bad(dcol + (long long)(r1 - 1) * W, U * (int)sizeof(Tout), out, out_bytes))
                        continue;
                }
                if (R.nc == 1) {
                    if (R.ones) {
                        if constexpr (sizeof(Tin) == sizeof(Tout)) {
                            if (warp_copy) {
                                copy_run<U>(R, r, r1, sdata, sbase, colb[0], swb[0], iwb[0], c.hb0, dcol, W);
                                continue;
                            }
                        }
                        if (kt_warp == 1)
                            blend_run<1, 1, true, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                        else
                            blend_run<1, KT, true, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                    } else if (kt_warp == 1) {
                        blend_run<1, 1, false, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                    } else {
                        blend_run<1, KT, false, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                    }
                } else if (R.nc == 2) {
                    if (kt_warp == 1)
                        blend_run<2, 1, false, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                    else
                        blend_run<2, KT, false, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                } else {
                    if (kt_warp == 1)
                        blend_run<4, 1, false, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                    else
                        blend_run<4, KT, false, Tin>(R, r, r1, sdata, sbase, wrow, KC, tm, colb, swb, iwb, c.hb0, dcol, W);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[q]);   // this warp is done with item k's rows and slot bases
    }
}

// Blend for any plan (guard-violating layouts can cover an index with more
// than two tiles per axis): one item per CTA, per-CTA cover tables in
// shared memory; same arithmetic grouping as the fast kernel.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads) blend_generic_kernel(const __grid_constant__ tdp_plan_t pg,
                                                                 const BlendArgs a) {
    __shared__ tdp_plan_t p;
    pdl_launch_dependents();
    load_plan(&p, pg);
    __syncthreads();
    pdl_wait();
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    Cov* fcov = reinterpret_cast<Cov*>(smem + a.off_a);
    int* hcnt = reinterpret_cast<int*>(smem + a.off_b);
    Cov* hcov = reinterpret_cast<Cov*>(smem + a.off_c);
    int* wcnt = reinterpret_cast<int*>(smem + a.off_d);
    Cov* wcov = reinterpret_cast<Cov*>(smem + a.off_e);
    StageSlot* table = reinterpret_cast<StageSlot*>(smem + a.off_stage);
    int* slotbase = reinterpret_cast<int*>(smem + a.off_slotbase);
    unsigned char* data = smem + a.off_data;
    const Tin* tiles = static_cast<const Tin*>(a.tiles);
    Tout* out = static_cast<Tout*>(a.out);
    const int F = p.dims[0], H = p.dims[1], W = p.dims[2], nw = p.num_tiles[2];
    const int fb = blockIdx.x / a.BC, bc = blockIdx.x - fb * a.BC;
    const BlendBox c = blend_box(p, a, fb);
    const uintptr_t limit = reinterpret_cast<uintptr_t>(tiles + a.tiles_numel) & ~uintptr_t(15);

    if (threadIdx.x == 0) {
        mbar_init(bar, 32);
        mbar_init_done();
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        blend_build_stage_table<Tin>(p, a, c, table);
        blend_stage_item(tiles, limit, table, c.nslots, bc, slotbase, data, 0, bar);
    } else {
        const int t = threadIdx.x - 32, nt = blockDim.x - 32;
        if (t == 0)
            for (int i = c.if_lo; i <= c.if_hi; ++i) fcov[i - c.if_lo] = Cov{i, axis_weight(p, 0, i, c.f)};
        for (int r = t; r < c.rows; r += nt) {
            int lo, hi;
            tdp::axis_cover(p, 1, c.hb0 + r, lo, hi);
            hcnt[r] = hi - lo + 1;
            for (int i = lo; i <= hi; ++i) hcov[r * a.kh + (i - lo)] = Cov{i, axis_weight(p, 1, i, c.hb0 + r)};
        }
        for (int col = t; col < W; col += nt) {
            int lo, hi;
            tdp::axis_cover(p, 2, col, lo, hi);
            wcnt[col] = hi - lo + 1;
            for (int i = lo; i <= hi; ++i) wcov[col * a.kw + (i - lo)] = Cov{i, axis_weight(p, 2, i, col)};
        }
    }
    if (!cta_wait(bar, 0)) {
        if (threadIdx.x == 0) {
            atomicOr(&g_device_error, kErrBlendWait);
            if (!mbar_wait_bounded(bar, 0)) atomicOr(&g_device_error, kErrDrain);
        }
        return;
    }

    const uint32_t sdata = smem_u32(data);
    const long long out0 = ((long long)bc * F + c.f) * H * W + (long long)c.hb0 * W;
    for (int it = threadIdx.x; it < c.rows * W; it += blockDim.x) {
        const int r = it / W, col = it - r * W, h = c.hb0 + r;
        float acc = 0.0f;
        for (int fa = 0; fa < c.NF; ++fa) {
            const float wf = fcov[fa].w;
            for (int k = 0; k < hcnt[r]; ++k) {
                const Cov hk = hcov[r * a.kh + k];
                const float wfh = __fmul_rn(wf, hk.w);
                const int sb = (fa * c.NH + (hk.i - c.ih_lo)) * nw;
                float inner = 0.0f;
                for (int q = 0; q < wcnt[col]; ++q) {
                    const Cov wq = wcov[col * a.kw + q];
                    const int off = slotbase[sb + wq.i] +
                                    (h * tdp::tile_size(p, 2, wq.i) + (col - p.start[2][wq.i])) * (int)sizeof(Tin);
                    inner = fmaf(wq.w, lds_elem(sdata + off, static_cast<const Tin*>(nullptr)), inner);
                }
                acc = fmaf(wfh, inner, acc);
            }
        }
        const float v[1] = {acc};
        store_cols<1>(out, out0 + it, v);
    }
}

// =================================================================== K3: window sum
// S(f,h,w) = sum over (frame tile, row tile) pairs of fma(r_f * r_h, inner(w), S)
// with inner(w) = sum over column tiles of r_w: the blend kernels' weights
// and grouping applied to tiles of ones, so S equals that blend bit for bit.
// With `tables`, each CTA first tabulates r_f and r_h per covering tile and
// inner(w) per column in shared memory (kf, kh: most tiles covering an index).
__global__ void __launch_bounds__(kThreads) window_sum_kernel(const __grid_constant__ tdp_plan_t p, float* max_abs_dev,
                                                              float* sum_out, int tables) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(16) unsigned char wsm[];
    const int F = p.dims[0], H = p.dims[1], W = p.dims[2];
    const int kf = p.max_cover[0], kh = p.max_cover[1];
    float* wf = reinterpret_cast<float*>(wsm);          // [F][kf]
    float* wh = wf + F * kf;                             // [H][kh]
    float* winner = wh + H * kh;                         // [W]
    int* fcnt = reinterpret_cast<int*>(winner + W);      // [F] covering frame tiles
    int* hcnt = fcnt + F;                                // [H]
    if (tables) {
        for (int f = threadIdx.x; f < F; f += blockDim.x) {
            int lo, hi;
            tdp::axis_cover(p, 0, f, lo, hi);
            fcnt[f] = hi - lo + 1;
            for (int i = lo; i <= hi; ++i) wf[f * kf + (i - lo)] = axis_weight(p, 0, i, f);
        }
        for (int h = threadIdx.x; h < H; h += blockDim.x) {
            int lo, hi;
            tdp::axis_cover(p, 1, h, lo, hi);
            hcnt[h] = hi - lo + 1;
            for (int i = lo; i <= hi; ++i) wh[h * kh + (i - lo)] = axis_weight(p, 1, i, h);
        }
        for (int w = threadIdx.x; w < W; w += blockDim.x) {
            int lo, hi;
            tdp::axis_cover(p, 2, w, lo, hi);
            float inner = 0.0f;
            for (int k = lo; k <= hi; ++k) inner = fmaf(axis_weight(p, 2, k, w), 1.0f, inner);
            winner[w] = inner;
        }
        __syncthreads();
    }
    const long long N = (long long)F * H * W;
    float worst = 0.0f;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < N;
         idx += (long long)gridDim.x * blockDim.x) {
        const int w = static_cast<int>(idx % W);
        const long long fh = idx / W;
        const int h = static_cast<int>(fh % H), f = static_cast<int>(fh / H);
        float S = 0.0f;
        if (tables) {
            const float in_w = winner[w];
            for (int i = 0; i < fcnt[f]; ++i) {
                const float a_f = wf[f * kf + i];
                for (int j = 0; j < hcnt[h]; ++j) S = fmaf(__fmul_rn(a_f, wh[h * kh + j]), in_w, S);
            }
        } else {
            int f0, f1, h0, h1, w0, w1;
            tdp::axis_cover(p, 0, f, f0, f1);
            tdp::axis_cover(p, 1, h, h0, h1);
            tdp::axis_cover(p, 2, w, w0, w1);
            float inner = 0.0f;
            for (int k = w0; k <= w1; ++k) inner = fmaf(axis_weight(p, 2, k, w), 1.0f, inner);
            for (int i = f0; i <= f1; ++i) {
                const float a_f = axis_weight(p, 0, i, f);
                for (int j = h0; j <= h1; ++j) S = fmaf(__fmul_rn(a_f, axis_weight(p, 1, j, h)), inner, S);
            }
        }
        if (sum_out) sum_out[idx] = S;
        worst = fmaxf(worst, fabsf(S - 1.0f));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, o));
    // Block maximum, then one atomic per block into the pre-zeroed result
    // (non-negative floats order like their bit patterns).
    __shared__ float warp_worst[kThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_worst[threadIdx.x >> 5] = worst;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.0f;
        for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, warp_worst[i]);
        atomicMax(reinterpret_cast<unsigned int*>(max_abs_dev), __float_as_uint(m));
    }
}

// Whether indices x and y of an axis have the same tuple of covering-tile
// weights (cnt: tiles per index, w: k weights per index).
__device__ __forceinline__ bool same_tuple(const int* cnt, const float* w, int k, int x, int y) {
    if (cnt[x] != cnt[y]) return false;
    for (int i = 0; i < cnt[x]; ++i)
        if (__float_as_uint(w[x * k + i]) != __float_as_uint(w[y * k + i])) return false;
    return true;
}

// Compacts the first index of every run of equal tuples on an axis of n
// indices into rep[]; returns the number of runs.  Whole group.
template <class G, typename Same>
__device__ int axis_runs(int n, int* rep, int* scan_sh, Same same) {
    int carry = 0;
    for (int x0 = 0; x0 < n; x0 += G::size()) {
        const int x = x0 + static_cast<int>(threadIdx.x);
        const int start = (x < n) && (x == 0 || !same(x, x - 1)) ? 1 : 0;
        int round_total;
        const int at = carry + group_excl_scan<G>(start, scan_sh, &round_total);
        if (start) rep[at] = x;
        carry += round_total;
    }
    G::sync();
    return carry;
}

// Shared bytes of window_max_group's tables and representatives.
inline long long window_max_bytes(const tdp_plan_t& p) {
    return 4LL * ((long long)p.dims[0] * p.max_cover[0] + (long long)p.dims[1] * p.max_cover[1] + p.dims[2] +
                  p.dims[0] + p.dims[1]) +
           4LL * ((long long)p.dims[0] + p.dims[1] + p.dims[2]);
}

// max |S - 1| over the volume by group G; the result is valid in thread 0.
// wsm: window_max_bytes(p) bytes; scan_sh: 33 ints; warp_worst: one float
// per warp of the group.
template <class G>
__device__ float window_max_group(const tdp_plan_t& p, unsigned char* wsm, int* scan_sh, float* warp_worst) {
    const int F = p.dims[0], H = p.dims[1], W = p.dims[2];
    const int kf = p.max_cover[0], kh = p.max_cover[1];
    const int tid = static_cast<int>(threadIdx.x), nthr = G::size();
    float* wf = reinterpret_cast<float*>(wsm);          // [F][kf]
    float* wh = wf + F * kf;                             // [H][kh]
    float* winner = wh + H * kh;                         // [W]
    int* fcnt = reinterpret_cast<int*>(winner + W);      // [F]
    int* hcnt = fcnt + F;                                // [H]
    int* frep = hcnt + H;                                // [F] run representatives
    int* hrep = frep + F;                                // [H]
    int* wrep = hrep + H;                                // [W]
    for (int f = tid; f < F; f += nthr) {
        int lo, hi;
        tdp::axis_cover(p, 0, f, lo, hi);
        fcnt[f] = hi - lo + 1;
        for (int i = lo; i <= hi; ++i) wf[f * kf + (i - lo)] = axis_weight(p, 0, i, f);
    }
    for (int h = tid; h < H; h += nthr) {
        int lo, hi;
        tdp::axis_cover(p, 1, h, lo, hi);
        hcnt[h] = hi - lo + 1;
        for (int i = lo; i <= hi; ++i) wh[h * kh + (i - lo)] = axis_weight(p, 1, i, h);
    }
    for (int w = tid; w < W; w += nthr) {
        int lo, hi;
        tdp::axis_cover(p, 2, w, lo, hi);
        float inner = 0.0f;
        for (int k = lo; k <= hi; ++k) inner = fmaf(axis_weight(p, 2, k, w), 1.0f, inner);
        winner[w] = inner;
    }
    G::sync();
    const int nf = axis_runs<G>(F, frep, scan_sh, [&](int x, int y) { return same_tuple(fcnt, wf, kf, x, y); });
    const int nh = axis_runs<G>(H, hrep, scan_sh, [&](int x, int y) { return same_tuple(hcnt, wh, kh, x, y); });
    const int nwc = axis_runs<G>(W, wrep, scan_sh,
                                 [&](int x, int y) { return __float_as_uint(winner[x]) == __float_as_uint(winner[y]); });
    float worst = 0.0f;
    for (int idx = tid; idx < nh * nwc; idx += nthr) {   // (row class, column class)
        const int hi = idx / nwc, h = hrep[hi];
        const float in_w = winner[wrep[idx - hi * nwc]];
        for (int fi = 0; fi < nf; ++fi) {
            const int f = frep[fi];
            float S = 0.0f;
            for (int i = 0; i < fcnt[f]; ++i) {
                const float a_f = wf[f * kf + i];
                for (int j = 0; j < hcnt[h]; ++j) S = fmaf(__fmul_rn(a_f, wh[h * kh + j]), in_w, S);
            }
            worst = fmaxf(worst, fabsf(S - 1.0f));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, o));
    if ((tid & 31) == 0) warp_worst[tid >> 5] = worst;
    G::sync();
    float m = 0.0f;
    if (tid == 0)
        for (int i = 0; i < (nthr >> 5); ++i) m = fmaxf(m, warp_worst[i]);
    return m;
}

// max |S - 1| alone (no per-element output), in one CTA.  S(f,h,w)
// depends on (f, h, w) only through each axis's tuple of covering-tile
// weights (for w: through inner(w)), and equal tuples give the same S bit
// for bit, so the maximum over the whole volume is the maximum over the
// triples of one representative index per run of equal tuples on each
// axis.  The tables are those of window_sum_kernel; the representatives
// follow them in shared memory.
__global__ void __launch_bounds__(kThreads) window_max_kernel(const __grid_constant__ tdp_plan_t p, float* max_abs_dev) {
    pdl_launch_dependents();
    extern __shared__ __align__(16) unsigned char wsm[];
    __shared__ int scan_sh[33];
    __shared__ float warp_worst[kThreads / 32];
    const float m = window_max_group<CtaGroup>(p, wsm, scan_sh, warp_worst);
    if (threadIdx.x == 0) {
        pdl_wait();   // the plan alone went in; the result may still be read by the previous kernel
        *max_abs_dev = m;
    }
    pdl_wait();       // finish after the previous kernel, so that finishing implies it finished
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

struct TokensArgs {
    const int* gen;
    int B, normalize;
    // positions (tile_pos NULL: not written)
    int* tile_pos;
    int* offsets;
    // conditioning selection (M = 0: none)
    int M;
    const int* cond;
    int* extent;
    unsigned char* keep;
    int* kept_idx;
    int* num_kept;
    int* tile_cond;
    int* slot_of;      // [T, B, M]: position in the tile's kept list, or -1 (NULL: not written)
};

constexpr int kPosCache = 4;   // tokens per thread kept in registers between reduce and write
constexpr int kCombineCols = 4;   // feature columns per lane per pass of the conditioning combine
constexpr int kCombineRound = 8;  // kept tiles of one token whose loads the combine issues together
constexpr int kCondOneCta = 2048;   // at most this many conditioning tokens: one CTA per tile tests them all

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

// Tile-local token j = (z, y, x) in a tile of sh rows of sw tokens, walked
// in steps of `step` tokens without a division per token.
struct TokenWalk {
    int x, y, z, sx, sy, sz;
    __device__ __forceinline__ void init(const TileTokens& tt, int j, int step) {
        x = j % tt.sw;
        const int r = j / tt.sw;
        y = r % tt.sh;
        z = r / tt.sh;
        sx = step % tt.sw;
        const int q = step / tt.sw;
        sy = q % tt.sh;
        sz = q / tt.sh;
    }
    __device__ __forceinline__ void next(const TileTokens& tt) {
        x += sx;
        y += sy;
        z += sz;
        if (x >= tt.sw) { x -= tt.sw; ++y; }
        if (y >= tt.sh) { y -= tt.sh; ++z; }
    }
    __device__ __forceinline__ long long token(const tdp_plan_t& p, const TileTokens& tt) const {
        return ((long long)(tt.f0 + z) * p.dims[1] + tt.h0 + y) * p.dims[2] + tt.w0 + x;
    }
};

// Keep test of a conditioning token already in registers (c[d] = [start,
// end) on axis d): a negative time start keeps it everywhere, else it must
// overlap the extent on every axis.
__device__ __forceinline__ bool keep_token(const int2 (&c)[3], const int ext[6]) {
    if (c[0].x < 0) return true;
    bool ok = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) ok = ok && (c[d].x < ext[2 * d + 1]) && (c[d].y > ext[2 * d]);
    return ok;
}

// One 8-CTA cluster per (tile, batch) does both token steps of the tile.
// Each CTA reads its chunk of the tile's generated tokens once (kept in
// registers, up to kPosCache per thread, when the positions are written),
// and the chunk minima of the starts and maxima of the ends meet through
// distributed shared memory: the tile's extent [TS, TE) per axis.  Then
// (positions) the CTA writes its chunk shifted by TS, and (conditioning)
// it tests its chunk of the conditioning tokens -- loaded before the
// reduction when the chunk fits one pass of the CTA -- against the extent,
// the chunks' kept counts meet through distributed shared memory, and it
// writes its kept tokens, compacted in their original order.  Every plan
// read here is uniform across the CTA, so the plan stays a parameter.
__global__ void __launch_bounds__(kThreads, 4) tokens_kernel(const __grid_constant__ tdp_plan_t p, const TokensArgs a) {
    __shared__ int ext_sh[6];
    __shared__ int scan_sh[33];
    __shared__ int kept_sh;
    pdl_launch_dependents();
    pdl_wait();   // positions may come from the previous kernel
    cg::cluster_group cluster = cg::this_cluster();
    const int tb = blockIdx.x / kCluster;
    const int t = tb / a.B, b = tb % a.B;
    const int nthr = static_cast<int>(blockDim.x);
    const long long N = (long long)p.dims[0] * p.dims[1] * p.dims[2];
    const TileTokens tt = tile_tokens(p, t);
    const int rank = static_cast<int>(cluster.block_rank());
    const int chunk = (tt.n + kCluster - 1) / kCluster;
    const int j0 = min(tt.n, rank * chunk), j1 = min(tt.n, j0 + chunk);
    const int* gen_b = a.gen + (long long)b * 3 * N * 2;
    const bool pos = a.tile_pos != nullptr;
    const bool cached = pos && chunk <= kPosCache * nthr;
    if (threadIdx.x < 6) ext_sh[threadIdx.x] = (threadIdx.x & 1) ? INT_MIN : INT_MAX;

    // Conditioning tokens: with at most kCondOneCta of them, cluster rank 0
    // tests all of them (no exchange of kept counts between the CTAs);
    // otherwise each CTA takes a chunk.  A CTA's tokens are loaded before
    // the extent reduction when they fit one pass of its threads.
    const bool solo = a.M <= kCondOneCta;
    const int mchunk = solo ? a.M : (a.M + kCluster - 1) / kCluster;
    const int m0 = solo ? 0 : min(a.M, rank * mchunk), m1 = solo ? (rank == 0 ? a.M : 0) : min(a.M, m0 + mchunk);
    const bool one_pass = m1 - m0 <= nthr;
    const int mm = m0 + static_cast<int>(threadIdx.x);
    const bool have_c = one_pass && mm < m1;
    int2 cv[3];
    if (have_c) {
#pragma unroll
        for (int d = 0; d < 3; ++d) cv[d] = *reinterpret_cast<const int2*>(a.cond + (((long long)b * 3 + d) * a.M + mm) * 2);
    }

    int2 v[kPosCache][3];
    int mn[3] = {INT_MAX, INT_MAX, INT_MAX}, mx[3] = {INT_MIN, INT_MIN, INT_MIN};
    TokenWalk tw;
    tw.init(tt, j0 + static_cast<int>(threadIdx.x), nthr);
    if (cached) {
#pragma unroll
        for (int k = 0; k < kPosCache; ++k) {
            const int j = j0 + static_cast<int>(threadIdx.x) + k * nthr;
            if (j < j1) {
                const long long n = tw.token(p, tt);
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    v[k][d] = *reinterpret_cast<const int2*>(gen_b + ((long long)d * N + n) * 2);
                    mn[d] = min(mn[d], v[k][d].x);
                    mx[d] = max(mx[d], v[k][d].y);
                }
            }
            tw.next(tt);
        }
    } else {
        for (int j = j0 + threadIdx.x; j < j1; j += nthr, tw.next(tt)) {
            const long long n = tw.token(p, tt);
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                const int2 x = *reinterpret_cast<const int2*>(gen_b + ((long long)d * N + n) * 2);
                mn[d] = min(mn[d], x.x);
                mx[d] = max(mx[d], x.y);
            }
        }
    }
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        mn[d] = warp_min(mn[d]);
        mx[d] = warp_max(mx[d]);
    }
    __syncthreads();  // ext_sh initialised
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            atomicMin(&ext_sh[2 * d], mn[d]);
            atomicMax(&ext_sh[2 * d + 1], mx[d]);
        }
    }
    cluster.sync();
    int ext[6];
#pragma unroll
    for (int d = 0; d < 3; ++d) { ext[2 * d] = INT_MAX; ext[2 * d + 1] = INT_MIN; }
    for (int r = 0; r < kCluster; ++r) {
        const int* peer = cluster.map_shared_rank(ext_sh, r);
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            ext[2 * d] = min(ext[2 * d], peer[2 * d]);
            ext[2 * d + 1] = max(ext[2 * d + 1], peer[2 * d + 1]);
        }
    }
    const long long row = (long long)t * a.B + b;  // (t, b) row of the per-tile outputs
    if (rank == 0 && threadIdx.x < 3 && a.offsets) a.offsets[row * 3 + threadIdx.x] = ext[2 * threadIdx.x];
    if (rank == 0 && threadIdx.x < 6 && a.extent) a.extent[row * 6 + threadIdx.x] = ext[threadIdx.x];

    // Conditioning pass 1: keep flags and this CTA's kept count, which meet
    // the other chunks' counts through distributed shared memory.
    int before = 0, total = 0, at_in = 0;
    bool kc = false;
    if (a.M > 0) {
        int total_cta;
        if (one_pass) {
            kc = have_c && keep_token(cv, ext);
            if (have_c) a.keep[row * a.M + mm] = kc ? 1 : 0;
            at_in = block_excl_scan(kc ? 1 : 0, scan_sh, &total_cta);
        } else {
            int mine = 0;
            for (int m = m0 + threadIdx.x; m < m1; m += nthr) {
                const bool k = cond_keep(a.cond, b, a.M, m, ext);
                a.keep[row * a.M + m] = k ? 1 : 0;
                mine += k;
            }
            block_excl_scan(mine, scan_sh, &total_cta);
        }
        if (solo) {
            total = total_cta;   // rank 0 holds every token; the other ranks hold none
        } else {
            if (threadIdx.x == 0) kept_sh = total_cta;
            cluster.sync();  // kept counts visible cluster-wide
            for (int r = 0; r < kCluster; ++r) {
                const int c = *cluster.map_shared_rank(&kept_sh, r);
                if (r < rank) before += c;
                total += c;
            }
        }
    }
    // Done reading the peers' shared memory; the matching wait ends the
    // kernel, so its latency overlaps the writes below.
    cluster.barrier_arrive();

    if (pos) {
        int off[3] = {ext[0], ext[2], ext[4]};
        if (!a.normalize) off[0] = off[1] = off[2] = 0;
        int* dst = a.tile_pos + tt.prefix * 6 * a.B + (long long)b * 3 * tt.n * 2;
        if (cached) {
#pragma unroll
            for (int k = 0; k < kPosCache; ++k) {
                const int j = j0 + static_cast<int>(threadIdx.x) + k * nthr;
                if (j < j1) {
#pragma unroll
                    for (int d = 0; d < 3; ++d)
                        *reinterpret_cast<int2*>(dst + ((long long)d * tt.n + j) * 2) =
                            make_int2(v[k][d].x - off[d], v[k][d].y - off[d]);
                }
            }
        } else {
            tw.init(tt, j0 + static_cast<int>(threadIdx.x), nthr);
            for (int j = j0 + threadIdx.x; j < j1; j += nthr, tw.next(tt)) {
                const long long n = tw.token(p, tt);
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    const int2 x = *reinterpret_cast<const int2*>(gen_b + ((long long)d * N + n) * 2);
                    *reinterpret_cast<int2*>(dst + ((long long)d * tt.n + j) * 2) =
                        make_int2(x.x - off[d], x.y - off[d]);
                }
            }
        }
    }

    // Conditioning pass 2: compacted indices and shifted positions, in the
    // original order; the slots after the last kept token get -1 / zeros.
    if (a.M > 0 && (a.kept_idx || a.tile_cond || a.slot_of)) {
        auto put = [&](int m, int at, int2 (&c)[3]) {
            if (a.kept_idx) a.kept_idx[row * a.M + at] = m;
            if (a.tile_cond) {
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    int2 q = c[d];
                    if (a.normalize) { q.x -= ext[2 * d]; q.y -= ext[2 * d]; }
                    *reinterpret_cast<int2*>(a.tile_cond + ((row * 3 + d) * a.M + at) * 2) = q;
                }
            }
        };
        if (one_pass) {
            if (kc) put(mm, before + at_in, cv);
            if (have_c && a.slot_of) a.slot_of[row * a.M + mm] = kc ? before + at_in : -1;
        } else {
            int base = before;
            for (int m00 = m0; m00 < m1; m00 += nthr) {
                const int m = m00 + threadIdx.x;
                const bool k = (m < m1) && cond_keep(a.cond, b, a.M, m, ext);
                int round_total;
                const int at = base + block_excl_scan(k ? 1 : 0, scan_sh, &round_total);
                if (m < m1 && a.slot_of) a.slot_of[row * a.M + m] = k ? at : -1;
                if (k) {
                    int2 c[3];
#pragma unroll
                    for (int d = 0; d < 3; ++d)
                        c[d] = *reinterpret_cast<const int2*>(a.cond + (((long long)b * 3 + d) * a.M + m) * 2);
                    put(m, at, c);
                }
                base += round_total;
            }
        }
        const int fill = a.M - total;
        const int fchunk = (fill + kCluster - 1) / kCluster;
        int q0 = total + min(fill, rank * fchunk), q1 = total + min(fill, (rank + 1) * fchunk);
        if (solo) { q0 = total; q1 = rank == 0 ? a.M : total; }
        for (int q = q0 + threadIdx.x; q < q1; q += nthr) {
            if (a.kept_idx) a.kept_idx[row * a.M + q] = -1;
            if (a.tile_cond) {
#pragma unroll
                for (int d = 0; d < 3; ++d)
                    *reinterpret_cast<int2*>(a.tile_cond + ((row * 3 + d) * a.M + q) * 2) = make_int2(0, 0);
            }
        }
    }
    if (rank == 0 && threadIdx.x == 0 && a.num_kept) a.num_kept[row] = total;   // 0 when M = 0 (rank 0 knows it)
    cluster.barrier_wait();  // no CTA leaves while a peer may read its shared memory

}

// count[i] = sum over tiles t of keep[t, i]; weight[i] = 1 / count[i] (IEEE
// fp32), 0 for a token no tile kept.
__device__ __forceinline__ void count_one(const unsigned char* keep, int T, int BM, int i, int* count, float* weight) {
    int c = 0;
    int t = 0;
    for (; t + 16 <= T; t += 16) {   // 16 independent loads in flight
        int k[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) k[u] = keep[(long long)(t + u) * BM + i];
#pragma unroll
        for (int u = 0; u < 16; ++u) c += k[u];
    }
    for (; t < T; ++t) c += keep[(long long)t * BM + i];
    count[i] = c;
    weight[i] = c ? 1.0f / static_cast<float>(c) : 0.0f;
}

__global__ void __launch_bounds__(kThreads) cond_count_kernel(const unsigned char* keep, int T, int BM,
                                                              int* count, float* weight) {
    pdl_launch_dependents();
    pdl_wait();   // the keep flags of the previous kernel
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < BM) count_one(keep, T, BM, i, count, weight);
}

// =================================================================== token steps in two launches
// tdp_extract_and_tokens splits the token steps at the extent: the extract
// launch reduces the partial extents of every (tile, batch) pair's K1 token
// chunks, spread over its CTAs (extent_chunk), and a second launch
// (tokens_finish_kernel) combines them and does the rest: positions,
// selection, counts and the window maximum.  Neither launch waits on
// another CTA; the partials pass through the caller's workspace.
constexpr int kJobTokenBatch = 4;   // tokens whose loads a thread keeps in flight
constexpr int kChunkShInts = 8;     // shared ints of an extent chunk
constexpr int kChunkTokens = 4 * 32 * 24;   // tokens of an extent chunk (one batch per extract compute thread)
constexpr int kFinishTokens = 4 * kThreads; // tokens of a finishing chunk (one batch per thread)

// Chunks of pair (t, b) in the extract launch (K1) and the finishing launch
// (K2): as many as the largest tile needs, so that a chunk is one batch.
inline int extent_chunks(const tdp_plan_t& p, int per_chunk) {
    long long n = 1;
    for (int t = 0; t < p.total_tiles; ++t) {
        int i_f, i_h, i_w;
        tdp::tile_coords(p, t, i_f, i_h, i_w);
        n = std::max(n, (long long)tdp::tile_size(p, 0, i_f) * tdp::tile_size(p, 1, i_h) * tdp::tile_size(p, 2, i_w));
    }
    return static_cast<int>((n + per_chunk - 1) / per_chunk);
}

// Chunks per (tile, batch) pair in the extract launch: one batch of loads
// per compute thread each, and at least as many chunks as spread the pairs
// over `grid` CTAs.
inline int extent_chunks_k1(const tdp_plan_t& p, long long J, int grid) {
    return std::max(extent_chunks(p, kChunkTokens), static_cast<int>(std::max(1LL, grid / std::max(1LL, J))));
}

// Tokens [j0, j1) of the tile's token walk: min start and max end per axis
// over this thread's share (j0 + thread, + G::size(), ...), kJobTokenBatch
// tokens' loads in flight.
template <class G>
__device__ __forceinline__ void extent_partial(const tdp_plan_t& p, const TileTokens& tt, const int* gen_b, long long N,
                                               int j0, int j1, int (&mn)[3], int (&mx)[3]) {
    const int nthr = G::size();
    TokenWalk tw;
    tw.init(tt, j0 + static_cast<int>(threadIdx.x), nthr);
    for (int j = j0 + static_cast<int>(threadIdx.x); j < j1; j += kJobTokenBatch * nthr) {
        long long n[kJobTokenBatch];
#pragma unroll
        for (int u = 0; u < kJobTokenBatch; ++u) {
            n[u] = j + u * nthr < j1 ? tw.token(p, tt) : -1;
            tw.next(tt);
        }
        int2 v[kJobTokenBatch][3];
#pragma unroll
        for (int u = 0; u < kJobTokenBatch; ++u)
            if (n[u] >= 0) {
#pragma unroll
                for (int d = 0; d < 3; ++d) v[u][d] = *reinterpret_cast<const int2*>(gen_b + ((long long)d * N + n[u]) * 2);
            }
#pragma unroll
        for (int u = 0; u < kJobTokenBatch; ++u)
            if (n[u] >= 0) {
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    mn[d] = min(mn[d], v[u][d].x);
                    mx[d] = max(mx[d], v[u][d].y);
                }
            }
    }
}

// Chunk q of the extract launch by group G: pair j = q / K1 = (tile j / B,
// batch j % B), part q % K1 of its token walk; writes its min start / max
// end per axis to partials[q] ((INT_MAX, INT_MIN) for an empty part).
// jsh: kChunkShInts ints of shared memory, free again on return.
template <class G>
__device__ void extent_chunk(const tdp_plan_t& p, const int* gen, int B, int K1, int q, int* partials, int* jsh) {
    const int tid = static_cast<int>(threadIdx.x);
    const int j = q / K1, c = q - j * K1, t = j / B, b = j - t * B;
    const long long N = (long long)p.dims[0] * p.dims[1] * p.dims[2];
    const TileTokens tt = tile_tokens(p, t);
    const int csz = (tt.n + K1 - 1) / K1;
    const int j0 = min(tt.n, c * csz), j1 = min(tt.n, j0 + csz);
    if (tid < 6) jsh[tid] = (tid & 1) ? INT_MIN : INT_MAX;
    int mn[3] = {INT_MAX, INT_MAX, INT_MAX}, mx[3] = {INT_MIN, INT_MIN, INT_MIN};
    extent_partial<G>(p, tt, gen + (long long)b * 3 * N * 2, N, j0, j1, mn, mx);
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        mn[d] = warp_min(mn[d]);
        mx[d] = warp_max(mx[d]);
    }
    G::sync();   // jsh initialised
    if ((tid & 31) == 0) {
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            atomicMin(&jsh[2 * d], mn[d]);
            atomicMax(&jsh[2 * d + 1], mx[d]);
        }
    }
    G::sync();
    if (tid < 6) partials[(long long)q * 6 + tid] = jsh[tid];
    G::sync();   // jsh is free for the next chunk
}

// The same reduction with its loads issued early: extent_chunk_issue copies
// the chunk's tokens (8 bytes per token and axis, plane-major) into shared
// memory with cp.async and returns at once; extent_chunk_finish, called
// later by every thread of the same group, reduces what each thread
// copied.  The copies' latency hides behind the caller's work in between.
// data: room for (chunk tokens) * 3 int2.
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}

struct ChunkSpan {
    int j0, j1;   // tokens [j0, j1) of the pair's token walk
};

__device__ __forceinline__ ChunkSpan chunk_span(const tdp_plan_t& p, int B, int K1, int q, TileTokens& tt, int& b) {
    const int j = q / K1, c = q - j * K1, t = j / B;
    b = j - t * B;
    tt = tile_tokens(p, t);
    const int csz = (tt.n + K1 - 1) / K1;
    ChunkSpan cs;
    cs.j0 = min(tt.n, c * csz);
    cs.j1 = min(tt.n, cs.j0 + csz);
    return cs;
}

template <class G>
__device__ void extent_chunk_issue(const tdp_plan_t& p, const int* gen, int B, int K1, int q, int2* data) {
    int b;
    TileTokens tt;
    const ChunkSpan cs = chunk_span(p, B, K1, q, tt, b);
    const long long N = (long long)p.dims[0] * p.dims[1] * p.dims[2];
    const int* gen_b = gen + (long long)b * 3 * N * 2;
    const int n = cs.j1 - cs.j0;
    TokenWalk tw;
    tw.init(tt, cs.j0 + static_cast<int>(threadIdx.x), G::size());
    for (int k = static_cast<int>(threadIdx.x); k < n; k += G::size(), tw.next(tt)) {
        const long long tok = tw.token(p, tt);
#pragma unroll
        for (int d = 0; d < 3; ++d) cp_async8(data + (long long)d * n + k, gen_b + ((long long)d * N + tok) * 2);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Thread-by-thread end of extent_chunk_issue: each thread waits for its own
// copies, reduces the tokens it copied, and its warp adds the result to
// partials[q] with atomic min / max -- no barrier, so the warps of the CTA
// finish independently.  partials[q] must hold (INT_MAX, INT_MIN) per axis
// before the first warp gets here (chunk_slot_init).
template <class G>
__device__ void extent_chunk_finish(const tdp_plan_t& p, int B, int K1, int q, const int2* data, int* partials) {
    int b;
    TileTokens tt;
    const ChunkSpan cs = chunk_span(p, B, K1, q, tt, b);
    const int n = cs.j1 - cs.j0;
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    int mn[3] = {INT_MAX, INT_MAX, INT_MAX}, mx[3] = {INT_MIN, INT_MIN, INT_MIN};
    for (int k = static_cast<int>(threadIdx.x); k < n; k += G::size()) {
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int2 v = data[(long long)d * n + k];
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
        int* slot = partials + (long long)q * 6;
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            if (mn[d] != INT_MAX) atomicMin(&slot[2 * d], mn[d]);
            if (mx[d] != INT_MIN) atomicMax(&slot[2 * d + 1], mx[d]);
        }
    }
}

// Sets partials[q] to (INT_MAX, INT_MIN) per axis (threads 0-5).
__device__ __forceinline__ void chunk_slot_init(int* partials, int q) {
    if (threadIdx.x < 6) partials[(long long)q * 6 + threadIdx.x] = (threadIdx.x & 1) ? INT_MIN : INT_MAX;
}

struct TokenFinishArgs {
    TokensArgs a;              // as tokens_kernel's
    int* count;                // [B*M] (M > 0): zeroed by the extract launch
    float* weight;             // [B*M] (M > 0)
    float* max_abs_dev;        // NULL: no window maximum
    const int* partials;       // [pairs * K1][6] from the extract launch
    int* arrivals;             // [B]: zeroed by the extract launch
    int K1, K2;                // chunks per pair: reduced by the extract launch / finished here
    int window_ctas;           // 1 with the window maximum (CTA 0), else 0
    int cond_ctas;             // pairs with M > 0, else 0: one conditioning CTA per pair
};

// Bytes of tokens_finish_kernel's dynamic shared memory: the window
// maximum's tables or a pair's partials, whichever is larger.
inline long long finish_smem(const tdp_plan_t& p, int K1, bool window) {
    return std::max(6LL * K1 * 4, window ? window_max_bytes(p) : 0LL);
}

// The pair's extent [TS, TE) per axis into ext_sh from its K1 partials,
// after the partial loads were issued into psh (threads < 6 * K1).
__device__ __forceinline__ void pair_extent(const int* psh, int K1, int* ext_sh) {
    __syncthreads();
    const int tid = static_cast<int>(threadIdx.x);
    if (tid < 6) {
        int e = (tid & 1) ? INT_MIN : INT_MAX;
        for (int k = 0; k < K1; ++k) e = (tid & 1) ? max(e, psh[k * 6 + tid]) : min(e, psh[k * 6 + tid]);
        ext_sh[tid] = e;
    }
    __syncthreads();
}

// The second launch of tdp_extract_and_tokens.  CTA roles by index:
//  * the window CTA (first, when asked for): max |S - 1| as
//    window_max_kernel computes it, from the plan alone, so it runs before
//    the wait for the extract launch and stores after it;
//  * conditioning CTAs (one per pair, with M > 0): the pair's extent from
//    its partials, the keep flags and kept lists as tokens_kernel computes
//    them, each kept token added to its count (zeroed by the extract
//    launch); the batch's last pair to finish (an arrival counter, also
//    zeroed by the extract launch) then writes the batch's weights
//    1 / count (IEEE fp32), so count equals the sum of the keep flags;
//  * chunk CTAs (pairs * K2): the pair's extent, the pair's offsets and
//    extent (part 0) and its part of the shifted positions, one batch of
//    loads per thread issued together with the partial loads.
__global__ void __launch_bounds__(kThreads, 1) tokens_finish_kernel(const __grid_constant__ tdp_plan_t p,
                                                                 const __grid_constant__ TokenFinishArgs f) {
    extern __shared__ __align__(16) unsigned char fsm[];
    __shared__ int scan_sh[33];
    __shared__ float warp_worst[kThreads / 32];
    __shared__ int ext_sh[6];
    __shared__ int last_sh;
    pdl_launch_dependents();
    const TokensArgs& a = f.a;
    const int tid = static_cast<int>(threadIdx.x);
    int blk = static_cast<int>(blockIdx.x);
    if (blk < f.window_ctas) {
        const float m = window_max_group<CtaGroup>(p, fsm, scan_sh, warp_worst);
        pdl_wait();   // the result may still be read by an earlier kernel
        if (tid == 0) *f.max_abs_dev = m;
        return;
    }
    blk -= f.window_ctas;
    // Everything derived from the plan alone is worked out before the wait
    // for the extract launch (the plan's reads are constant-cache misses on
    // a dependent chain); global data is read after it.
    const long long N = (long long)p.dims[0] * p.dims[1] * p.dims[2];
    int* psh = reinterpret_cast<int*>(fsm);   // the pair's partials
    if (blk < f.cond_ctas) {
        const int j = blk, t = j / a.B, b = j - t * a.B;
        const long long row = (long long)t * a.B + b;   // (t, b) row of the per-tile outputs
        const int T = p.total_tiles;
        pdl_wait();   // the partial extents of the extract launch
        const int pv = tid < 6 * f.K1 ? f.partials[(long long)j * f.K1 * 6 + tid] : 0;
        int2 cv[3];
        if (tid < a.M) {
#pragma unroll
            for (int d = 0; d < 3; ++d) cv[d] = *reinterpret_cast<const int2*>(a.cond + (((long long)b * 3 + d) * a.M + tid) * 2);
        }
        if (tid < 6 * f.K1) psh[tid] = pv;
        pair_extent(psh, f.K1, ext_sh);
        int ext[6];
#pragma unroll
        for (int i = 0; i < 6; ++i) ext[i] = ext_sh[i];
        // keep flags, then the kept tokens compacted in their original
        // order, one block scan per round
        int total = 0;
        for (int m0 = 0; m0 < a.M; m0 += kThreads) {
            const int m = m0 + tid;
            const bool in = m < a.M;
            if (in && m0 > 0) {
#pragma unroll
                for (int d = 0; d < 3; ++d) cv[d] = *reinterpret_cast<const int2*>(a.cond + (((long long)b * 3 + d) * a.M + m) * 2);
            }
            const bool k = in && keep_token(cv, ext);
            if (in) a.keep[row * a.M + m] = k ? 1 : 0;
            if (k) atomicAdd(&f.count[(long long)b * a.M + m], 1);
            int round_total;
            const int at = total + block_excl_scan(k ? 1 : 0, scan_sh, &round_total);
            if (in && a.slot_of) a.slot_of[row * a.M + m] = k ? at : -1;
            if (k && a.kept_idx) a.kept_idx[row * a.M + at] = m;
            if (k && a.tile_cond) {
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    int2 q = cv[d];
                    if (a.normalize) { q.x -= ext[2 * d]; q.y -= ext[2 * d]; }
                    *reinterpret_cast<int2*>(a.tile_cond + ((row * 3 + d) * a.M + at) * 2) = q;
                }
            }
            total += round_total;
        }
        if (a.kept_idx || a.tile_cond || a.slot_of) {
            for (int q = total + tid; q < a.M; q += kThreads) {
                if (a.kept_idx) a.kept_idx[row * a.M + q] = -1;
                if (a.tile_cond) {
#pragma unroll
                    for (int d = 0; d < 3; ++d)
                        *reinterpret_cast<int2*>(a.tile_cond + ((row * 3 + d) * a.M + q) * 2) = make_int2(0, 0);
                }
            }
        }
        if (tid == 0 && a.num_kept) a.num_kept[row] = total;
        // the batch's last pair to get here writes its weights
        __threadfence();   // this CTA's count additions before its arrival
        __syncthreads();
        if (tid == 0) last_sh = atomicAdd(&f.arrivals[b], 1) == T - 1;
        __syncthreads();
        if (last_sh) {
            __threadfence();
            for (int m = tid; m < a.M; m += kThreads) {
                const int c = __ldcg(&f.count[(long long)b * a.M + m]);
                f.weight[(long long)b * a.M + m] = c ? 1.0f / static_cast<float>(c) : 0.0f;
            }
        }
        return;
    }
    blk -= f.cond_ctas;
    const int j = blk / f.K2, c = blk - j * f.K2, t = j / a.B, b = j - t * a.B;
    const long long row = (long long)t * a.B + b;
    const TileTokens tt = tile_tokens(p, t);
    const int* gen_b = a.gen + (long long)b * 3 * N * 2;
    // this part's tokens: at most kJobTokenBatch per thread (K2 sees to it)
    const int csz = (tt.n + f.K2 - 1) / f.K2;
    const int j0 = min(tt.n, c * csz), j1 = min(tt.n, j0 + csz);
    long long n[kJobTokenBatch];
    int2 v[kJobTokenBatch][3];
    if (a.tile_pos) {
        TokenWalk tw;
        tw.init(tt, j0 + tid, kThreads);
#pragma unroll
        for (int u = 0; u < kJobTokenBatch; ++u) {
            n[u] = j0 + tid + u * kThreads < j1 ? tw.token(p, tt) : -1;
            tw.next(tt);
        }
    }
    pdl_wait();   // the partial extents of the extract launch
    // the partial first (the extent waits on it), then the positions
    const int pv = tid < 6 * f.K1 ? f.partials[(long long)j * f.K1 * 6 + tid] : 0;
    if (a.tile_pos) {
#pragma unroll
        for (int u = 0; u < kJobTokenBatch; ++u)
            if (n[u] >= 0) {
#pragma unroll
                for (int d = 0; d < 3; ++d) v[u][d] = *reinterpret_cast<const int2*>(gen_b + ((long long)d * N + n[u]) * 2);
            }
    }
    if (tid < 6 * f.K1) psh[tid] = pv;
    pair_extent(psh, f.K1, ext_sh);
    if (c == 0 && tid < 3 && a.offsets) a.offsets[row * 3 + tid] = ext_sh[2 * tid];
    if (c == 0 && tid < 6 && a.extent) a.extent[row * 6 + tid] = ext_sh[tid];
    if (a.tile_pos) {
        // shifted by TS (by 0 without normalize)
        const int o0 = a.normalize ? ext_sh[0] : 0, o1 = a.normalize ? ext_sh[2] : 0, o2 = a.normalize ? ext_sh[4] : 0;
        int* dst = a.tile_pos + tt.prefix * 6 * a.B + (long long)b * 3 * tt.n * 2;
#pragma unroll
        for (int u = 0; u < kJobTokenBatch; ++u)
            if (n[u] >= 0) {
                const long long k = j0 + tid + u * kThreads;
                *reinterpret_cast<int2*>(dst + (0 * (long long)tt.n + k) * 2) = make_int2(v[u][0].x - o0, v[u][0].y - o0);
                *reinterpret_cast<int2*>(dst + (1 * (long long)tt.n + k) * 2) = make_int2(v[u][1].x - o1, v[u][1].y - o1);
                *reinterpret_cast<int2*>(dst + (2 * (long long)tt.n + k) * 2) = make_int2(v[u][2].x - o2, v[u][2].y - o2);
            }
    }
}

// =================================================================== slab blend
// Output rows [row0, row1) of the blend, one element per thread (grid
// stride), for the sharded blend: per covering (frame tile, row tile) pair,
// in order, inner = sum over the covering column tiles, in order, of
// fmaf(r_w, value, inner), then acc = fmaf(r_f * r_h (rounded), inner,
// acc) -- the grouping and order of every blend kernel, so the slab equals
// those rows of the full blend bit for bit.  Only tiles meeting the slab's
// rows are read.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads) blend_slab_kernel(const __grid_constant__ tdp_plan_t p, const Tin* tiles,
                                                              long long tiles_numel, int BC, int row0, int row1,
                                                              Tout* out) {
    pdl_launch_dependents();
    pdl_wait();   // the tiles may come from the previous kernel
    const int F = p.dims[0], W = p.dims[2], R = row1 - row0;
    const long long n = (long long)BC * F * R * W;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int w = static_cast<int>(e % W);
        long long q = e / W;
        const int h = row0 + static_cast<int>(q % R);
        q /= R;
        const int f = static_cast<int>(q % F);
        const long long bc = q / F;
        int flo, fhi, hlo, hhi, wlo, whi;
        tdp::axis_cover(p, 0, f, flo, fhi);
        tdp::axis_cover(p, 1, h, hlo, hhi);
        tdp::axis_cover(p, 2, w, wlo, whi);
        float acc = 0.0f;
        for (int i_f = flo; i_f <= fhi; ++i_f) {
            const float rf = tdp::axis_weight(p, 0, i_f, f);
            const int sf = tdp::tile_size(p, 0, i_f), zf = f - p.start[0][i_f];
            for (int i_h = hlo; i_h <= hhi; ++i_h) {
                const float wfh = __fmul_rn(rf, tdp::axis_weight(p, 1, i_h, h));
                const int sh = tdp::tile_size(p, 1, i_h), y = h - p.start[1][i_h];
                float inner = 0.0f;
                for (int i_w = wlo; i_w <= whi; ++i_w) {
                    const int sw = tdp::tile_size(p, 2, i_w);
                    const long long off = (long long)BC * tdp::tile_prefix_volume(p, i_f, i_h, i_w) +
                                          ((bc * sf + zf) * sh + y) * sw + (w - p.start[2][i_w]);
                    if (index_bad(off < 0 || off >= tiles_numel)) continue;
                    inner = fmaf(tdp::axis_weight(p, 2, i_w, w), to_f32(tiles[off]), inner);
                }
                acc = fmaf(wfh, inner, acc);
            }
        }
        out[e] = from_f32<Tout>(acc);
    }
}

// =================================================================== K6: conditioning combine
// out[b, m, :] = sum over tiles t keeping token m (slot_of[t, b, m] >= 0),
// in increasing t, of weight[b, m] * tile_out[t, b, slot, :]: the 1/k blend
// of a conditioning token's per-tile outputs, fp32 accumulation, one store.
// One warp per (b, m); its lanes look up the tiles' slots 32 at a time and
// then walk the feature dimension.

// 4 contiguous features as fp32 (a 4-feature row start is 8- or 16-byte aligned).
__device__ __forceinline__ void load_feat4(const __nv_bfloat16* q, float (&v)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(q);
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void load_feat4(const float* q, float (&v)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(q);
    v[0] = u.x;
    v[1] = u.y;
    v[2] = u.z;
    v[3] = u.w;
}
__device__ __forceinline__ void store_feat4(__nv_bfloat16* q, const float (&v)[4]) {
    uint2 u;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(u.x) : "f"(v[1]), "f"(v[0]));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(u.y) : "f"(v[3]), "f"(v[2]));
    *reinterpret_cast<uint2*>(q) = u;
}
__device__ __forceinline__ void store_feat4(float* q, const float (&v)[4]) {
    *reinterpret_cast<float4*>(q) = make_float4(v[0], v[1], v[2], v[3]);
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads) cond_combine_kernel(int T, int BM, int M, int D, const Tin* tile_out,
                                                                const int* slot_of, const float* weight, Tout* out) {
    pdl_launch_dependents();
    pdl_wait();   // slots, weights and tile outputs may come from the previous kernel
    const int lane = threadIdx.x & 31;
    const int bm = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (bm >= BM) return;
    const float w = weight[bm];
    // With D a multiple of 4 a lane takes 4 contiguous features, one load
    // per tile; otherwise features lane, lane + 32, ... one at a time.
    const bool vec = D % kCombineCols == 0;
    for (int d0 = 0; d0 < D; d0 += 32 * kCombineCols) {
        float acc[kCombineCols];
#pragma unroll
        for (int i = 0; i < kCombineCols; ++i) acc[i] = 0.0f;
        const int dv = d0 + lane * kCombineCols;
        for (int t0 = 0; t0 < T; t0 += 32) {
            const int t = t0 + lane;
            const int slot = t < T ? slot_of[(long long)t * BM + bm] : -1;
            unsigned kept = __ballot_sync(0xffffffffu, slot >= 0);
            while (kept) {
                // up to kCombineRound kept tiles per round, lowest first: their
                // loads are issued together, then added in increasing tile order
                float v[kCombineRound][kCombineCols];
                bool has[kCombineRound];   // warp-uniform: `kept` is a ballot
#pragma unroll
                for (int j = 0; j < kCombineRound; ++j) {
                    has[j] = kept != 0;
                    const int src = has[j] ? __ffs(kept) - 1 : 0;
                    kept &= kept - 1;
                    const int st = __shfl_sync(0xffffffffu, slot, src);
                    const long long row = ((long long)(t0 + src) * BM + (bm - bm % M) + st) * D;   // (t, b, st)
                    if (vec) {
                        if (has[j] && dv < D) {
                            load_feat4(tile_out + row + dv, v[j]);
                        } else {
#pragma unroll
                            for (int i = 0; i < kCombineCols; ++i) v[j][i] = 0.0f;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < kCombineCols; ++i) {
                            const int d = d0 + i * 32 + lane;
                            v[j][i] = (has[j] && d < D) ? to_f32(tile_out[row + d]) : 0.0f;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < kCombineRound; ++j)
                    if (has[j]) {
#pragma unroll
                        for (int i = 0; i < kCombineCols; ++i) acc[i] = fmaf(w, v[j][i], acc[i]);
                    }
            }
        }
        if (vec) {
            if (dv < D) store_feat4(out + (long long)bm * D + dv, acc);
        } else {
#pragma unroll
            for (int i = 0; i < kCombineCols; ++i) {
                const int d = d0 + i * 32 + lane;
                if (d < D) out[(long long)bm * D + d] = from_f32<Tout>(acc[i]);
            }
        }
    }
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

// Shared-memory layout of an extract CTA: one barrier per stage, the slot
// table and the staged bands.
struct ExtractLayout {
    int off_slots, off_data, stage_bytes, total;
};

ExtractLayout extract_layout(const tdp_plan_t& p, int band_rows, int esz) {
    const int nbands = (p.dims[1] + band_rows - 1) / band_rows;
    ExtractLayout L;
    L.off_slots = round_up(8 * kExtractStages, 16);
    L.off_data = round_up(L.off_slots + max_slots_for(p, band_rows, nbands) * (int)sizeof(ExtractSlot), 16);
    const long long stage = (long long)round_up(band_rows * p.dims[2] * esz, 16) + 16;
    const long long total = L.off_data + kExtractStages * stage;
    L.stage_bytes = stage > INT_MAX ? INT_MAX : static_cast<int>(stage);
    L.total = total > INT_MAX ? INT_MAX : static_cast<int>(total);
    return L;
}

// Shared-memory layout of a blend CTA: barriers, then the fast kernel's
// per-row (frame tile, row tile) table or the generic kernel's per-axis
// cover tables, then the slot tables and the staged tile rows -- two
// stages for the (persistent) fast kernel, one for the generic kernel.
struct BlendLayout {
    int off_a, off_b, off_c, off_d, off_e, off_slotbase, off_stage, off_data, off_tab;
    int max_slots, data_bytes, total;
    bool fast;
};

// Largest sum of padded staged runs over all (frame, band) boxes.
long long blend_data_bytes(const tdp_plan_t& p, int band_rows, int esz) {
    const int H = p.dims[1], nw = p.num_tiles[2];
    const int nbands = (H + band_rows - 1) / band_rows;
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
                for (int iw = 0; iw < nw; ++iw) sum += round_up(rows * tdp::tile_size(p, 2, iw) * esz, 16) + 16;
            }
            worst = std::max(worst, sum * (fhi - flo + 1));
        }
    }
    return worst;
}

BlendLayout blend_layout(const tdp_plan_t& p, int band_rows, int esz) {
    const int kf = p.max_cover[0], kh = p.max_cover[1], kw = p.max_cover[2], W = p.dims[2];
    const int nbands = (p.dims[1] + band_rows - 1) / band_rows;
    BlendLayout L;
    L.fast = kf <= 2 && kh <= 2 && kw <= 2;
    L.max_slots = max_slots_for(p, band_rows, nbands);
    int o = L.fast ? round_up(16 * kBlendQueue + 8, 16) : 16;  // mbarriers
    if (L.fast) {
        L.off_a = o; o = round_up(o + 64 + band_rows * (int)sizeof(Run), 16);         // header, runs
        L.off_b = o; o = round_up(o + band_rows * kf * kh * 4, 16);                   // w_fh per row and pair
        L.off_c = L.off_d = L.off_e = o;
    } else {
        L.off_a = o; o = round_up(o + kf * (int)sizeof(Cov), 16);                     // fcov
        L.off_b = o; o = round_up(o + band_rows * 4, 16);                             // hcnt
        L.off_c = o; o = round_up(o + band_rows * kh * (int)sizeof(Cov), 16);         // hcov
        L.off_d = o; o = round_up(o + W * 4, 16);                                     // wcnt
        L.off_e = o; o = round_up(o + W * kw * (int)sizeof(Cov), 16);                 // wcov
    }
    L.off_tab = -1;
    const long long tab_bytes = (long long)sizeof(AxisEnt) * ((long long)p.dims[0] + p.dims[1] + W);
    if (L.fast && tab_bytes <= kBlendTabBudget) { L.off_tab = o; o = round_up(o + static_cast<int>(tab_bytes), 16); }
    L.off_stage = o; o = round_up(o + L.max_slots * (int)sizeof(StageSlot), 16);
    L.off_slotbase = o; o = round_up(o + (L.fast ? kBlendQueue : 1) * L.max_slots * 4, 16);
    L.off_data = o;
    // largest item; the fast kernel's ring holds at least two of them and
    // takes the rest of the budget
    const long long item = blend_data_bytes(p, band_rows, esz);
    long long data = item;
    if (L.fast) data = std::max(2 * item, (long long)(kBlendSmemBudget - o) / 16 * 16);
    const long long total = o + data;
    L.data_bytes = data > INT_MAX ? INT_MAX : static_cast<int>(data);
    L.total = total > INT_MAX ? INT_MAX : static_cast<int>(total);
    return L;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

// Grid of a persistent kernel: every resident CTA slot of the GPU, at most
// one CTA per item.
template <typename K>
tdp_status persistent_grid(K kernel, int smem, long long items, unsigned* grid, int threads = kThreads) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (e != cudaSuccess) return cuda_status(e);
    const long long slots = (long long)std::max(1, per_sm) * std::max(1, sm_count());
    *grid = static_cast<unsigned>(std::min(items, slots));
    return TDP_OK;
}

template <typename K>
tdp_status set_smem(K kernel, int bytes) {
    if (bytes <= 48 * 1024) return TDP_OK;
    return cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
}

// Launch with programmatic stream serialization (the kernel may start while
// its predecessor in the stream finishes; see pdl_wait) and, with
// cluster > 1, clusters of that many CTAs.
template <typename K, typename... Args>
tdp_status launch(K kernel, long long blocks, int threads, int smem, cudaStream_t stream, int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    unsigned n = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, args...));
}

template <typename K, typename... Args>
tdp_status launch_cluster(K kernel, long long blocks, cudaStream_t stream, Args... args) {
    return launch(kernel, blocks, kThreads, 0, stream, kCluster, args...);
}

// Most column tiles that cover any of U adjacent output columns (the fast
// blend's term count; at most 3 under the guard for U = 2).
int max_terms(const tdp_plan_t& p, int U) {
    int best = 1;
    for (int c = 0; c < p.dims[2]; c += U) {
        int lo, hi, l2, h2;
        tdp::axis_cover(p, 2, c, lo, hi);
        for (int v = 1; v < U && c + v < p.dims[2]; ++v) {
            tdp::axis_cover(p, 2, c + v, l2, h2);
            lo = std::min(lo, l2);
            hi = std::max(hi, h2);
        }
        best = std::max(best, hi - lo + 1);
    }
    return best;
}

// The per-group item costs of the fast blend's split (see ItemCosts); an
// equal split when there are more groups than the table holds.
ItemCosts item_costs(const tdp_plan_t& p, int band_rows, int nbands, int BC) {
    ItemCosts ic;
    std::memset(&ic, 0, sizeof(ic));
    const int ng = p.dims[0] * nbands;
    if (ng > kCostGroups) return ic;
    const long long SW = p.prefix[2][p.num_tiles[2]], W = p.dims[2];
    for (int g = 0; g < ng; ++g) {
        const int f = g / nbands, hb0 = (g % nbands) * band_rows, hb1 = std::min(p.dims[1], hb0 + band_rows);
        int lo, hi;
        tdp::axis_cover(p, 0, f, lo, hi);
        long long rows = 0;   // band rows times the row tiles covering each
        for (int i = 0; i < p.num_tiles[1]; ++i)
            rows += std::max(0, std::min(hb1, p.end[1][i]) - std::max(hb0, p.start[1][i]));
        ic.cum[g + 1] = ic.cum[g] + ((long long)(hb1 - hb0) * W + (long long)(hi - lo + 1) * rows * SW) * BC;
    }
    if (ic.cum[ng] >= (1LL << 46)) return ItemCosts{};   // keeps (CTA index) * total inside 64 bits
    ic.groups = ng;
    return ic;
}

static_assert(sizeof(tdp_plan_t) + sizeof(BlendArgs) <= 4096, "blend kernel parameters stay within 4 KB");

template <typename Tin, typename Tout>
tdp_status launch_blend_stream(const tdp_plan_t& p, int BC, const void* tiles, long long tiles_numel, void* out,
                               cudaStream_t stream, bool* taken, int row0, int row1);

template <typename Tin, typename Tout>
tdp_status launch_blend(const tdp_plan_t& p, int BC, const void* tiles, long long tiles_numel, void* out,
                        cudaStream_t stream) {
    bool taken = false;
    const tdp_status sst = launch_blend_stream<Tin, Tout>(p, BC, tiles, tiles_numel, out, stream, &taken, 0, p.dims[1]);
    if (sst != TDP_OK || taken) return sst;
    int band_rows = p.dims[1];
    BlendLayout L;
    for (;;) {
        L = blend_layout(p, band_rows, (int)sizeof(Tin));
        if (L.total <= kBlendSmemBudget || band_rows == 1) break;
        band_rows = std::max(1, band_rows / 2);
    }
    if (L.total > 200 * 1024) return TDP_ERR_UNSUPPORTED;
    const int nbands = (p.dims[1] + band_rows - 1) / band_rows;
    const long long items = (long long)BC * p.dims[0] * nbands;
    if (items > INT_MAX) return TDP_ERR_INVALID_ARG;
    BlendArgs a;
    a.tiles = tiles;
    a.out = out;
    a.tiles_numel = tiles_numel;
    a.BC = BC;
    a.band_rows = band_rows;
    a.nbands = nbands;
    a.n_items = static_cast<int>(items);
    a.off_a = L.off_a;
    a.off_b = L.off_b;
    a.off_c = L.off_c;
    a.off_d = L.off_d;
    a.off_e = L.off_e;
    a.off_slotbase = L.off_slotbase;
    a.off_stage = L.off_stage;
    a.off_data = L.off_data;
    a.off_tab = L.off_tab;
    a.max_slots = L.max_slots;
    a.data_bytes = L.data_bytes;
    a.kf = p.max_cover[0];
    a.kh = p.max_cover[1];
    a.kw = p.max_cover[2];
    a.costs = item_costs(p, band_rows, nbands, BC);
    const bool pairs = p.dims[2] % 2 == 0;
    {
        // column units ordered by the number of column tiles they touch
        // (stable), so that the consumer warps share one term count
        const int U = pairs ? 2 : 1, W = p.dims[2], ncu = (W + U - 1) / U;
        a.ordered = ncu <= kMaxOrdered ? 1 : 0;
        if (a.ordered) {
            uint8_t cls[kMaxOrdered];
            int count[kMaxOrdered + 2] = {0};
            for (int u = 0; u < ncu; ++u) {
                int lo, hi, l2, h2;
                tdp::axis_cover(p, 2, u * U, lo, hi);
                for (int v = 1; v < U && u * U + v < W; ++v) {
                    tdp::axis_cover(p, 2, u * U + v, l2, h2);
                    lo = std::min(lo, l2);
                    hi = std::max(hi, h2);
                }
                cls[u] = static_cast<uint8_t>(hi - lo + 1);
                ++count[cls[u] + 1];
            }
            for (int k = 1; k <= kMaxOrdered + 1; ++k) count[k] += count[k - 1];   // first slot per class
            for (int u = 0; u < ncu; ++u) a.order[count[cls[u]]++] = static_cast<uint16_t>(u);
        }
    }
    auto go = [&](auto kernel, bool persistent) -> tdp_status {
        tdp_status st = set_smem(kernel, L.total);
        if (st != TDP_OK) return st;
        unsigned grid = static_cast<unsigned>(items);
        const int threads = persistent ? kBlendThreads : kThreads;
        if (persistent && (st = persistent_grid(kernel, L.total, items, &grid, threads)) != TDP_OK) return st;
        return launch(kernel, grid, threads, L.total, stream, 1, p, a);
    };
    // Pair stores need every output row to start on a 4-byte (bf16) or
    // 8-byte (fp32) boundary: W even.
    if (!L.fast) return go(blend_generic_kernel<Tin, Tout>, false);
    const int kt = max_terms(p, pairs ? 2 : 1);
    if (pairs) {
        if (kt == 1) return go(blend_fast_kernel<Tin, Tout, 2, 1>, true);
        if (kt == 2) return go(blend_fast_kernel<Tin, Tout, 2, 2>, true);
        return go(blend_fast_kernel<Tin, Tout, 2, 3>, true);
    }
    if (kt == 1) return go(blend_fast_kernel<Tin, Tout, 1, 1>, true);
    return go(blend_fast_kernel<Tin, Tout, 1, 2>, true);
}

#include "tdp_stream.cuh"

}  // namespace

namespace tdp {
// Shared with the token-major translation unit.
tdp_status record_cuda(cudaError_t e) { return cuda_status(e); }
int device_sm_count() { return sm_count(); }
}  // namespace tdp

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
    if ((long long)B * C > INT_MAX) return TDP_ERR_INVALID_ARG;
    bool taken = false;
    const tdp_status sst = esz == 2 ? launch_extract_stream<uint16_t>(p, B * C, latent, tiles, stream, &taken)
                                    : launch_extract_stream<uint32_t>(p, B * C, latent, tiles, stream, &taken);
    if (sst != TDP_OK || taken) return sst;
    int band_rows = p.dims[1];
    ExtractLayout L;
    for (;;) {
        L = extract_layout(p, band_rows, esz);
        if (L.total <= kExtractSmemBudget || band_rows == 1) break;
        band_rows = std::max(1, band_rows / 2);
    }
    if (L.total > 200 * 1024) return TDP_ERR_UNSUPPORTED;
    const int nbands = (p.dims[1] + band_rows - 1) / band_rows;
    const long long items = (long long)B * C * p.dims[0] * nbands;
    if (items > INT_MAX || (long long)B * C > INT_MAX) return TDP_ERR_INVALID_ARG;
    ExtractArgs a{latent, tiles, (long long)B * C * p.dims[0] * p.dims[1] * p.dims[2],
                  (long long)B * C * tdp::total_volume(p), B * C, band_rows, nbands,
                  static_cast<int>(items), L.off_slots, L.off_data, L.stage_bytes};
    auto go = [&](auto kernel) -> tdp_status {
        tdp_status st = set_smem(kernel, L.total);
        if (st != TDP_OK) return st;
        unsigned grid = 0;
        if ((st = persistent_grid(kernel, L.total, items, &grid)) != TDP_OK) return st;
        return launch(kernel, grid, kThreads, L.total, stream, 1, p, a);
    };
    return esz == 2 ? go(extract_kernel<uint16_t>) : go(extract_kernel<uint32_t>);
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
    const long long n = (long long)BC * tdp::total_volume(*plan);
    if (in_dtype == TDP_BF16 && out_dtype == TDP_BF16)
        return launch_blend<__nv_bfloat16, __nv_bfloat16>(*plan, BC, tiles, n, out, stream);
    if (in_dtype == TDP_BF16 && out_dtype == TDP_F32)
        return launch_blend<__nv_bfloat16, float>(*plan, BC, tiles, n, out, stream);
    if (in_dtype == TDP_F32 && out_dtype == TDP_BF16)
        return launch_blend<float, __nv_bfloat16>(*plan, BC, tiles, n, out, stream);
    return launch_blend<float, float>(*plan, BC, tiles, n, out, stream);
}

// Workspace of tdp_extract_and_tokens: the partial extents, then one
// arrival counter per batch.
inline long long token_workspace_ints(long long J, int K1, int B) { return J * K1 * 6 + B; }

int64_t tdp_extract_and_tokens_workspace(const tdp_plan_t* plan, int32_t B) {
    if (!tdp::plan_is_valid(plan) || B < 0) return -1;
    const long long J = (long long)plan->total_tiles * B;
    return round_up(token_workspace_ints(J, extent_chunks_k1(*plan, J, kStreamMaxGrid), B) * 4, 16LL);
}

tdp_status tdp_extract_and_tokens(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype, const void* latent,
                                  void* tiles, const int32_t* gen_pos, int32_t normalize, int32_t* tile_pos,
                                  int32_t* offsets, int32_t M, const int32_t* cond_pos, int32_t* tile_extent,
                                  uint8_t* keep, int32_t* count, float* weight, int32_t* kept_idx,
                                  int32_t* num_kept, int32_t* tile_cond_pos, int32_t* slot_of, float* max_abs_dev,
                                  void* workspace, int64_t workspace_bytes, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || C < 0 || M < 0 || workspace_bytes < 0) return TDP_ERR_INVALID_ARG;
    const int esz = dtype_size(dtype);
    if (!esz) return TDP_ERR_INVALID_ARG;
    if (B == 0) return max_abs_dev ? tdp_window_sum(plan, max_abs_dev, nullptr, stream) : TDP_OK;
    if (C > 0 && (!latent || !tiles)) return TDP_ERR_INVALID_ARG;
    if (!gen_pos || (tile_pos && !offsets)) return TDP_ERR_INVALID_ARG;
    if (M > 0 && (!cond_pos || !tile_extent || !keep || !count || !weight)) return TDP_ERR_INVALID_ARG;
    const void* ptrs[] = {latent, tiles, gen_pos, tile_pos, offsets, cond_pos, tile_extent, keep, count,
                          weight, kept_idx, num_kept, tile_cond_pos, slot_of, max_abs_dev, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return TDP_ERR_ALIGNMENT;
    const tdp_plan_t& p = *plan;
    const long long J = (long long)p.total_tiles * B;
    if ((long long)B * C > INT_MAX || (long long)kCluster * J > INT_MAX || (long long)B * M > INT_MAX)
        return TDP_ERR_INVALID_ARG;
    const TokensArgs a{gen_pos, B, normalize ? 1 : 0, tile_pos, offsets, M, cond_pos, tile_extent, keep, kept_idx,
                       num_kept, tile_cond_pos, slot_of};
    // the two-launch form: the streaming extract reduces the partial extents
    const int K1 = extent_chunks_k1(p, J, std::min(sm_count(), kStreamMaxGrid)), K2 = extent_chunks(p, kFinishTokens);
    const long long need = token_workspace_ints(J, K1, B) * 4;
    const long long cond_ctas = M > 0 ? J : 0;
    const long long fsmem = finish_smem(p, K1, max_abs_dev != nullptr);
    const long long fgrid = J * K2 + cond_ctas + (max_abs_dev ? 1 : 0);
    if (C > 0 && workspace && workspace_bytes >= need && fsmem <= 40 * 1024 && 6LL * K1 <= kThreads &&
        fgrid <= INT_MAX) {
        bool taken = false;
        int* partials = static_cast<int*>(workspace);
        int* arrivals = partials + J * K1 * 6;
        const StreamZero zero{M > 0 ? count : nullptr, B * M, arrivals, B};
        const tdp_status sst =
            esz == 2 ? launch_extract_stream<uint16_t>(p, B * C, latent, tiles, stream, &taken, gen_pos, B, K1, partials, zero)
                     : launch_extract_stream<uint32_t>(p, B * C, latent, tiles, stream, &taken, gen_pos, B, K1, partials, zero);
        if (sst != TDP_OK) return sst;
        if (taken) {
            const TokenFinishArgs fa{a, count, weight, max_abs_dev, partials, arrivals, K1, K2, max_abs_dev ? 1 : 0,
                                     static_cast<int>(cond_ctas)};
            tdp_status st = set_smem(tokens_finish_kernel, static_cast<int>(fsmem));
            if (st != TDP_OK) return st;
            return launch(tokens_finish_kernel, fgrid, kThreads, static_cast<int>(fsmem), stream, 1, p, fa);
        }
    }
    // otherwise the separate kernels in turn
    if (C > 0) {
        const tdp_status st = tdp_extract(plan, B, C, dtype, latent, tiles, stream);
        if (st != TDP_OK) return st;
    }
    tdp_status st = tdp_tokens(plan, B, gen_pos, normalize, tile_pos, offsets, M, cond_pos, tile_extent, keep, count,
                               weight, kept_idx, num_kept, tile_cond_pos, slot_of, stream);
    if (st != TDP_OK) return st;
    return max_abs_dev ? tdp_window_sum(plan, max_abs_dev, nullptr, stream) : TDP_OK;
}

tdp_status tdp_extract_and_tokens_no_alloc(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype,
                                           const void* latent, void* tiles, const int32_t* gen_pos,
                                           int32_t normalize, int32_t* tile_pos, int32_t* offsets, int32_t M,
                                           const int32_t* cond_pos, int32_t* tile_extent, uint8_t* keep,
                                           int32_t* count, float* weight, int32_t* kept_idx, int32_t* num_kept,
                                           int32_t* tile_cond_pos, int32_t* slot_of, float* max_abs_dev,
                                           cudaStream_t stream) {
    const int64_t need = tdp_extract_and_tokens_workspace(plan, B);
    if (need < 0) return TDP_ERR_INVALID_ARG;
    if (need > (int64_t)sizeof(g_token_scratch)) return TDP_ERR_UNSUPPORTED;
    void* scratch = nullptr;   // this device's instance of the library's scratch array
    const tdp_status st = cuda_status(cudaGetSymbolAddress(&scratch, g_token_scratch));
    if (st != TDP_OK) return st;
    return tdp_extract_and_tokens(plan, B, C, dtype, latent, tiles, gen_pos, normalize, tile_pos, offsets, M,
                                  cond_pos, tile_extent, keep, count, weight, kept_idx, num_kept, tile_cond_pos,
                                  slot_of, max_abs_dev, scratch, (int64_t)sizeof(g_token_scratch), stream);
}

tdp_status tdp_blend_slab(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype in_dtype, const void* tiles,
                          int32_t row0, int32_t row1, tdp_dtype out_dtype, void* out, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || C < 0) return TDP_ERR_INVALID_ARG;
    if (!dtype_size(in_dtype) || !dtype_size(out_dtype)) return TDP_ERR_INVALID_ARG;
    if (row0 < 0 || row1 < row0 || row1 > plan->dims[1]) return TDP_ERR_INVALID_ARG;
    if (B == 0 || C == 0 || row0 == row1) return TDP_OK;
    if (!tiles || !out) return TDP_ERR_INVALID_ARG;
    if (!aligned16(tiles) || !aligned16(out)) return TDP_ERR_ALIGNMENT;
    if ((long long)B * C > INT_MAX) return TDP_ERR_INVALID_ARG;
    const int BC = B * C;
    const long long n = (long long)BC * plan->dims[0] * (row1 - row0) * plan->dims[2];
    const long long blocks = std::min<long long>((n + kThreads - 1) / kThreads, 8LL * std::max(1, sm_count()));
    auto go = [&](auto tin, auto tout) {
        using Ti = decltype(tin);
        using To = decltype(tout);
        // the streaming blend restricted to the slab's rows where it takes the plan
        bool taken = false;
        const tdp_status sst = launch_blend_stream<Ti, To>(*plan, BC, tiles, (long long)BC * tdp::total_volume(*plan),
                                                           out, stream, &taken, row0, row1);
        if (sst != TDP_OK || taken) return sst;
        return launch(blend_slab_kernel<Ti, To>, blocks, kThreads, 0, stream, 1, *plan, static_cast<const Ti*>(tiles),
                      (long long)BC * tdp::total_volume(*plan), BC, row0, row1, static_cast<To*>(out));
    };
    if (in_dtype == TDP_BF16 && out_dtype == TDP_BF16) return go(__nv_bfloat16(), __nv_bfloat16());
    if (in_dtype == TDP_BF16 && out_dtype == TDP_F32) return go(__nv_bfloat16(), 0.0f);
    if (in_dtype == TDP_F32 && out_dtype == TDP_BF16) return go(0.0f, __nv_bfloat16());
    return go(0.0f, 0.0f);
}

tdp_status tdp_window_sum(const tdp_plan_t* plan, float* max_abs_dev, float* sum_out, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || !max_abs_dev) return TDP_ERR_INVALID_ARG;
    if (!aligned16(max_abs_dev) || (sum_out && !aligned16(sum_out))) return TDP_ERR_ALIGNMENT;
    const tdp_plan_t& p = *plan;
    const long long N = (long long)p.dims[0] * p.dims[1] * p.dims[2];
    const long long tab = 4LL * ((long long)p.dims[0] * p.max_cover[0] + (long long)p.dims[1] * p.max_cover[1] +
                                 p.dims[2] + p.dims[0] + p.dims[1]);
    const int tables = tab <= 32 * 1024 ? 1 : 0;
    const int smem = tables ? static_cast<int>(tab) : 0;
    if (!sum_out && tables) {
        // the maximum alone: one CTA over the runs of equal weight tuples
        const long long reps = window_max_bytes(p);
        if (reps <= 40 * 1024) {
            tdp_status st = set_smem(window_max_kernel, static_cast<int>(reps));
            if (st != TDP_OK) return st;
            return launch(window_max_kernel, 1, kThreads, static_cast<int>(reps), stream, 1, p, max_abs_dev);
        }
    }
    tdp_status st = cuda_status(cudaMemsetAsync(max_abs_dev, 0, sizeof(float), stream));
    if (st != TDP_OK) return st;
    const long long blocks = std::min<long long>((N + 4LL * kThreads - 1) / (4LL * kThreads), 2LL * std::max(1, sm_count()));
    return launch(window_sum_kernel, blocks, kThreads, smem, stream, 1, p, max_abs_dev, sum_out, tables);
}

tdp_status tdp_tokens(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos, int32_t normalize,
                      int32_t* tile_pos, int32_t* offsets, int32_t M, const int32_t* cond_pos,
                      int32_t* tile_extent, uint8_t* keep, int32_t* count, float* weight, int32_t* kept_idx,
                      int32_t* num_kept, int32_t* tile_cond_pos, int32_t* slot_of, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || M < 0) return TDP_ERR_INVALID_ARG;
    if (B == 0) return TDP_OK;
    if (!gen_pos || (tile_pos && !offsets)) return TDP_ERR_INVALID_ARG;
    if (M > 0 && (!cond_pos || !tile_extent || !keep || !count || !weight)) return TDP_ERR_INVALID_ARG;
    const void* ptrs[] = {gen_pos, tile_pos, offsets, cond_pos, tile_extent, keep,
                          count, weight, kept_idx, num_kept, tile_cond_pos, slot_of};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return TDP_ERR_ALIGNMENT;
    const long long blocks = (long long)kCluster * plan->total_tiles * B;
    if (blocks > INT_MAX || (long long)B * M > INT_MAX) return TDP_ERR_INVALID_ARG;
    TokensArgs a{gen_pos, B, normalize ? 1 : 0, tile_pos, offsets, M, cond_pos, tile_extent, keep, kept_idx,
                 num_kept, tile_cond_pos, slot_of};
    tdp_status st = launch_cluster(tokens_kernel, blocks, stream, *plan, a);
    if (st != TDP_OK || M == 0) return st;
    const int BM = B * M;
    return launch(cond_count_kernel, (BM + kThreads - 1) / kThreads, kThreads, 0, stream, 1,
                  static_cast<const unsigned char*>(keep), plan->total_tiles, BM, count, weight);
}

tdp_status tdp_positions(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos, int32_t normalize,
                         int32_t* tile_pos, int32_t* offsets, cudaStream_t stream) {
    if (!tile_pos || !offsets) return TDP_ERR_INVALID_ARG;
    return tdp_tokens(plan, B, gen_pos, normalize, tile_pos, offsets, 0, nullptr, nullptr, nullptr, nullptr,
                      nullptr, nullptr, nullptr, nullptr, nullptr, stream);
}

tdp_status tdp_cond_select(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos, int32_t M,
                           const int32_t* cond_pos, int32_t normalize, int32_t* tile_extent, uint8_t* keep,
                           int32_t* count, float* weight, int32_t* kept_idx, int32_t* num_kept,
                           int32_t* tile_cond_pos, cudaStream_t stream) {
    if (!tile_extent) return TDP_ERR_INVALID_ARG;
    return tdp_tokens(plan, B, gen_pos, normalize, nullptr, nullptr, M, cond_pos, tile_extent, keep, count, weight,
                      kept_idx, num_kept, tile_cond_pos, nullptr, stream);
}

tdp_status tdp_cond_combine(const tdp_plan_t* plan, int32_t B, int32_t M, int32_t D, tdp_dtype in_dtype,
                            const void* tile_cond_out, const int32_t* slot_of, const float* weight,
                            tdp_dtype out_dtype, void* out, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || M < 0 || D < 0) return TDP_ERR_INVALID_ARG;
    if (!dtype_size(in_dtype) || !dtype_size(out_dtype)) return TDP_ERR_INVALID_ARG;
    if (B == 0 || M == 0 || D == 0) return TDP_OK;
    if (!tile_cond_out || !slot_of || !weight || !out) return TDP_ERR_INVALID_ARG;
    const void* ptrs[] = {tile_cond_out, slot_of, weight, out};
    for (const void* q : ptrs)
        if (!aligned16(q)) return TDP_ERR_ALIGNMENT;
    const long long BM = (long long)B * M;
    if (BM > INT_MAX || (long long)plan->total_tiles * BM * D > (1LL << 62)) return TDP_ERR_INVALID_ARG;
    const int warps = kThreads / 32;
    const long long blocks = (BM + warps - 1) / warps;
    const int T = plan->total_tiles;
    auto go = [&](auto kernel, const auto* in, auto* o) {
        return launch(kernel, blocks, kThreads, 0, stream, 1, T, static_cast<int>(BM), M, D, in, slot_of, weight, o);
    };
    const bool ib = in_dtype == TDP_BF16, ob = out_dtype == TDP_BF16;
    if (ib && ob) return go(cond_combine_kernel<__nv_bfloat16, __nv_bfloat16>,
                            static_cast<const __nv_bfloat16*>(tile_cond_out), static_cast<__nv_bfloat16*>(out));
    if (ib) return go(cond_combine_kernel<__nv_bfloat16, float>, static_cast<const __nv_bfloat16*>(tile_cond_out),
                      static_cast<float*>(out));
    if (ob) return go(cond_combine_kernel<float, __nv_bfloat16>, static_cast<const float*>(tile_cond_out),
                      static_cast<__nv_bfloat16*>(out));
    return go(cond_combine_kernel<float, float>, static_cast<const float*>(tile_cond_out), static_cast<float*>(out));
}

tdp_status tdp_launch_geometry(const tdp_plan_t* plan, int32_t B, int32_t C, int32_t blend, tdp_dtype in_dtype,
                               tdp_dtype out_dtype, int32_t sm_count, tdp_launch_geometry_t* geometry,
                               int32_t* cta_start, int32_t cta_start_len, void* tables, int32_t tables_bytes,
                               int32_t* table_offsets, int32_t row0, int32_t row1) {
    if (!tdp::plan_is_valid(plan) || !geometry || B < 1 || C < 1 || sm_count < 1 || cta_start_len < 0 ||
        tables_bytes < 0)
        return TDP_ERR_INVALID_ARG;
    if (row0 < 0 || row1 <= row0 || row1 > plan->dims[1] || (!blend && (row0 != 0 || row1 != plan->dims[1])))
        return TDP_ERR_INVALID_ARG;
    const int isz = dtype_size(in_dtype), osz = dtype_size(out_dtype);
    if (!isz || !osz || (!blend && isz != osz)) return TDP_ERR_INVALID_ARG;
    if ((long long)B * C > INT_MAX) return TDP_ERR_INVALID_ARG;
    std::memset(geometry, 0, sizeof(*geometry));
    int kt = 0;
    if (!stream_eligible(*plan, blend != 0, isz, osz, &kt)) return TDP_OK;
    static thread_local StreamLaunch L;   // 9 KB: kept off the caller's stack
    const tdp_status st = stream_geometry(*plan, blend != 0, B * C, isz, osz, sm_count, L, StreamJobPlan{}, row0, row1);
    if (st == TDP_ERR_UNSUPPORTED) return TDP_OK;
    if (st != TDP_OK) return st;
    geometry->streaming = 1;
    geometry->band_rows = L.a.band_rows;
    geometry->nbands = L.a.nbands;
    geometry->units = L.a.n_units;
    geometry->grid = L.grid;
    geometry->stages = L.a.nstages;
    geometry->stage_bytes = L.a.stage_bytes;
    geometry->max_runs = L.a.max_runs;
    geometry->shared_bytes = L.smem;
    geometry->off_hdr = L.a.off_hdr;
    geometry->off_data = L.a.off_data;
    geometry->chunks_per_row = blend ? L.a.cpr : 0;
    geometry->column_terms = blend ? kt : 0;
    if (blend) {
        for (int c = 0; c < kChunkClasses; ++c) {
            geometry->class_first[c] = L.a.tfirst[c];
            geometry->row_groups[c] = L.a.grp[c];
            geometry->row_step[c] = L.a.gstep[c];
            if (L.a.grp[c] > 0)
                geometry->rows_per_thread =
                    std::max(geometry->rows_per_thread, (L.a.band_rows + L.a.grp[c] - 1) / L.a.grp[c]);
        }
    }
    geometry->threads = 32 * (blend ? kStreamBlendWarps : kStreamExtractWarps);
    geometry->run_slot = blend ? L.a.run_slot : 0;
    geometry->table_bytes = 16 * L.a.t_words;
    if (tables) std::memcpy(tables, L.tb.w, static_cast<size_t>(std::min(tables_bytes, 16 * L.a.t_words)));
    if (table_offsets) {
        const int32_t offs[7] = {L.a.t_band, L.a.t_frame, L.a.t_row, L.a.t_fcon, L.a.t_wcon, L.a.t_runs, L.a.t_chunk};
        std::memcpy(table_offsets, offs, sizeof(offs));
    }
    if (cta_start && cta_start_len > L.grid)
        for (int i = 0; i <= L.grid; ++i) cta_start[i] = L.sp.start[i];
    return TDP_OK;
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
