// Token-major tile extract and blend of libtdp (sm_103a).
//
// The per-tile transformer consumes a tile as a sequence of its N_t tokens,
// each carrying all C channels ("Tiled Data Parallelism (TDP)", What it is
// and When to use it; the tile's tokens are its sub-grid of the generated
// token grid, in row-major (f, h, w) order, Position normalization).  These
// kernels move tiles between the channel-first latent [B, C, F, H, W] and
// packed token-major tiles [T][B, N_t, C] without a separate transpose pass:
//
//   tokens[t][b, n, c] = latent[b, c, f0+k, h0+y, w0+x],  n = (k*h_t + y)*w_t + x
//   out[b, c, f, h, w] = sum_t r_f r_h r_w * tokens[t][b, n_t(f, h, w), c]
//
// Work unit: one latent row (b, f, h) over a block of columns and all C
// channels.  Its channel-first side is C row segments of the latent; its
// token-major side is, for every tile row crossing it, one contiguous run
// of tokens (C channels each).  A unit is transposed through shared memory
// held as [column][16-byte channel chunk], the chunk index XOR-swizzled by
// the column so that both the column-wise and the chunk-wise passes are
// free of bank conflicts.  Global traffic is one read and one write per
// element: the latent side is read (extract) or written (blend) once, each
// tile's tokens are written (extract) or read (blend) once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "tdp.h"
#include "tdp_geometry.h"

namespace tdp {
bool plan_is_valid(const tdp_plan_t* p);
tdp_status record_cuda(cudaError_t e);   // also remembered for tdp_last_cuda_error
int device_sm_count();
}  // namespace tdp

namespace {

constexpr int kTmThreads = 256;
constexpr int kTmItems = 4;                            // 16-byte chunks per thread per unit (at most, in the blend)
constexpr int kTmChunks = kTmThreads * kTmItems;       // chunks of one unit's token side
constexpr int kTmKw = 2;                               // column tiles per column kept in registers

using tdp::axis_weight;

struct TmArgs {
    const void* src;
    void* dst;
    long long fhw;        // F * H * W
    int B, C;
    int J;                // 16-byte chunks per token in the token-major buffer
    int jf;               // blend: fp32 chunks (4 channels) per column in shared memory
    int pmask, pfmask;    // swizzle masks: min(largest power of two <= chunks, 8) - 1
    int ipt, lpt;         // blend: chunks of one token per thread (4, 2 or 1) and threads per token
    int xb, nxb;          // columns per unit, column blocks per latent row
    int units;            // B * F * H * nxb
};

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Physical chunk of logical chunk j of a shared row of n chunks, for column
// x: inside every aligned group of mask+1 chunks that lies wholly in the row
// the low bits are XOR-ed with the column's, so that 8 neighbouring columns
// hit 8 different bank groups; a trailing partial group keeps its order.
__device__ __forceinline__ int swz(int j, int x, int mask, int n) { return (j | mask) < n ? (j ^ (x & mask)) : j; }

// The blend's fp32 rows: the same, with the column's low three bits
// permuted (bit 0 to the top) when 8 chunks are swizzled, so that two
// neighbouring columns also fall in opposite halves of the 8 groups.
__device__ __forceinline__ int swzf(int j, int x, int mask, int n) {
    const int f = mask == 7 ? (((x & 1) << 2) | ((x >> 1) & 3)) : (x & mask);
    return (j | mask) < n ? (j ^ f) : j;
}

// Units are numbered in mixed radix (batch, frame, row, column block); a CTA
// walks its units with a constant stride, digit by digit.
struct UnitWalk {
    int xb, h, f, b;        // current unit
    int sxb, sh, sf, sb;    // stride
};

__device__ __forceinline__ void unit_digits(const tdp_plan_t& p, const TmArgs& a, int u, int& xb, int& h, int& f,
                                            int& b) {
    xb = u % a.nxb;
    u /= a.nxb;
    h = u % p.dims[1];
    u /= p.dims[1];
    f = u % p.dims[0];
    b = u / p.dims[0];
}

__device__ __forceinline__ UnitWalk unit_walk(const tdp_plan_t& p, const TmArgs& a, int u0, int stride) {
    UnitWalk w;
    unit_digits(p, a, u0, w.xb, w.h, w.f, w.b);
    unit_digits(p, a, stride, w.sxb, w.sh, w.sf, w.sb);
    return w;
}

// Each digit plus the stride's digit plus a carry stays below twice the radix.
__device__ __forceinline__ void unit_next(const tdp_plan_t& p, const TmArgs& a, UnitWalk& w) {
    w.xb += w.sxb;
    int c = w.xb >= a.nxb;
    if (c) w.xb -= a.nxb;
    w.h += w.sh + c;
    c = w.h >= p.dims[1];
    if (c) w.h -= p.dims[1];
    w.f += w.sf + c;
    c = w.f >= p.dims[0];
    if (c) w.f -= p.dims[0];
    w.b += w.sb + c;
}

struct Unit {
    int b, f, h, x0, xbu;     // latent row, first column and columns of the block
};

__device__ __forceinline__ Unit unit_of(const tdp_plan_t& p, const TmArgs& a, const UnitWalk& w) {
    const int x0 = w.xb * a.xb;
    return Unit{w.b, w.f, w.h, x0, min(a.xb, p.dims[2] - x0)};
}

// Element offset of channel 0 of the unit's first column in the latent.
__device__ __forceinline__ long long latent_row(const tdp_plan_t& p, const TmArgs& a, const Unit& U) {
    return ((long long)U.b * a.C * p.dims[0] + U.f) * p.dims[1] * (long long)p.dims[2] +
           (long long)U.h * p.dims[2] + U.x0;
}

// Token index, in the packed buffer, of row (k, y) of the tiles of frame
// tile i_f and row tile i_h for batch b, as A + Bm * P_w + Cm * w_t with P_w
// and w_t the column tile's width prefix and width:
//   B * (volume of the tiles before it) + ((b * f_t + k) * h_t + y) * w_t.
struct TileRow {
    long long A, Bm, Cm;
};

__device__ __forceinline__ TileRow tile_row(const tdp_plan_t& p, int B, int b, int i_f, int i_h, int k, int y) {
    const long long sf = tdp::tile_size(p, 0, i_f), sh = tdp::tile_size(p, 1, i_h);
    const long long SW = p.prefix[2][p.num_tiles[2]];
    TileRow r;
    r.A = (long long)B * ((long long)p.prefix[0][i_f] * p.prefix[1][p.num_tiles[1]] * SW + sf * p.prefix[1][i_h] * SW);
    r.Bm = (long long)B * sf * sh;
    r.Cm = ((long long)b * sf + k) * sh + y;
    return r;
}

__device__ __forceinline__ long long row_token(const tdp_plan_t& p, const TileRow& r, int i_w) {
    return r.A + r.Bm * p.prefix[2][i_w] + r.Cm * tdp::tile_size(p, 2, i_w);
}

// ------------------------------------------------------------------ extract
// Pass 1 reads the unit's C x xbu latent block column-wise (a warp reads 32
// neighbouring columns, or column pairs, of one channel row) and stores
// 16-byte channel chunks per column; pass 2 writes each column's chunks to
// every tile token that holds it (a warp writes whole tokens).  The next
// unit's latent block is loaded into registers while the current one is
// written out.
//
// PAIR (even W and column blocks): an item is two neighbouring columns,
// loaded 4 bytes (bf16) or 8 bytes (fp32) at a time, and the shared rows
// swizzle by the column pair, so that the 8 even (or odd) columns a
// quarter-warp stores still fall in 8 bank groups.
template <typename E> struct PairOf;
template <> struct PairOf<uint16_t> { using type = uint32_t; };
template <> struct PairOf<uint32_t> { using type = uint2; };

__device__ __forceinline__ void split_pair(const uint32_t (&v)[8], uint4& c0, uint4& c1) {
    c0 = make_uint4(__byte_perm(v[0], v[1], 0x5410), __byte_perm(v[2], v[3], 0x5410), __byte_perm(v[4], v[5], 0x5410),
                    __byte_perm(v[6], v[7], 0x5410));
    c1 = make_uint4(__byte_perm(v[0], v[1], 0x7632), __byte_perm(v[2], v[3], 0x7632), __byte_perm(v[4], v[5], 0x7632),
                    __byte_perm(v[6], v[7], 0x7632));
}
__device__ __forceinline__ void split_pair(const uint2 (&v)[4], uint4& c0, uint4& c1) {
    c0 = make_uint4(v[0].x, v[1].x, v[2].x, v[3].x);
    c1 = make_uint4(v[0].y, v[1].y, v[2].y, v[3].y);
}

template <bool PAIR>
__device__ __forceinline__ int swz_extract(int j, int x, int mask, int n) {
    return swz(j, PAIR ? (x >> 1) : x, mask, n);
}

template <typename E, bool PAIR>   // raw element: uint16_t (bf16) or uint32_t (fp32); a bit copy
__global__ void __launch_bounds__(kTmThreads, 4) extract_tokens_kernel(const __grid_constant__ tdp_plan_t p,
                                                                       const TmArgs a) {
    constexpr int VEC = 16 / sizeof(E);
    constexpr int NI = PAIR ? kTmItems / 2 : kTmItems;   // items per thread
    using L = typename std::conditional<PAIR, typename PairOf<E>::type, E>::type;
    __shared__ uint4 sbuf[kTmChunks];
    const E* __restrict__ src = static_cast<const E*>(a.src);
    uint4* __restrict__ dst = static_cast<uint4*>(a.dst);
    const int tid = threadIdx.x;
    const int J = a.J;
    // pass 2: a thread's first (column, chunk) of a run and its step
    const int tq = tid / J, tr = tid % J;
    const int sx2 = kTmThreads / J, sj2 = kTmThreads % J;

    L v[NI][VEC];
    int ix[NI], ij[NI];   // item: column (or column pair) and chunk
    // pass 1: a thread's first (column, chunk) of a block of xbu columns and its step
    int c_xbu = -1, x1 = 0, j1 = 0, sx1 = 0, sj1 = 0;

    auto load = [&](const Unit& U) {
        const int ncol = PAIR ? U.xbu / 2 : U.xbu;   // items per chunk index
        if (U.xbu != c_xbu) {
            c_xbu = U.xbu;
            x1 = tid % ncol;
            j1 = tid / ncol;
            sx1 = kTmThreads % ncol;
            sj1 = kTmThreads / ncol;
        }
        const E* base = src + latent_row(p, a, U);
        int x = x1, j = j1;
#pragma unroll
        for (int r = 0; r < NI; ++r) {
            ix[r] = x;
            ij[r] = j < J ? j : -1;
            if (ij[r] >= 0) {
                const L* s = reinterpret_cast<const L*>(base + (long long)j * VEC * a.fhw + (PAIR ? 2 * x : x));
                const long long step = a.fhw / (PAIR ? 2 : 1);   // one channel row, in loads
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[r][e] = __ldg(s + e * step);
            }
            x += sx1;
            j += sj1;
            if (x >= ncol) {
                x -= ncol;
                ++j;
            }
        }
    };

    pdl_wait();
    int u = blockIdx.x;
    if (u >= a.units) return;
    UnitWalk walk = unit_walk(p, a, u, gridDim.x);
    Unit U = unit_of(p, a, walk);
    load(U);
    while (true) {
#pragma unroll
        for (int r = 0; r < NI; ++r) {
            if (ij[r] < 0) continue;
            if constexpr (PAIR) {
                uint4 c0, c1;
                split_pair(v[r], c0, c1);
                const int x0c = 2 * ix[r];
                sbuf[x0c * J + swz_extract<PAIR>(ij[r], x0c, a.pmask, J)] = c0;
                sbuf[(x0c + 1) * J + swz_extract<PAIR>(ij[r], x0c + 1, a.pmask, J)] = c1;
            } else {
                uint4 w;
                if constexpr (VEC == 8) {
                    w.x = (uint32_t)v[r][0] | ((uint32_t)v[r][1] << 16);
                    w.y = (uint32_t)v[r][2] | ((uint32_t)v[r][3] << 16);
                    w.z = (uint32_t)v[r][4] | ((uint32_t)v[r][5] << 16);
                    w.w = (uint32_t)v[r][6] | ((uint32_t)v[r][7] << 16);
                } else {
                    w = make_uint4(v[r][0], v[r][1], v[r][2], v[r][3]);
                }
                sbuf[ix[r] * J + swz_extract<PAIR>(ij[r], ix[r], a.pmask, J)] = w;
            }
        }
        __syncthreads();
        const Unit cur = U;
        const int un = u + gridDim.x;
        if (un < a.units) {
            unit_next(p, a, walk);
            U = unit_of(p, a, walk);
            load(U);
        }

        int flo, fhi, hlo, hhi, wlo, whi;
        tdp::axis_cover(p, 0, cur.f, flo, fhi);
        tdp::axis_cover(p, 1, cur.h, hlo, hhi);
        tdp::axis_range_cover(p, 2, cur.x0, cur.x0 + cur.xbu, wlo, whi);
        for (int i_f = flo; i_f <= fhi; ++i_f) {
            const int k = cur.f - p.start[0][i_f];
            for (int i_h = hlo; i_h <= hhi; ++i_h) {
                const TileRow tr_ = tile_row(p, a.B, cur.b, i_f, i_h, k, cur.h - p.start[1][i_h]);
                for (int i_w = wlo; i_w <= whi; ++i_w) {
                    const int w0 = p.start[2][i_w];
                    const int sb = min(p.end[2][i_w], cur.x0 + cur.xbu);
                    const long long row = row_token(p, tr_, i_w) - w0;   // + global column
                    int x = max(w0, cur.x0) + tq, j = tr;
                    while (x < sb) {
                        const int xl = x - cur.x0;
                        dst[(row + x) * J + j] = sbuf[xl * J + swz_extract<PAIR>(j, xl, a.pmask, J)];
                        x += sx2;
                        j += sj2;
                        if (j >= J) {
                            j -= J;
                            ++x;
                        }
                    }
                }
            }
        }
        __syncthreads();
        if (un >= a.units) break;
        u = un;
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ blend
template <typename T> struct Elems;
template <> struct Elems<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static __device__ __forceinline__ void fma_into(float (&acc)[8], const uint4& v, float w) {
        const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
            acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xffff0000u), acc[2 * i + 1]);
        }
    }
};
template <> struct Elems<float> {
    static constexpr int kVec = 4;
    static __device__ __forceinline__ void fma_into(float (&acc)[4], const uint4& v, float w) {
        acc[0] = fmaf(w, __uint_as_float(v.x), acc[0]);
        acc[1] = fmaf(w, __uint_as_float(v.y), acc[1]);
        acc[2] = fmaf(w, __uint_as_float(v.z), acc[2]);
        acc[3] = fmaf(w, __uint_as_float(v.w), acc[3]);
    }
};

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Pass 1: every thread owns ipt 16-byte chunks of one column's token (its
// chunks lit, lit + lpt, ...; lpt threads share a token, so a warp reads
// contiguous 16*lpt-byte pieces of 32/lpt tokens per load) and accumulates,
// in fp32 registers, the weighted tokens of every tile covering the column:
// one address per covering column tile, and all of one (frame tile, row
// tile) pair's loads issued before any is used.  The sums go to shared
// memory as fp32 [column][C]; pass 2 writes the C latent row segments, a
// warp storing 32 neighbouring columns of one channel.  With bf16 tokens a
// chunk j holds two fp32 chunks, kept at j and J + j.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kTmThreads, 3) blend_tokens_kernel(const __grid_constant__ tdp_plan_t p,
                                                                     const TmArgs a) {
    constexpr int VEC = Elems<Tin>::kVec;
    constexpr int FCH = VEC / 4;          // fp32 chunks per 16-byte chunk
    __shared__ float4 sacc[2 * kTmChunks];
    const uint4* __restrict__ src = static_cast<const uint4*>(a.src);
    Tout* __restrict__ out = static_cast<Tout*>(a.dst);
    const int tid = threadIdx.x;
    const int J = a.J, lpt = a.lpt, ipt = a.ipt;
    const int xcol = tid / lpt, lit = tid - xcol * lpt;   // the thread's column in a unit, its first chunk

    // the column's first covering column tile, how many cover it, and the
    // first kTmKw of their column weights
    int wlo = 0, ncov = 0;
    float ww[kTmKw];
#pragma unroll
    for (int q = 0; q < kTmKw; ++q) ww[q] = 0.0f;
    int cached_x0 = -1;
    // pass 2: columns per pass, the thread's first column and channel group, and the group step
    int c_xbu = -1, xt = 1, x2 = 0, q2 = 0, sq2 = 1;

    pdl_wait();
    int u = blockIdx.x;
    UnitWalk walk = unit_walk(p, a, min(u, a.units - 1), gridDim.x);
    for (; u < a.units; u += gridDim.x, unit_next(p, a, walk)) {
        const Unit U = unit_of(p, a, walk);
        const bool mine = xcol < U.xbu;
        if (U.x0 != cached_x0) {
            cached_x0 = U.x0;
            ncov = 0;
            wlo = 0;
            if (mine) {
                const int w = U.x0 + xcol;
                int lo, hi;
                tdp::axis_cover(p, 2, w, lo, hi);
                wlo = lo;
                ncov = hi - lo + 1;
#pragma unroll
                for (int q = 0; q < kTmKw; ++q) ww[q] = axis_weight(p, 2, min(lo + q, hi), w);
            }
        }

        float acc[kTmItems][VEC];
#pragma unroll
        for (int r = 0; r < kTmItems; ++r)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[r][e] = 0.0f;

        int flo, fhi, hlo, hhi;
        tdp::axis_cover(p, 0, U.f, flo, fhi);
        tdp::axis_cover(p, 1, U.h, hlo, hhi);
        const int w = U.x0 + xcol;
        for (int i_f = flo; i_f <= fhi; ++i_f) {
            const float wf = axis_weight(p, 0, i_f, U.f);
            const int k = U.f - p.start[0][i_f];
            for (int i_h = hlo; i_h <= hhi; ++i_h) {
                const float wfh = __fmul_rn(wf, axis_weight(p, 1, i_h, U.h));
                const TileRow tr_ = tile_row(p, a.B, U.b, i_f, i_h, k, U.h - p.start[1][i_h]);
                uint4 v[kTmKw][kTmItems];
#pragma unroll
                for (int q = 0; q < kTmKw; ++q)
                    if (q < ncov) {
                        const int i_w = wlo + q;
                        const uint4* s = src + (row_token(p, tr_, i_w) + (w - p.start[2][i_w])) * J + lit;
#pragma unroll
                        for (int r = 0; r < kTmItems; ++r)
                            if (r < ipt) v[q][r] = __ldg(s + r * lpt);
                    }
#pragma unroll
                for (int q = 0; q < kTmKw; ++q)
                    if (q < ncov) {
                        const float wq = __fmul_rn(wfh, ww[q]);
#pragma unroll
                        for (int r = 0; r < kTmItems; ++r)
                            if (r < ipt) Elems<Tin>::fma_into(acc[r], v[q][r], wq);
                    }
                // Columns covered by more than kTmKw column tiles (only when
                // the partition-of-unity guard is off): one tile at a time.
                for (int i_w = wlo + kTmKw; i_w < wlo + ncov; ++i_w) {
                    const uint4* s = src + (row_token(p, tr_, i_w) + (w - p.start[2][i_w])) * J + lit;
                    const float wq = __fmul_rn(wfh, axis_weight(p, 2, i_w, w));
#pragma unroll
                    for (int r = 0; r < kTmItems; ++r)
                        if (r < ipt) Elems<Tin>::fma_into(acc[r], __ldg(s + r * lpt), wq);
                }
            }
        }

        if (mine) {
#pragma unroll
            for (int r = 0; r < kTmItems; ++r) {
                if (r >= ipt) break;
                const int j = lit + r * lpt;
#pragma unroll
                for (int c = 0; c < FCH; ++c)
                    sacc[xcol * a.jf + swzf(c * J + j, xcol, a.pfmask, a.jf)] =
                        make_float4(acc[r][4 * c], acc[r][4 * c + 1], acc[r][4 * c + 2], acc[r][4 * c + 3]);
            }
        }
        __syncthreads();

        if (U.xbu != c_xbu) {
            c_xbu = U.xbu;
            xt = min(c_xbu, kTmThreads);
            x2 = tid % xt;
            q2 = tid / xt;
            sq2 = kTmThreads / xt;
        }
        if (q2 < sq2) {
            Tout* const orow = out + latent_row(p, a, U);
            const long long qstride = 4LL * sq2 * a.fhw;
            for (int x = x2; x < U.xbu; x += xt) {
                Tout* o = orow + 4LL * q2 * a.fhw + x;
                for (int qc = q2; qc < a.jf; qc += sq2, o += qstride) {
                    // channels 4qc..4qc+3: chunk qc / FCH, its fp32 half qc % FCH
                    const int slot = FCH == 2 ? ((qc & 1) * J + (qc >> 1)) : qc;
                    const float4 s = sacc[x * a.jf + swzf(slot, x, a.pfmask, a.jf)];
                    store_out(o, s.x);
                    store_out(o + a.fhw, s.y);
                    store_out(o + 2 * a.fhw, s.z);
                    store_out(o + 3 * a.fhw, s.w);
                }
            }
        }
        __syncthreads();
    }
    pdl_launch_dependents();
}

// =================================================================== host side
bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }
int dtype_size(tdp_dtype d) { return d == TDP_F32 ? 4 : (d == TDP_BF16 ? 2 : 0); }
int swizzle_mask(int chunks) {
    int m = 1;
    while (m * 2 <= std::min(chunks, 8)) m *= 2;
    return m - 1;
}

// Unit geometry of both calls; `esz` is the token-major element size.
// Extract: kTmChunks chunks per unit.  Blend: one column per lpt threads.
tdp_status tm_args(const tdp_plan_t& p, int B, int C, int esz, bool blend, TmArgs& a) {
    if ((static_cast<long long>(C) * esz) % 16 != 0) return TDP_ERR_UNSUPPORTED;
    const long long J = static_cast<long long>(C) * esz / 16;
    if (J > kTmChunks) return TDP_ERR_UNSUPPORTED;
    a.ipt = J % 4 == 0 ? 4 : (J % 2 == 0 ? 2 : 1);
    a.lpt = static_cast<int>(J / a.ipt);
    if (blend && a.lpt > kTmThreads) return TDP_ERR_UNSUPPORTED;
    const int W = p.dims[2];
    const int xb_max = blend ? kTmThreads / a.lpt : static_cast<int>(kTmChunks / J);
    const int nxb = (W + xb_max - 1) / xb_max;
    const int xb = (W + nxb - 1) / nxb;   // balanced column blocks
    const long long units = static_cast<long long>(B) * p.dims[0] * p.dims[1] * nxb;
    if (units > INT_MAX || static_cast<long long>(B) * C > INT_MAX) return TDP_ERR_INVALID_ARG;
    a.fhw = static_cast<long long>(p.dims[0]) * p.dims[1] * W;
    a.B = B;
    a.C = C;
    a.J = static_cast<int>(J);
    a.jf = C / 4;
    a.pmask = swizzle_mask(a.J);
    a.pfmask = swizzle_mask(a.jf);
    a.xb = xb;
    a.nxb = nxb;
    a.units = static_cast<int>(units);
    return TDP_OK;
}

template <typename K>
tdp_status tm_launch(K kernel, const tdp_plan_t& p, const TmArgs& a, cudaStream_t stream) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kTmThreads, 0);
    if (e != cudaSuccess) return tdp::record_cuda(e);
    const long long slots = static_cast<long long>(std::max(1, per_sm)) * std::max(1, tdp::device_sm_count());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<long long>(a.units, slots)), 1, 1);
    cfg.blockDim = dim3(kTmThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return tdp::record_cuda(cudaLaunchKernelEx(&cfg, kernel, p, a));
}

}  // namespace

extern "C" {

tdp_status tdp_extract_tokens(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype, const void* latent,
                              void* tokens, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || C < 0) return TDP_ERR_INVALID_ARG;
    const int esz = dtype_size(dtype);
    if (!esz) return TDP_ERR_INVALID_ARG;
    if (B == 0 || C == 0) return TDP_OK;
    if (!latent || !tokens) return TDP_ERR_INVALID_ARG;
    if (!aligned16(latent) || !aligned16(tokens)) return TDP_ERR_ALIGNMENT;
    TmArgs a{};
    tdp_status st = tm_args(*plan, B, C, esz, false, a);
    if (st != TDP_OK) return st;
    a.src = latent;
    a.dst = tokens;
    // column pairs: every row and every column block start on an even column
    const bool pair = plan->dims[2] % 2 == 0 && a.xb % 2 == 0;
    if (esz == 2)
        return pair ? tm_launch(extract_tokens_kernel<uint16_t, true>, *plan, a, stream)
                    : tm_launch(extract_tokens_kernel<uint16_t, false>, *plan, a, stream);
    return pair ? tm_launch(extract_tokens_kernel<uint32_t, true>, *plan, a, stream)
                : tm_launch(extract_tokens_kernel<uint32_t, false>, *plan, a, stream);
}

tdp_status tdp_blend_tokens(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype in_dtype, const void* tokens,
                            tdp_dtype out_dtype, void* out, cudaStream_t stream) {
    if (!tdp::plan_is_valid(plan) || B < 0 || C < 0) return TDP_ERR_INVALID_ARG;
    const int esz = dtype_size(in_dtype);
    if (!esz || !dtype_size(out_dtype)) return TDP_ERR_INVALID_ARG;
    if (B == 0 || C == 0) return TDP_OK;
    if (!tokens || !out) return TDP_ERR_INVALID_ARG;
    if (!aligned16(tokens) || !aligned16(out)) return TDP_ERR_ALIGNMENT;
    TmArgs a{};
    tdp_status st = tm_args(*plan, B, C, esz, true, a);
    if (st != TDP_OK) return st;
    a.src = tokens;
    a.dst = out;
    const bool ib = in_dtype == TDP_BF16, ob = out_dtype == TDP_BF16;
    if (ib && ob) return tm_launch(blend_tokens_kernel<__nv_bfloat16, __nv_bfloat16>, *plan, a, stream);
    if (ib) return tm_launch(blend_tokens_kernel<__nv_bfloat16, float>, *plan, a, stream);
    if (ob) return tm_launch(blend_tokens_kernel<float, __nv_bfloat16>, *plan, a, stream);
    return tm_launch(blend_tokens_kernel<float, float>, *plan, a, stream);
}

}  // extern "C"
