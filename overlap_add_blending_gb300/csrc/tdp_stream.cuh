// Streaming extract and blend.  Included by tdp_kernels.cu inside its
// anonymous namespace, after the barrier and launch helpers.
//
// Source: "Tiled Data Parallelism (TDP)", What it is -- each tile is the
// latent's sub-box (extract), and the tiles' outputs are recombined with
// separable trapezoidal masks that sum to 1 (blend); the split and window
// are those the mold issue #673 measures ("A bug found while porting").
//
// Layout facts the design rests on (dense packed tiles [T][B,C,f,h,w]):
//   * a latent row (W elements) is 16-byte aligned whenever W * esz is a
//     multiple of 16, so a band of latent rows is one aligned span, and
//     blend output rows are whole 16-byte chunks;
//   * a tile row is generally NOT 16-byte aligned (a bf16 row of 39
//     elements is 78 bytes), but the rows of one tile slice inside a row
//     band are contiguous: a run, staged as the 16-byte chunks around it,
//     its bytes keeping their address mod 16.
// The realignment between the two is left to the shared-memory load unit,
// which reads 2-byte elements and 4-byte words at any address of their
// size: extract writes the packed tiles in coalesced 8-byte groups, each
// element loaded from the staged band on its own; blend reads a term's
// window of tile elements as 32-bit words joined by one byte permute each,
// and writes the latent as 16-byte chunks, one per thread.
//
// Work units are (b*C + c, frame, row band) boxes of the latent, numbered
// u = (f * nbands + band) * BC + bc, so that consecutive units share their
// tile geometry.  CTA i (one per SM) takes units [split[i], split[i+1]), a
// contiguous range the host balances by bytes moved.  One producer warp
// stages units ahead into a ring of fixed-size shared-memory stages with
// bulk copies (cp.async.bulk, completing on the stage's "full" mbarrier);
// the compute warps release a stage on its "empty" mbarrier.  Plan-only
// tables -- covers and 1-D trapezoid weights per frame and row, run offsets
// per band, each blend thread's column terms -- are built once per launch
// on the host (IEEE fp32, the same values the device computes) and passed
// with the launch.  Every wait is bounded (kWaitNs); after a timeout a
// kernel records a code in the device error word, lets its own copies land
// (bounded, with a distinct code if they do not) and returns.

constexpr int kStreamExtractWarps = 24;   // compute warps; one more warp stages
constexpr int kStreamBlendWarps = 19;   // 20 warps with the producer: 5 per SM sub-partition at up to 96 registers
constexpr int kStreamExtractThreads = 32 * (kStreamExtractWarps + 1);
constexpr int kStreamBlendThreads = 32 * (kStreamBlendWarps + 1);
constexpr int kStreamMaxStageRuns = 64;     // blend: runs per stage, two per producer lane

constexpr int kStreamMaxStages = 8;
constexpr int kStreamMaxGrid = 256;        // CTAs the split table holds (one per SM)
constexpr int kStreamTableWords = 512;     // 16-byte words of plan tables passed with a launch
constexpr int kStreamPad = 32;             // guard bytes before and after a stage's data

struct StreamSplit {
    int start[kStreamMaxGrid + 1];   // CTA i: units [start[i], start[i+1])
};

struct StreamTables {
    uint4 w[kStreamTableWords];
};

// ------------------------------------------------------------------ table entries
// Row band: its rows [hb0, hb1) and the row tiles meeting it, [ihlo, ihlo + NHB).
struct __align__(16) BandEnt {
    int hb0, hb1, ihlo, NHB;
};

// Covering tiles of one frame: the first, their count (<= 2) and r_f.
struct __align__(16) FrameEnt {
    int lo, n;
    float w[2];
};

// Covering tiles of one row: the first, their count (<= 2) and r_h.
struct __align__(16) RowEnt {
    int lo, n;
    float w[2];
};

// Per frame tile: the packed offset of its first (row tile, column tile)
// block per b*C + c element, its size and its first frame.
struct __align__(16) FrameCon {
    long long base;   // prefix_f(i_f) * (sum of row-tile sizes) * (sum of column-tile sizes)
    int sf, fs;
};

// Per column tile (extract): width, first column, the step of one warp
// pass over a span (32 groups of 8 bytes) in (tile rows, columns), and
// 1 / width.
struct __align__(16) ColCon {
    int sw, ws, dq, dr;
    float inv_sw;
    int pad[3];
};

// One (row tile meeting a band, column tile) run of a band: everything of
// its packed offset that does not depend on the frame tile, b*C + c or the
// frame.  Its element offset for frame tile i_f, slice bc and frame f is
//   BC * (base_f + sf * A) + (bc * sf + f - fs) * slice + vrow.
struct __align__(16) RunEnt {
    long long A;      // prefix_h(i_h) * (sum of column-tile sizes) + h_t * prefix_w(i_w)
    int slice;        // h_t * w_t: elements of one (bc, frame) slice of the tile
    int vrow;         // (first band row - tile's first row) * w_t
    int len;          // elements of the run (its rows times w_t)
    int src_rel;      // extract: byte offset of the run's (row 0, column 0) in the staged band
    int iw;           // its column tile
    int r0b;          // blend: its first row (a latent row) times its tile row's bytes
};

// Blend: the column tiles ("terms") touching one 16-byte output chunk, each
// with its tile row's bytes and the chunk's byte offset in the tile row
// (may be negative), r_w per column (0 where the tile does not reach) and
// the columns it reaches (bit m: column m of the chunk).  The entries are
// ordered by class -- 0: one term reaching every column with r_w = 1; 1:
// one term otherwise; 2, 3: two, three terms -- and `col` is the chunk
// column an entry describes.
struct __align__(16) ChunkEnt {
    int nq;
    int iw[3], swb[3], xob[3];
    float rw[3][8];
    uint32_t in[3];
    int col, cls;
};
constexpr int kChunkClasses = 4;

struct StreamArgs {
    const void* src;          // extract: latent; blend: packed tiles
    void* dst;                // extract: packed tiles; blend: latent
    long long src_bytes;      // size of the source buffer (blend: its last 16-byte chunk may be partial)
    long long dst_bytes;      // size of the destination buffer (index checks of debug builds)
    int F, H, W, nw;          // latent frames, rows, columns; column tiles
    int BC, band_rows, nbands, n_units;
    int row0, row1;           // the rows [row0, row1) the bands cover (the whole H but for a slab blend,
                              // whose output holds rows row0.. of each (b, c, f) plane)
    int nstages, stage_bytes;
    int run_slot, max_runs, runs_per_band;   // blend: shared bytes per staged run, runs per unit, per band
    int cpr;                  // blend: 16-byte chunks per latent row
    int tfirst[4], grp[4], gstep[4];   // blend, per chunk class: first compute thread, row groups (threads
                                       // per entry), the groups' step per unit
    int cwarps;                        // blend: compute warps holding chunk entries (the rest return at once)
    int ncls[4];              // blend: chunk entries per class, in table order
    int esz;                  // element size of the staged data (extract: latent; blend: tiles)
    // tables, as 16-byte word offsets into StreamTables (and its shared copy)
    int t_band, t_frame, t_row, t_fcon, t_wcon, t_runs, t_chunk, t_words;
    int off_full, off_empty, off_tab, off_hdr, off_data;   // shared layout (bytes)
};

// Work the extract launch does besides its units in tdp_extract_and_tokens:
// the partial extents of the (tile, batch) pairs' token chunks (the first
// pass of the token steps, spread over the grid; the second launch of the
// call finishes them).  The compute warps of a CTA with chunks reduce them
// first, while its producer warp already stages the CTA's first units; the
// host's split gives that CTA correspondingly fewer units.
constexpr int kJobNone = 0, kJobExtent = 1;
constexpr int kChunkLead = 5;   // units before a CTA's last at which its last chunk's loads are issued
struct StreamJobs {
    static constexpr bool kEnabled = true;
    int kind;                       // kJobNone or kJobExtent
    int B;                          // pair j is (tile j / B, batch j % B)
    int K1;                         // chunks per pair: chunk q is pair q / K1, part q % K1
    int off_job;                    // shared offset of the chunks' scratch (bytes)
    int start[kStreamMaxGrid + 1];  // CTA i reduces chunks [start[i], start[i + 1])
    const int* gen;                 // generated positions [B, 3, N, 2]
    int* partials;                  // [pairs * K1][6]: per chunk, min start / max end per axis
    int* zero_a;                    // CTA 0 sets zero_a[0, nzero_a) and zero_b[0, nzero_b) to 0
    int* zero_b;                    // (the finishing launch's counters)
    int nzero_a, nzero_b;
    tdp_plan_t p;
};

// The launch argument of an extract without jobs (a plain tdp_extract): a
// separate instantiation, so that it carries neither the job parameters
// nor their registers.
struct NoJobs {
    static constexpr bool kEnabled = false;
};

// Ints the extract launch sets to zero for the launch after it.
struct StreamZero {
    int* a;
    int na;
    int* b;
    int nb;
};

static_assert(sizeof(StreamArgs) + sizeof(StreamSplit) + sizeof(StreamTables) + sizeof(StreamJobs) <= 32764,
              "streaming kernel parameters fit the 32 KB parameter space");
static_assert(kChunkTokens == kJobTokenBatch * 32 * kStreamExtractWarps,
              "an extent chunk is one batch of loads per extract compute thread");

// ------------------------------------------------------------------ device helpers
// Raise the transaction count of the barrier's current phase without
// arriving (the bulk copies issued after it complete against it).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Bounded wait for the copies of units [k0, k1) of a ring of S stages to
// land (after a timeout, so that no copy is still writing shared memory
// when the CTA exits).  Records kErrDrain if they do not.
__device__ __forceinline__ void drain_stages(uint64_t* full, int S, int k0, int k1) {
    for (int k = k0; k < k1; ++k)
        if (!mbar_wait_bounded(&full[k % S], (k / S) & 1)) atomicOr(&g_device_error, kErrDrain);
}

// NW words of the bytes at shared offset `a` (a multiple of ESZ), read as
// 32-bit words: for 2-byte elements at a 2-mod-4 offset, NW + 1 aligned
// words joined pairwise by a byte permute (the load unit does the rest of
// the alignment).
template <int ESZ, int NW>
__device__ __forceinline__ void lds_words_at(const unsigned char* smem, uint32_t a, uint32_t (&w)[NW]) {
    if constexpr (ESZ == 4) {
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = *reinterpret_cast<const uint32_t*>(smem + a + 4u * k);
    } else {
        const uint32_t b = a & ~3u;
        uint32_t r[NW + 1];
#pragma unroll
        for (int k = 0; k <= NW; ++k) r[k] = *reinterpret_cast<const uint32_t*>(smem + b + 4u * k);
        const uint32_t sel = (a & 2u) ? 0x5432u : 0x3210u;
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = __byte_perm(r[k], r[k + 1], sel);
    }
}

// A 16-byte store of output written once (streaming: evict-first in L2).
__device__ __forceinline__ void stg_u4(void* p, const uint4& v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// A position in the ring of S stages: use j of the ring is stage j mod S
// in its (j / S)-th round, whose parity is the phase a "full" wait on that
// stage expects (and the one before it, the phase of the "empty" wait
// before the stage is refilled).  Kept incrementally, without dividing.
struct RingPos {
    int s = 0;          // stage
    uint32_t ph = 0u;   // parity of the round
    __device__ __forceinline__ void next(int S) {
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Decodes unit u = (f * nbands + band) * BC + bc into (bc, f, band) and
// steps to u + 1 without dividing.
struct UnitCursor {
    int bc, f, band, BC, nbands;
    __device__ __forceinline__ void init(int u, int BC_, int nbands_) {
        BC = BC_;
        nbands = nbands_;
        bc = u % BC;
        const int g = u / BC;
        band = g % nbands;
        f = g / nbands;
    }
    __device__ __forceinline__ void next() {
        if (++bc == BC) {
            bc = 0;
            if (++band == nbands) { band = 0; ++f; }
        }
    }
};

// Element offset in the packed tiles of a run (an entry of the run table)
// for frame tile fc, slice bc and frame f.
__device__ __forceinline__ long long run_e0(const RunEnt& r, const FrameCon& fc, int BC, int bc, int f) {
    return (long long)BC * (fc.base + (long long)fc.sf * r.A) + ((long long)bc * fc.sf + (f - fc.fs)) * r.slice +
           r.vrow;
}

// The CTA's shared memory: ring barriers, the table copy, run-base entries
// (blend) and the ring.
struct StreamSmem {
    uint64_t* full;            // [nstages]
    uint64_t* empty;           // [nstages]
    const BandEnt* bands;      // [nbands]
    const FrameEnt* frames;    // [F]
    const RowEnt* rows;        // [H] (blend)
    const FrameCon* fcon;      // [n_f]
    const ColCon* wcon;        // [n_w] (extract)
    const RunEnt* runs;        // [nbands][runs_per_band]
    const ChunkEnt* chunks;    // [cpr] (blend)
};

// Common prologue: the tables into shared memory, the ring barriers, then
// the wait for the previous kernel in the stream (programmatic dependent
// launch), so that only this set-up overlaps it and no thread touches
// global data before it completes.  `full_count`: producer arrivals that
// complete a stage; `warps`: compute warps that release one.
__device__ __forceinline__ StreamSmem stream_prologue(const StreamArgs& a, const StreamTables& tb, unsigned char* smem,
                                                      uint32_t full_count, uint32_t warps) {
    pdl_launch_dependents();
    uint4* tab = reinterpret_cast<uint4*>(smem + a.off_tab);
    for (int i = threadIdx.x; i < a.t_words; i += blockDim.x) tab[i] = tb.w[i];
    StreamSmem m;
    m.full = reinterpret_cast<uint64_t*>(smem + a.off_full);
    m.empty = reinterpret_cast<uint64_t*>(smem + a.off_empty);
    m.bands = reinterpret_cast<const BandEnt*>(tab + a.t_band);
    m.frames = reinterpret_cast<const FrameEnt*>(tab + a.t_frame);
    m.rows = reinterpret_cast<const RowEnt*>(tab + a.t_row);
    m.fcon = reinterpret_cast<const FrameCon*>(tab + a.t_fcon);
    m.wcon = reinterpret_cast<const ColCon*>(tab + a.t_wcon);
    m.runs = reinterpret_cast<const RunEnt*>(tab + a.t_runs);
    m.chunks = reinterpret_cast<const ChunkEnt*>(tab + a.t_chunk);
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nstages; ++s) {
            mbar_init(&m.full[s], full_count);
            mbar_init(&m.empty[s], warps);
        }
        mbar_init_done();
    }
    __syncthreads();
    pdl_wait();
    return m;
}

// =================================================================== extract
// Staging: the band's latent rows, one contiguous aligned span, one bulk
// copy by the producer warp's lane 0 (evict-first in L2: read once, while
// the tiles written here are read next by the blend).
// Writing: for every covering (frame tile, row tile, column tile), the run
// of that tile's rows inside the band is a contiguous span of the packed
// tiles.  The spans of successive units are dealt to the warps round robin
// (a unit's first span goes to the warp after the one that took the
// previous unit's last); lane l writes the span's
// 8-byte groups l, l + 32, ... (coalesced 256-byte warp stores) from its
// first 8-byte boundary on.  A group is four bf16 elements (two fp32), each
// loaded from the staged band at its own address -- the shared load does
// the realignment -- and those past the end of a tile row come from the
// next one, W - w_t latent columns further on.  A lane tracks its group's
// (row, column) and band address incrementally.  The few elements before
// the first boundary and after the last whole group are written one by one
// by lanes 0-7 and 8-15.
template <typename E, typename J>
__global__ void __launch_bounds__(kStreamExtractThreads, 1)
    extract_stream_kernel(const __grid_constant__ StreamArgs a, const __grid_constant__ StreamSplit sp,
                          const __grid_constant__ StreamTables tb, const __grid_constant__ J jb) {
    constexpr int esz = static_cast<int>(sizeof(E));
    constexpr int EPQ = 8 / esz;   // elements per 8-byte group
    constexpr int kWarps = kStreamExtractWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    const StreamSmem m = stream_prologue(a, tb, smem, 1, kWarps);
    const int first = sp.start[blockIdx.x], last = sp.start[blockIdx.x + 1];
    int job0 = 0, job1 = 0;
    bool zeroes = false;
    if constexpr (J::kEnabled) {
        job0 = jb.kind == kJobExtent ? jb.start[blockIdx.x] : 0;
        job1 = jb.kind == kJobExtent ? jb.start[blockIdx.x + 1] : 0;
        zeroes = jb.kind == kJobExtent && blockIdx.x == 0;
    }
    if (first >= last && job0 >= job1 && !zeroes) return;
    const int S = a.nstages, n = last - first;
    const int F = a.F, H = a.H, W = a.W, nw = a.nw;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kWarps) {
        // ---- producer: lane 0 stages one latent band per unit
        if (lane != 0) return;
        const unsigned char* lat = static_cast<const unsigned char*>(a.src);
        UnitCursor cs;
        cs.init(first, a.BC, a.nbands);
        int k = 0;
        RingPos rp;
        bool ok = true;
        for (; k < n; ++k, cs.next(), rp.next(S)) {
            const int s = rp.s;
            if (k >= S && !mbar_wait_backoff(&m.empty[s], rp.ph ^ 1u)) { ok = false; break; }
            const BandEnt b = m.bands[cs.band];
            const uint32_t bytes = static_cast<uint32_t>((b.hb1 - b.hb0) * W * esz);
            const unsigned char* g = lat + (((long long)cs.bc * F + cs.f) * H + b.hb0) * (long long)W * esz;
            const bool in = !range_bad(g, bytes, a.src, a.src_bytes) &&
                            !index_bad(static_cast<int>(bytes) > a.stage_bytes - 2 * kStreamPad);
            fence_proxy_async();   // the compute warps' reads of this stage come before the copy's writes
            mbar_arrive_expect_tx(&m.full[s], in ? bytes : 0u);
            if (in) bulk_copy_g2s_once(smem + a.off_data + s * a.stage_bytes + kStreamPad, g, bytes, &m.full[s]);
        }
        if (!ok) {
            atomicOr(&g_device_error, kErrExtractWait);
            drain_stages(m.full, S, max(0, k - S), k);   // the copies still in flight
        }
        return;
    }

    // ---- compute warps: the CTA's token chunks and units.  Chunks before
    // the last are reduced first; the last one's loads are issued
    // kChunkLead units before the end and each warp reduces its share two
    // units before the end, into the chunk's slot with atomics, so that
    // the loads' latency hides behind the units and no barrier stops the
    // warps.
    using G = WarpsGroup<32 * kWarps>;
    int* jsh = nullptr;
    int2* cdata = nullptr;
    bool async_chunk = false;
    if constexpr (J::kEnabled) {
        jsh = reinterpret_cast<int*>(smem + jb.off_job);
        cdata = reinterpret_cast<int2*>(smem + jb.off_job + 4 * kChunkShInts);
        if (zeroes) {
            for (int i = threadIdx.x; i < jb.nzero_a; i += 32 * kWarps) jb.zero_a[i] = 0;
            for (int i = threadIdx.x; i < jb.nzero_b; i += 32 * kWarps) jb.zero_b[i] = 0;
        }
        async_chunk = job1 > job0;
        for (int q = job0; q < job1 - 1; ++q) extent_chunk<G>(jb.p, jb.gen, jb.B, jb.K1, q, jb.partials, jsh);
        if (async_chunk) {
            chunk_slot_init(jb.partials, job1 - 1);
            G::sync();   // the slot is set before any warp adds to it
        }
    }
    const int k_issue = max(0, n - kChunkLead);         // the last chunk's loads go out before this unit
    const int k_fin = max(k_issue, n - 2);               // and each warp reduces its share after this one
    bool chunk_done = !async_chunk;
    if constexpr (J::kEnabled) {
        if (async_chunk && n == 0) extent_chunk_issue<G>(jb.p, jb.gen, jb.B, jb.K1, job1 - 1, cdata);
    }
    unsigned char* tiles = static_cast<unsigned char*>(a.dst);
    UnitCursor c;
    c.init(first, a.BC, a.nbands);
    int rot = 0;   // the warp that takes the unit's first span: the spans are dealt round robin across units
    RingPos rp;
    for (int k = 0; k < n; ++k, c.next(), rp.next(S)) {
        if constexpr (J::kEnabled) {
            if (async_chunk && k == k_issue) extent_chunk_issue<G>(jb.p, jb.gen, jb.B, jb.K1, job1 - 1, cdata);
        }
        const int s = rp.s;
        if (!mbar_wait_bounded(&m.full[s], rp.ph)) {
            if (lane == 0) atomicOr(&g_device_error, kErrExtractWait);
            break;   // no release: the producer gives up and drains (the chunk below still meets its barriers)
        }
        const BandEnt b = m.bands[c.band];
        const FrameEnt fe = m.frames[c.f];
        const int nr = b.NHB * nw, nspans = fe.n * nr;
        const RunEnt* band_runs = m.runs + c.band * a.runs_per_band;
        const uint32_t band_off = static_cast<uint32_t>(a.off_data + s * a.stage_bytes + kStreamPad);
        const uint32_t band_end = band_off + static_cast<uint32_t>((b.hb1 - b.hb0) * W * esz);   // (index checks)
        int spn = warp - rot;
        if (spn < 0) spn += kWarps;
        rot = (rot + nspans) % kWarps;
#pragma unroll 1
        for (; spn < nspans; spn += kWarps) {
            const int fa = spn >= nr ? 1 : 0, rr = spn - fa * nr;
            const RunEnt re = band_runs[rr];
            const int iw = re.iw;
            const ColCon wc = m.wcon[iw];
            const int sw = wc.sw, len = re.len;
            E* g0 = reinterpret_cast<E*>(tiles) + run_e0(re, m.fcon[fe.lo + fa], a.BC, c.bc, c.f);
            const uint32_t src0 = band_off + static_cast<uint32_t>(re.src_rel);
            const uint32_t wrap = static_cast<uint32_t>((W - sw) * esz);
            // the body: 8-byte groups of EPQ elements from the span's first 8-byte
            // boundary on; the elements before it (head) and after the last
            // whole group (tail) are written one by one
            const int hd = static_cast<int>(((8u - (reinterpret_cast<uintptr_t>(g0) & 7u)) & 7u) / esz);
            const int nq = len > hd ? (len - hd) / EPQ : 0;
            int qi = lane;
            if (qi < nq) {
                // (x, ad): tile column and band offset of the group's first element
                const int e = hd + EPQ * qi;
                const int y = small_div(e, wc.inv_sw);
                int x = e - y * sw;
                uint32_t ad = src0 + static_cast<uint32_t>((y * W + x) * esz);
                const uint32_t step = static_cast<uint32_t>((wc.dq * W + wc.dr) * esz);
                uint2* dst = reinterpret_cast<uint2*>(g0 + e);
#pragma unroll 1
                for (; qi < nq; qi += 32) {
                    // element m of the group sits m elements on, or, from the
                    // first one past the tile row on, W - w_t columns further
                    const int k1 = sw - x;
                    uint2 v;
                    if constexpr (kDebugChecks) {
                        // the group's loads rise from ad to its last element's; its store is 8 bytes
                        const uint32_t last = ad + static_cast<uint32_t>((EPQ - 1) * esz) + (k1 <= EPQ - 1 ? wrap : 0u);
                        if (index_bad(ad < band_off || last + esz > band_end) ||
                            range_bad(dst, 8, tiles, a.dst_bytes))
                            break;
                    }
                    if constexpr (esz == 2) {
                        const uint32_t e0 = *reinterpret_cast<const uint16_t*>(smem + ad);
                        const uint32_t e1 = *reinterpret_cast<const uint16_t*>(smem + ad + 2u + (k1 <= 1 ? wrap : 0u));
                        const uint32_t e2 = *reinterpret_cast<const uint16_t*>(smem + ad + 4u + (k1 <= 2 ? wrap : 0u));
                        const uint32_t e3 = *reinterpret_cast<const uint16_t*>(smem + ad + 6u + (k1 <= 3 ? wrap : 0u));
                        v.x = __byte_perm(e0, e1, 0x5410u);
                        v.y = __byte_perm(e2, e3, 0x5410u);
                    } else {
                        v.x = *reinterpret_cast<const uint32_t*>(smem + ad);
                        v.y = *reinterpret_cast<const uint32_t*>(smem + ad + 4u + (k1 <= 1 ? wrap : 0u));
                    }
                    *dst = v;
                    dst += 32;
                    x += wc.dr;
                    ad += step;
                    if (x >= sw) {
                        x -= sw;
                        ad += wrap;
                    }
                }
            }
            // head elements (lanes 0 .. hd-1) and tail elements (lanes 8 ..)
            const int tl = len - hd - EPQ * nq;
            const int eh = lane < 8 ? lane : hd + EPQ * nq + (lane - 8);
            if ((lane < 8 && lane < hd && lane < len) || (lane >= 8 && lane - 8 < tl)) {
                const int y = small_div(eh, wc.inv_sw), x = eh - y * sw;
                const uint32_t sa = src0 + static_cast<uint32_t>((y * W + x) * esz);
                if (!index_bad(sa < band_off || sa + esz > band_end) && !range_bad(g0 + eh, esz, tiles, a.dst_bytes))
                    g0[eh] = *reinterpret_cast<const E*>(smem + sa);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.empty[s]);
        if constexpr (J::kEnabled) {
            if (k == k_fin && !chunk_done) {
                extent_chunk_finish<G>(jb.p, jb.B, jb.K1, job1 - 1, cdata, jb.partials);
                chunk_done = true;
            }
        }
    }
    // (a CTA without units, or a warp that gave up waiting: its copies
    // must land before the CTA's shared memory goes)
    if constexpr (J::kEnabled) {
        if (!chunk_done) extent_chunk_finish<G>(jb.p, jb.B, jb.K1, job1 - 1, cdata, jb.partials);
    }
}

// =================================================================== blend
// Staging: one stage per covering frame tile of the unit (a unit of a frame
// two tiles cover takes two consecutive stages).  A stage holds the frame
// tile's runs -- one per (row tile meeting the band, column tile) -- each in
// its own fixed slot, as the 16-byte chunks around it, one bulk copy per run
// by the producer warp's lanes (lane l takes runs l, l + 32, ...).  A run's base entry (the
// shared offset its slice's tile element (0, 0) would have if the whole
// slice were staged, less the tile's first latent row times its row bytes,
// so that latent row h of the tile starts at entry + h * row bytes) goes to
// the run-base table; elements in the tile buffer's
// last, partial 16 bytes are loaded plainly.  Lane 0 then arrives once on
// the stage's barrier with the stage's bulk bytes (publishing the warp's
// entries and plain loads) before the lanes issue their copies: one
// arrival per stage, as every arrival on one barrier is serialised.
// Compute: a thread owns one 16-byte output chunk column j (E = 16 / sizeof
// (Tout) latent columns) for the whole kernel and every G-th row of each
// band from a start that moves on each unit, G the row groups of its
// chunk's class (each class in whole warps of its own).  Its column tiles
// ("terms", at most KT) are fixed, so their offsets, r_w weights and masks
// live in registers.
// Per output row and covering (frame tile, row tile) pair it forms inner =
// sum over terms of r_w * value, then acc = fma(w_fh, inner, acc) with
// w_fh = r_f * r_h rounded: the same weights, grouping and order as the
// window-sum kernel, so the blend of ones equals the window sum bit for
// bit.  Elements of a term's window that its tile does not reach are masked
// to +0 before use (their weight is 0 as well), so whatever the window's
// other bytes hold never reaches the sum.
template <typename Tin, int E, int KT>
struct ColTerms {
    static constexpr int NW = E * static_cast<int>(sizeof(Tin)) / 4;   // raw words per window
    int nq;                 // column tiles touching the chunk (<= KT)
    bool one;               // one term reaching every column of the chunk (no masking needed)
    int iw[KT];             // column tile
    int swb[KT], xob[KT];   // tile row bytes; byte offset of column j*E in the tile row (may be < 0)
    float2 rw[KT][E / 2];   // r_w per column (0 where the tile does not reach)
    uint32_t wmask[KT][NW]; // raw-word masks: ones over the elements the tile reaches
};

template <typename Tin, int E, int KT>
__device__ __forceinline__ void col_terms(const ChunkEnt& c, ColTerms<Tin, E, KT>& t) {
    constexpr int esz = static_cast<int>(sizeof(Tin));
    t.nq = c.nq;
    t.one = c.nq == 1 && c.in[0] == (1u << E) - 1;
#pragma unroll
    for (int q = 0; q < KT; ++q) {
        t.iw[q] = c.iw[q];
        t.swb[q] = c.swb[q];
        t.xob[q] = c.xob[q];
#pragma unroll
        for (int m = 0; m < E; m += 2) t.rw[q][m / 2] = make_float2(c.rw[q][m], c.rw[q][m + 1]);
        const uint32_t in = c.in[q];
#pragma unroll
        for (int w = 0; w < ColTerms<Tin, E, KT>::NW; ++w) {
            if constexpr (esz == 2)
                t.wmask[q][w] = ((in >> (2 * w)) & 1u ? 0x0000ffffu : 0u) | ((in >> (2 * w + 1)) & 1u ? 0xffff0000u : 0u);
            else
                t.wmask[q][w] = (in >> w) & 1u ? 0xffffffffu : 0u;
        }
    }
}

// inner += r_w * (term q's masked window at shared offset `ad`), per fp32
// pair.  MASK false: the term reaches every column of the chunk (its mask is
// all ones), so the window is used as loaded.
template <typename Tin, int E, int KT, bool MASK = true>
__device__ __forceinline__ void add_term(const unsigned char* smem, uint32_t ad, const ColTerms<Tin, E, KT>& t, int q,
                                         float2 (&inner)[E / 2], uint32_t lo, uint32_t hi) {
    constexpr int esz = static_cast<int>(sizeof(Tin));
    constexpr int NW = ColTerms<Tin, E, KT>::NW;
    // (debug builds) the window's aligned words inside the ring [lo, hi)
    if (index_bad((ad & ~3u) < lo || (ad & ~3u) + 4u * (NW + 1) > hi)) return;
    uint32_t w[NW];
    lds_words_at<esz, NW>(smem, ad, w);
    if constexpr (MASK) {
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] &= t.wmask[q][k];
    }
    float2 x[E / 2];
    if constexpr (esz == 2) {
#pragma unroll
        for (int k = 0; k < E / 2; ++k) x[k] = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
    } else {
#pragma unroll
        for (int k = 0; k < E / 2; ++k) x[k] = make_float2(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1]));
    }
#pragma unroll
    for (int k = 0; k < E / 2; ++k) inner[k] = __ffma2_rn(t.rw[q][k], x[k], inner[k]);
}

template <typename Tout, int E>
__device__ __forceinline__ void store_chunk(unsigned char* dst, const float2 (&acc)[E / 2]) {
    if constexpr (sizeof(Tout) == 2) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[k]) : "f"(acc[k].y), "f"(acc[k].x));
        stg_u4(dst, make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        stg_u4(dst, make_uint4(__float_as_uint(acc[0].x), __float_as_uint(acc[0].y), __float_as_uint(acc[1].x),
                               __float_as_uint(acc[1].y)));
    }
}

// The output chunk of a term whose weights are all 1: its elements, as the
// weighted sum computes them (fma(1, x, 0) = x, then rounded to Tout).
template <typename Tin, typename Tout, int E>
__device__ __forceinline__ void copy_chunk(const unsigned char* smem, uint32_t ad, unsigned char* dst, uint32_t lo,
                                           uint32_t hi) {
    constexpr int esz = static_cast<int>(sizeof(Tin));
    constexpr int NW = E * esz / 4;
    if (index_bad((ad & ~3u) < lo || (ad & ~3u) + 4u * (NW + 1) > hi)) return;
    uint32_t w[NW];
    lds_words_at<esz, NW>(smem, ad, w);
    if constexpr (sizeof(Tin) == sizeof(Tout)) {
        stg_u4(dst, make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        float2 acc[E / 2];
        if constexpr (esz == 2) {
#pragma unroll
            for (int k = 0; k < E / 2; ++k) acc[k] = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
        } else {
#pragma unroll
            for (int k = 0; k < E / 2; ++k) acc[k] = make_float2(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1]));
        }
        store_chunk<Tout, E>(dst, acc);
    }
}

// SLAB: the output holds rows row0 .. row1 - 1 of each (b, c, f) plane (a
// slab of tdp_blend_slab) rather than all H (its own instantiation, so that
// the whole-latent blend's code is not touched by the slab's offsets).
template <typename Tin, typename Tout, int KT, bool SLAB>
__global__ void __launch_bounds__(kStreamBlendThreads, 1)
    blend_stream_kernel(const __grid_constant__ StreamArgs a, const __grid_constant__ StreamSplit sp,
                        const __grid_constant__ StreamTables tb) {
    constexpr int esz = static_cast<int>(sizeof(Tin));
    constexpr int osz = static_cast<int>(sizeof(Tout));
    constexpr int E = 16 / osz;   // output elements per chunk
    constexpr int kWarps = kStreamBlendWarps;   // compute warps
    constexpr int q1 = KT > 1 ? 1 : 0, q2 = KT > 2 ? 2 : 0;
    extern __shared__ __align__(128) unsigned char smem[];
    // only the compute warps holding chunk entries release stages
    const StreamSmem m = stream_prologue(a, tb, smem, 1, static_cast<uint32_t>(a.cwarps));
    const int first = sp.start[blockIdx.x], last = sp.start[blockIdx.x + 1];
    if (first >= last) return;
    const int S = a.nstages, n = last - first;
    const int F = a.F, W = a.W, nw = a.nw;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int* const hdr0 = reinterpret_cast<int*>(smem + a.off_hdr);
    if (warp >= a.cwarps && warp < kWarps) return;   // a compute warp without entries

    if (warp == kWarps) {
        // ---- producer warp
        const unsigned char* tiles = static_cast<const unsigned char*>(a.src);
        const uintptr_t base = reinterpret_cast<uintptr_t>(tiles);
        const uintptr_t limit = (base + static_cast<uintptr_t>(a.src_bytes)) & ~uintptr_t(15);
        UnitCursor cs;
        cs.init(first, a.BC, a.nbands);
        int j = 0;   // stages filled so far
        RingPos rp;  // stage j's place in the ring
        bool ok = true;
        for (int k = 0; k < n && ok; ++k, cs.next()) {
            const BandEnt b = m.bands[cs.band];
            const FrameEnt fe = m.frames[cs.f];
            const int nr = b.NHB * nw;
            const RunEnt* band_runs = m.runs + cs.band * a.runs_per_band;
            for (int fa = 0; fa < fe.n; ++fa, ++j, rp.next(S)) {
                const int s = rp.s;
                const bool lane_ok = j < S || mbar_wait_backoff(&m.empty[s], rp.ph ^ 1u);
                if (!__all_sync(0xffffffffu, lane_ok)) { ok = false; break; }
                const FrameCon fc = m.fcon[fe.lo + fa];
                const uint32_t stage_off = static_cast<uint32_t>(a.off_data + s * a.stage_bytes + kStreamPad);
                int* hdr = hdr0 + s * a.max_runs;
                // each lane's runs (at most kRunsPerLane of them): entries and plain tail loads first
                constexpr int kRunsPerLane = kStreamMaxStageRuns / 32;
                uintptr_t cp_lo[kRunsPerLane];
                uint32_t cp_n[kRunsPerLane], cp_slot[kRunsPerLane];
                uint32_t bytes = 0;
#pragma unroll
                for (int i = 0; i < kRunsPerLane; ++i) {
                    const int r = lane + 32 * i;
                    cp_n[i] = 0;
                    if (r >= nr) continue;
                    const RunEnt re = band_runs[r];
                    const uintptr_t g0 = base + static_cast<uintptr_t>(run_e0(re, fc, a.BC, cs.bc, cs.f)) * esz;
                    const uintptr_t g1 = g0 + static_cast<uintptr_t>(re.len) * esz;
                    const uintptr_t lo = g0 & ~uintptr_t(15);
                    const uintptr_t up = (g1 + 15) & ~uintptr_t(15);
                    uintptr_t hi = up <= limit ? up : (g1 & ~uintptr_t(15));   // bulk part; past it, the buffer's tail
                    if (hi < lo) hi = lo;
                    const uint32_t slot = stage_off + static_cast<uint32_t>(r * a.run_slot);
                    if constexpr (kDebugChecks) {
                        // the run's slot inside the stage and the table, its bytes inside the tile buffer
                        const uint32_t stage_end = stage_off + static_cast<uint32_t>(a.stage_bytes - 2 * kStreamPad);
                        const uintptr_t top = hi > g1 ? hi : g1;   // the bulk part or the plain tail, whichever ends later
                        if (index_bad(r >= a.max_runs || slot + static_cast<uint32_t>(top - lo) > stage_end) ||
                            range_bad(reinterpret_cast<const void*>(lo), static_cast<long long>(hi - lo), a.src,
                                      a.src_bytes) ||
                            range_bad(reinterpret_cast<const void*>(g0), static_cast<long long>(g1 - g0), a.src,
                                      a.src_bytes))
                            continue;
                    }
                    hdr[r] = static_cast<int>(slot + static_cast<uint32_t>(g0 - lo)) - re.r0b;
                    for (uintptr_t t = (hi > g0 ? hi : g0); t < g1; t += esz)
                        *reinterpret_cast<Tin*>(smem + slot + static_cast<uint32_t>(t - lo)) =
                            *reinterpret_cast<const Tin*>(t);
                    cp_lo[i] = lo;
                    cp_n[i] = static_cast<uint32_t>(hi - lo);
                    cp_slot[i] = slot;
                    bytes += cp_n[i];
                }
                // one arrival announces the stage's bytes (and publishes the
                // warp's entries and plain loads), then the copies
                bytes = __reduce_add_sync(0xffffffffu, bytes);
                __syncwarp();
                fence_proxy_async();   // the compute warps' reads of this stage come before the copies' writes
                if (lane == 0) mbar_arrive_expect_tx(&m.full[s], bytes);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < kRunsPerLane; ++i)
                    if (cp_n[i])
                        bulk_copy_g2s_once(smem + cp_slot[i], reinterpret_cast<const void*>(cp_lo[i]), cp_n[i], &m.full[s]);
            }
        }
        if (!ok && lane == 0) {
            atomicOr(&g_device_error, kErrBlendWait);
            drain_stages(m.full, S, max(0, j - S), j);   // the copies still in flight
        }
        return;
    }

    // ---- compute warps.  Thread t takes one (row group, chunk entry) pair,
    // class by class: the entries of class c (chunk table order) times its
    // G_c row groups fill the threads from the class's first (a warp
    // boundary where the classes fit), row group major, so that the lanes of
    // a warp share one class and mostly one row cover.  Row group g of an
    // entry computes band rows g', g' + G_c, ... of the unit, g' = g in the
    // CTA's first unit and moved on by a fixed step (band rows mod G_c)
    // each unit, so that the groups with one row more take turns.
    int G = 1, gp = 0, gstep = 0, ent = 0, cls = 0;
    bool active = false;
    {
        const int t = static_cast<int>(threadIdx.x);
        int before = 0;   // entries of the classes before q
#pragma unroll
        for (int q = 0; q < kChunkClasses; ++q) {
            const int nc = a.ncls[q], gq = a.grp[q], t0 = a.tfirst[q];
            if (nc > 0 && t >= t0 && t < t0 + nc * gq) {
                const int l = t - t0;
                gp = l / nc;
                ent = before + (l - gp * nc);
                cls = q;
                G = gq;
                gstep = a.gstep[q];
                active = true;
            }
            before += nc;
        }
    }
    ColTerms<Tin, E, KT> tm;
    int jc = 0;
    if (active) {
        col_terms<Tin, E, KT>(m.chunks[ent], tm);
        jc = m.chunks[ent].col;
    }
    unsigned char* out = static_cast<unsigned char*>(a.dst);
    const uint32_t ring_lo = static_cast<uint32_t>(a.off_data);   // (index checks) the staged data
    const uint32_t ring_hi = ring_lo + static_cast<uint32_t>(S * a.stage_bytes);
    UnitCursor c;
    c.init(first, a.BC, a.nbands);
    RingPos r0;   // the unit's first stage
    for (int k = 0; k < n; ++k, c.next()) {
        const FrameEnt fe = m.frames[c.f];
        RingPos r1 = r0;   // the one after it
        r1.next(S);
        const int s0 = r0.s, s1 = r1.s;
        bool landed = mbar_wait_bounded(&m.full[s0], r0.ph);
        if (landed && fe.n > 1) landed = mbar_wait_bounded(&m.full[s1], r1.ph);
        if (!landed) {
            if (lane == 0) atomicOr(&g_device_error, kErrBlendWait);
            return;   // no release: the producer gives up and drains
        }
        if (active) {
            const BandEnt b = m.bands[c.band];
            const int* hdr_f0 = hdr0 + s0 * a.max_runs;
            const int* hdr_f1 = hdr0 + s1 * a.max_runs;
            // the byte offset of row h of this chunk column in the output plane of (bc, f) is
            // obase + h * W * osz (for a slab, obase itself may be negative in its first plane)
            long long obase;
            if constexpr (SLAB)
                obase = ((((long long)c.bc * F + c.f) * (a.row1 - a.row0) - a.row0) * W + (long long)jc * E) * osz;
            else
                obase = ((((long long)c.bc * F + c.f) * a.H) * W + (long long)jc * E) * osz;
            unsigned char* const oplane = out + obase;
#pragma unroll 1
            for (int h = b.hb0 + gp; h < b.hb1; h += G) {
                const RowEnt re = m.rows[h];
                if (cls == 0 && fe.n == 1 && re.n == 1 && fe.w[0] == 1.0f && re.w[0] == 1.0f) {
                    // one tile, weight 1 on every axis: the output is its elements
                    const int* hrun = hdr_f0 + (re.lo - b.ihlo) * nw;
                    const uint32_t ad = static_cast<uint32_t>(hrun[tm.iw[0]] + h * tm.swb[0] + tm.xob[0]);
                    if (!range_bad(oplane + (long long)h * W * osz, 16, out, a.dst_bytes))
                        copy_chunk<Tin, Tout, E>(smem, ad, oplane + (long long)h * W * osz, ring_lo, ring_hi);
                    continue;
                }
                const int npairs = fe.n * re.n;
                int hx[KT];   // each term's row offset in its tile run: h * row bytes + the chunk's column bytes
#pragma unroll
                for (int q = 0; q < KT; ++q) hx[q] = h * tm.swb[q] + tm.xob[q];
                float2 acc[E / 2];
#pragma unroll
                for (int mm = 0; mm < E / 2; ++mm) acc[mm] = make_float2(0.0f, 0.0f);
#pragma unroll 1
                for (int pi = 0; pi < npairs; ++pi) {
                    // pairs in (frame tile, row tile) order
                    const int fa = pi >= re.n ? 1 : 0, jh = pi - fa * re.n;
                    const int ih = re.lo + jh;
                    const float wfh = __fmul_rn(fa ? fe.w[1] : fe.w[0], jh ? re.w[1] : re.w[0]);
                    const int* hrun = (fa ? hdr_f1 : hdr_f0) + (ih - b.ihlo) * nw;
                    float2 inner[E / 2];
#pragma unroll
                    for (int mm = 0; mm < E / 2; ++mm) inner[mm] = make_float2(0.0f, 0.0f);
                    const uint32_t ad0 = static_cast<uint32_t>(hrun[tm.iw[0]] + hx[0]);
                    if (tm.one) {
                        add_term<Tin, E, KT, false>(smem, ad0, tm, 0, inner, ring_lo, ring_hi);
                    } else {
                        add_term<Tin, E, KT>(smem, ad0, tm, 0, inner, ring_lo, ring_hi);
                        if (KT > 1 && tm.nq > 1)
                            add_term<Tin, E, KT>(smem, static_cast<uint32_t>(hrun[tm.iw[q1]] + hx[q1]),
                                                 tm, q1, inner, ring_lo, ring_hi);
                        if (KT > 2 && tm.nq > 2)
                            add_term<Tin, E, KT>(smem, static_cast<uint32_t>(hrun[tm.iw[q2]] + hx[q2]),
                                                 tm, q2, inner, ring_lo, ring_hi);
                    }
                    const float2 w2 = make_float2(wfh, wfh);
#pragma unroll
                    for (int mm = 0; mm < E / 2; ++mm) acc[mm] = __ffma2_rn(w2, inner[mm], acc[mm]);
                }
                if (!range_bad(oplane + (long long)h * W * osz, 16, out, a.dst_bytes))
                    store_chunk<Tout, E>(oplane + (long long)h * W * osz, acc);
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&m.empty[s0]);
            if (fe.n > 1) mbar_arrive(&m.empty[s1]);
        }
        r0 = r1;
        if (fe.n > 1) r0.next(S);
        gp += gstep;
        if (gp >= G) gp -= G;
    }
}

// =================================================================== host side
constexpr int kStreamUnitsPerCta = 12;          // wanted units per CTA (tail balance)
constexpr int kStreamSmemBudget = 200 * 1024;   // dynamic shared memory of the one CTA per SM

// 1-D trapezoid of tile i on axis d at x, as the device computes it
// (axis_weight): IEEE fp32 division, the two ramps multiplied and rounded.
inline float host_axis_weight(const tdp_plan_t& p, int d, int i, int x) {
    const float o1 = static_cast<float>(p.overlap[d] + 1);
    float up = 1.0f, dn = 1.0f;
    if (i > 0) up = std::fmin(1.0f, static_cast<float>(x - p.start[d][i] + 1) / o1);
    if (i < p.num_tiles[d] - 1) dn = std::fmin(1.0f, static_cast<float>(p.end[d][i] - x) / o1);
    volatile float r = up * dn;   // one fp32 rounding, as on the device
    return r;
}

inline int host_nf(const tdp_plan_t& p, int f) {
    int lo, hi;
    tdp::axis_cover(p, 0, f, lo, hi);
    return hi - lo + 1;
}
inline int host_nhb(const tdp_plan_t& p, int hb0, int hb1) {
    int lo, hi;
    tdp::axis_range_cover(p, 1, hb0, hb1, lo, hi);
    return hi - lo + 1;
}

// Tile rows (summed over the row tiles meeting the band) times the frame
// tiles covering f: the band's runs hold this many rows of every column tile.
inline long long host_run_rows(const tdp_plan_t& p, int f, int hb0, int hb1) {
    long long rows = 0;
    for (int i = 0; i < p.num_tiles[1]; ++i)
        rows += std::max(0, std::min(hb1, p.end[1][i]) - std::max(hb0, p.start[1][i]));
    return rows * host_nf(p, f);
}

struct StreamLaunch {
    StreamArgs a;
    StreamSplit sp;
    StreamTables tb;
    StreamJobs jb;
    int grid = 0, smem = 0;
};

// Jobs a launch takes besides its units, with their cost in the split's
// measure (bytes a unit moves) and the shared scratch they need.
constexpr int kStreamSmemMax = 227 * 1024;     // dynamic shared memory a CTA may opt in to
constexpr long long kExtentCostPerToken = 4;    // a token chunk's share of its CTA, per token
struct StreamJobPlan {
    int kind = kJobNone;
    int B = 0;                // kJobExtent: batch
    int K1 = 0;               // kJobExtent: chunks per (tile, batch) pair
    int scratch = 0;          // shared bytes of the chunks' scratch
};

// Shared bytes one staged run may take: its 16-byte chunks, at most
// round16(len) + 16 bytes, for the longest run of any band.
inline int host_run_slot(const tdp_plan_t& p, int band_rows, int nbands, int row0, int row1, int esz) {
    int slot = 16;
    for (int bi = 0; bi < nbands; ++bi) {
        const int hb0 = row0 + bi * band_rows, hb1 = std::min(row1, hb0 + band_rows);
        int hlo, hhi;
        tdp::axis_range_cover(p, 1, hb0, hb1, hlo, hhi);
        for (int i_h = hlo; i_h <= hhi; ++i_h) {
            const int rows = std::min(p.end[1][i_h], hb1) - std::max(p.start[1][i_h], hb0);
            for (int iw = 0; iw < p.num_tiles[2]; ++iw)
                slot = std::max(slot, round_up(rows * tdp::tile_size(p, 2, iw) * esz, 16) + 16);
        }
    }
    return slot;
}

// Table words (16 bytes each) of a launch; section offsets in `a`.
inline int stream_table_words(const tdp_plan_t& p, bool blend, StreamArgs& a) {
    auto words = [](long long bytes) { return static_cast<int>((bytes + 15) / 16); };
    int o = 0;
    a.t_band = o; o += words((long long)a.nbands * sizeof(BandEnt));
    a.t_frame = o; o += words((long long)p.dims[0] * sizeof(FrameEnt));
    a.t_row = o; o += blend ? words((long long)p.dims[1] * sizeof(RowEnt)) : 0;
    a.t_fcon = o; o += words((long long)p.num_tiles[0] * sizeof(FrameCon));
    a.t_wcon = o; o += blend ? 0 : words((long long)p.num_tiles[2] * sizeof(ColCon));
    a.t_runs = o; o += words((long long)a.nbands * a.runs_per_band * sizeof(RunEnt));
    a.t_chunk = o; o += blend ? words((long long)a.cpr * sizeof(ChunkEnt)) : 0;
    a.t_words = o;
    return o;
}

// Shared layout for one band height: barriers, tables, run-base entries
// (blend), then the ring of stages, each sized to the largest staged piece
// (blend: one frame tile's runs of a band; extract: the band's latent
// rows).  False when the tables or two stages do not
// fit.  a.cpr and a.esz must be set.
inline bool stream_layout(const tdp_plan_t& p, bool blend, int band_rows, StreamArgs& a, int& smem) {
    const int H = p.dims[1], W = p.dims[2];
    const int r0 = a.row0, r1 = a.row1;   // the bands' rows
    if (r0 < 0 || r1 > H || r1 <= r0) return false;
    a.band_rows = band_rows;
    a.nbands = (r1 - r0 + band_rows - 1) / band_rows;
    int nhb_max = 1;
    for (int bi = 0; bi < a.nbands; ++bi)
        nhb_max = std::max(nhb_max, host_nhb(p, r0 + bi * band_rows, std::min(r1, r0 + bi * band_rows + band_rows)));
    a.runs_per_band = nhb_max * p.num_tiles[2];
    a.max_runs = blend ? a.runs_per_band : 0;   // one frame tile's runs per stage
    if (a.max_runs > kStreamMaxStageRuns) return false;
    a.run_slot = blend ? host_run_slot(p, band_rows, a.nbands, r0, r1, a.esz) : 0;
    const long long data = blend ? (long long)a.max_runs * a.run_slot : (long long)band_rows * W * a.esz;
    if (data > INT_MAX / 8) return false;
    if (stream_table_words(p, blend, a) > kStreamTableWords) return false;
    a.stage_bytes = round_up(static_cast<int>(data), 16) + 2 * kStreamPad;
    a.off_full = 0;
    a.off_empty = 8 * kStreamMaxStages;
    a.off_tab = 16 * kStreamMaxStages;
    a.off_hdr = a.off_tab + 16 * a.t_words;
    const long long per_stage = a.stage_bytes + 4LL * a.max_runs;
    const long long S = std::min<long long>(kStreamMaxStages, (kStreamSmemBudget - a.off_hdr - 128) / per_stage);
    if (S < 2) return false;
    a.nstages = static_cast<int>(S);
    a.off_data = round_up(a.off_hdr + a.nstages * 4 * a.max_runs, 128);
    smem = a.off_data + a.nstages * a.stage_bytes;
    return smem <= kStreamSmemBudget;
}

// The plan tables of a launch (host only; the layout's offsets in L.a).
inline void stream_tables(const tdp_plan_t& p, bool blend, StreamLaunch& L) {
    StreamArgs& a = L.a;
    std::memset(&L.tb, 0, sizeof(L.tb));
    unsigned char* base = reinterpret_cast<unsigned char*>(L.tb.w);
    const int F = p.dims[0], H = p.dims[1], nw = p.num_tiles[2];
    const long long SH = p.prefix[1][p.num_tiles[1]], SW = p.prefix[2][nw];
    BandEnt* bands = reinterpret_cast<BandEnt*>(base + 16 * a.t_band);
    for (int bi = 0; bi < a.nbands; ++bi) {
        BandEnt& b = bands[bi];
        b.hb0 = a.row0 + bi * a.band_rows;
        b.hb1 = std::min(a.row1, b.hb0 + a.band_rows);
        int lo, hi;
        tdp::axis_range_cover(p, 1, b.hb0, b.hb1, lo, hi);
        b.ihlo = lo;
        b.NHB = hi - lo + 1;
    }
    FrameEnt* frames = reinterpret_cast<FrameEnt*>(base + 16 * a.t_frame);
    for (int f = 0; f < F; ++f) {
        int lo, hi;
        tdp::axis_cover(p, 0, f, lo, hi);
        frames[f].lo = lo;
        frames[f].n = hi - lo + 1;
        frames[f].w[0] = host_axis_weight(p, 0, lo, f);
        frames[f].w[1] = hi > lo ? host_axis_weight(p, 0, lo + 1, f) : 0.0f;
    }
    if (blend) {
        RowEnt* rows = reinterpret_cast<RowEnt*>(base + 16 * a.t_row);
        for (int h = 0; h < H; ++h) {
            int lo, hi;
            tdp::axis_cover(p, 1, h, lo, hi);
            RowEnt& r = rows[h];
            r.lo = lo;
            r.n = hi - lo + 1;
            r.w[0] = host_axis_weight(p, 1, lo, h);
            r.w[1] = hi > lo ? host_axis_weight(p, 1, lo + 1, h) : 0.0f;
        }
    }
    FrameCon* fcon = reinterpret_cast<FrameCon*>(base + 16 * a.t_fcon);
    for (int i = 0; i < p.num_tiles[0]; ++i) {
        fcon[i].base = (long long)p.prefix[0][i] * SH * SW;
        fcon[i].sf = tdp::tile_size(p, 0, i);
        fcon[i].fs = p.start[0][i];
    }
    if (!blend) {
        ColCon* wcon = reinterpret_cast<ColCon*>(base + 16 * a.t_wcon);
        for (int i = 0; i < nw; ++i) {
            ColCon& c = wcon[i];
            c.sw = tdp::tile_size(p, 2, i);
            c.ws = p.start[2][i];
            const int step = 32 * (8 / a.esz);   // elements of one warp pass (32 8-byte groups)
            c.dq = step / c.sw;
            c.dr = step - c.dq * c.sw;
            c.inv_sw = 1.0f / static_cast<float>(c.sw);
        }
    }
    RunEnt* runs = reinterpret_cast<RunEnt*>(base + 16 * a.t_runs);
    for (int bi = 0; bi < a.nbands; ++bi) {
        const BandEnt& b = bands[bi];
        for (int rr = 0; rr < a.runs_per_band; ++rr) {
            const int jh = rr / nw, iw = rr - jh * nw, ih = b.ihlo + jh;
            RunEnt r{};
            if (jh < b.NHB) {
                const int hs = p.start[1][ih], sh = tdp::tile_size(p, 1, ih), sw = tdp::tile_size(p, 2, iw);
                const int r0 = std::max(hs, b.hb0), r1 = std::min(p.end[1][ih], b.hb1);
                r.A = (long long)p.prefix[1][ih] * SW + (long long)sh * p.prefix[2][iw];
                r.slice = sh * sw;
                r.vrow = (r0 - hs) * sw;
                r.len = (r1 - r0) * sw;
                r.src_rel = ((r0 - b.hb0) * p.dims[2] + p.start[2][iw]) * a.esz;
                r.iw = iw;
                r.r0b = r0 * sw * a.esz;
            }
            runs[bi * a.runs_per_band + rr] = r;
        }
    }
    if (blend) {
        ChunkEnt* chunks = reinterpret_cast<ChunkEnt*>(base + 16 * a.t_chunk);
        const int E = p.dims[2] / a.cpr;   // output elements per chunk
        std::vector<ChunkEnt> ents(a.cpr);
        for (int jc = 0; jc < a.cpr; ++jc) {
            const int c0 = jc * E;
            int lo, hi, l2, h2;
            tdp::axis_cover(p, 2, c0, lo, hi);
            tdp::axis_cover(p, 2, c0 + E - 1, l2, h2);
            ChunkEnt& ce = ents[jc];
            std::memset(&ce, 0, sizeof(ce));
            ce.nq = h2 - lo + 1;
            for (int q = 0; q < 3; ++q) {
                const int i = std::min(lo + q, h2);
                const bool real = lo + q <= h2;
                const int w0 = p.start[2][i], w1 = p.end[2][i];
                ce.iw[q] = i;
                ce.swb[q] = (w1 - w0) * a.esz;
                ce.xob[q] = (c0 - w0) * a.esz;
                for (int mm = 0; mm < E; ++mm) {
                    const int col = c0 + mm;
                    const bool in = real && col >= w0 && col < w1;
                    ce.rw[q][mm] = in ? host_axis_weight(p, 2, i, col) : 0.0f;
                    if (in) ce.in[q] |= 1u << mm;
                }
            }
            ce.col = jc;
            bool ones = ce.nq == 1 && ce.in[0] == (1u << E) - 1;
            for (int mm = 0; mm < E && ones; ++mm) ones = ce.rw[0][mm] == 1.0f;
            ce.cls = ones ? 0 : std::min(ce.nq, kChunkClasses - 1);
        }
        // entries grouped by class (stable), so that a warp's chunks share one
        std::stable_sort(ents.begin(), ents.end(), [](const ChunkEnt& x, const ChunkEnt& y) { return x.cls < y.cls; });
        for (int c = 0; c < kChunkClasses; ++c) a.ncls[c] = 0;
        for (int k = 0; k < a.cpr; ++k) {
            chunks[k] = ents[k];
            ++a.ncls[ents[k].cls];
        }
    }
}

// CTA i takes the units from the first one whose bytes-so-far reach i / G
// of the total.  gcost[g] is the cost of one unit of group g = f * nbands +
// band, and the units of a group are its BC (b, c) planes: u = g * BC + bc.
// With `reserve`, CTA i first runs jobs of cost reserve[i]: its share of
// the units is (units' cost + all jobs' cost) / G less that, at least 0.
inline void stream_split(const std::vector<long long>& gcost, long long BC, int G, StreamSplit& sp,
                         const std::vector<long long>* reserve = nullptr) {
    const int NG = static_cast<int>(gcost.size());
    std::vector<__int128> cum(NG + 1, 0);   // cost of all units of the groups before g
    for (int g = 0; g < NG; ++g) cum[g + 1] = cum[g] + (__int128)gcost[g] * BC;
    const long long n = BC * NG;
    std::vector<__int128> share(G + 1, 0);   // CTAs before i: their shares of the units, in G-ths
    __int128 jobs = 0;
    if (reserve)
        for (int i = 0; i < G; ++i) jobs += (*reserve)[i];
    for (int i = 0; i < G; ++i) {
        __int128 c = 1;
        if (reserve) {
            c = cum[NG] + jobs - (__int128)G * (*reserve)[i];
            if (c < 0) c = 0;
        }
        share[i + 1] = share[i] + c;
    }
    if (share[G] == 0)
        for (int i = 0; i <= G; ++i) share[i] = i;
    for (int i = 0; i <= G; ++i) {
        const __int128 target = cum[NG] * share[i] / share[G];
        const int g = static_cast<int>(std::upper_bound(cum.begin(), cum.end(), target) - cum.begin()) - 1;
        long long u = n;
        if (g < NG) {
            const __int128 rem = target - cum[g];
            const long long bc = static_cast<long long>((rem + gcost[g] - 1) / gcost[g]);
            u = std::min(n, (long long)g * BC + std::min(bc, BC));
        }
        if (i == G) u = n;
        sp.start[i] = static_cast<int>(u);
    }
    for (int i = 1; i <= G; ++i) sp.start[i] = std::max(sp.start[i], sp.start[i - 1]);
}

// Column tiles touching any E-column chunk (the blend's term count).
inline int host_col_terms(const tdp_plan_t& p, int E) {
    int best = 1;
    for (int c0 = 0; c0 + E <= p.dims[2]; c0 += E) {
        int lo, hi, l2, h2;
        tdp::axis_cover(p, 2, c0, lo, hi);
        tdp::axis_cover(p, 2, c0 + E - 1, l2, h2);
        best = std::max(best, h2 - lo + 1);
    }
    return best;
}

// Blend: the compute threads of each chunk class c and its row groups G_c
// (threads per chunk entry).  Each class starts on a warp boundary, so
// that no warp holds two classes (a warp would run both code paths one
// after the other), and gets whole warps: first as few as hold one group
// per entry, then, while warps are left, one more to the class whose
// threads carry the most rows; G_c is as many groups per entry as its
// warps hold.  (Weighting the classes by their terms gained nothing on
// the 4K tiling.)  If the classes do not fit in whole warps they are
// packed one after another with one group each.  A group's step per unit
// is band rows mod G_c.
inline void blend_row_groups(const int (&ncls)[kChunkClasses], int band_rows, int warps, int (&tfirst)[kChunkClasses],
                             int (&grp)[kChunkClasses], int (&gstep)[kChunkClasses]) {
    int wc[kChunkClasses], used = 0;
    for (int c = 0; c < kChunkClasses; ++c) {
        wc[c] = (ncls[c] + 31) / 32;
        used += wc[c];
    }
    auto groups = [&](int c) { return std::min(band_rows, 32 * wc[c] / ncls[c]); };
    if (used <= warps) {
        for (;;) {
            int best = -1;
            double worst = 0.0;
            for (int c = 0; c < kChunkClasses; ++c) {
                if (ncls[c] == 0 || groups(c) >= band_rows) continue;
                const double load = static_cast<double>(band_rows) / groups(c);
                if (load > worst) {
                    worst = load;
                    best = c;
                }
            }
            if (best < 0 || used == warps) break;
            ++wc[best];
            ++used;
        }
        int t = 0;
        for (int c = 0; c < kChunkClasses; ++c) {
            tfirst[c] = t;
            grp[c] = ncls[c] > 0 ? groups(c) : 0;
            t += 32 * wc[c];
        }
    } else {
        int t = 0;
        for (int c = 0; c < kChunkClasses; ++c) {
            tfirst[c] = t;
            grp[c] = ncls[c] > 0 ? 1 : 0;
            t += ncls[c];
        }
    }
    for (int c = 0; c < kChunkClasses; ++c) gstep[c] = grp[c] > 0 ? band_rows % grp[c] : 0;
}

// Picks the band height, the ring, the split and the tables for `sms` SMs
// (host only).  A band is at least `min_rows` tall -- blend: the compute
// threads over the chunks per row, so that a thread has about a row in
// every unit; extract: about 2 KB of latent, so that the warps' spans are
// not mostly partial.  The tallest such band that leaves kStreamUnitsPerCta
// units per CTA wins; failing that the shortest such band (the most
// units); failing that any band that fits.
inline tdp_status stream_geometry(const tdp_plan_t& p, bool blend, int BC, int esz_src, int esz_dst, int sms,
                                  StreamLaunch& L, const StreamJobPlan& jobs = StreamJobPlan{}, int row0 = 0,
                                  int row1 = -1) {
    const int F = p.dims[0], H = p.dims[1], W = p.dims[2];
    if (row1 < 0) row1 = H;
    if (row0 < 0 || row1 > H || row1 <= row0) return TDP_ERR_UNSUPPORTED;
    const int HS = row1 - row0;   // the rows the bands split
    sms = std::max(1, std::min(sms, kStreamMaxGrid));
    const int cpr = blend ? W * esz_dst / 16 : 0;
    const int rg = blend ? std::max(1, 32 * kStreamBlendWarps / std::max(1, cpr)) : 1;
    const int min_rows = std::min(HS, blend ? rg : std::max(1, (2048 + W * esz_src - 1) / (W * esz_src)));
    const long long want = (long long)kStreamUnitsPerCta * sms;
    std::vector<int> heights;   // one per band count, tallest first
    for (int nb = 1; nb <= HS; ++nb) {
        const int br = (HS + nb - 1) / nb;
        if (heights.empty() || heights.back() != br) heights.push_back(br);
    }
    auto units_of = [&](int br) { return (long long)BC * F * ((HS + br - 1) / br); };
    auto fits = [&](int br) {
        StreamArgs a{};
        a.cpr = cpr;
        a.esz = esz_src;
        a.row0 = row0;
        a.row1 = row1;
        int smem = 0;
        return units_of(br) <= INT_MAX && stream_layout(p, blend, br, a, smem);
    };
    int chosen = -1;
    for (int br : heights)   // tallest band with enough units that fits
        if (br >= min_rows && units_of(br) >= want && fits(br)) { chosen = br; break; }
    for (auto it = heights.rbegin(); chosen < 0 && it != heights.rend(); ++it)   // else the most units
        if (*it >= min_rows && fits(*it)) chosen = *it;
    for (int br : heights)
        if (chosen < 0 && fits(br)) chosen = br;
    if (chosen < 0) return TDP_ERR_UNSUPPORTED;
    std::memset(&L.a, 0, sizeof(L.a));
    L.a.cpr = cpr;
    L.a.esz = esz_src;   // extract stages the latent, blend the tiles
    L.a.row0 = row0;
    L.a.row1 = row1;
    if (!stream_layout(p, blend, chosen, L.a, L.smem)) return TDP_ERR_UNSUPPORTED;
    L.a.F = F;
    L.a.H = H;
    L.a.W = W;
    L.a.nw = p.num_tiles[2];
    L.a.BC = BC;
    L.a.n_units = BC * F * L.a.nbands;
    L.grid = static_cast<int>(std::min<long long>((long long)L.a.n_units, (long long)sms));
    stream_tables(p, blend, L);
    if (blend) {
        blend_row_groups(L.a.ncls, L.a.band_rows, kStreamBlendWarps, L.a.tfirst, L.a.grp, L.a.gstep);
        int end = 0;
        for (int c = 0; c < kChunkClasses; ++c)
            if (L.a.ncls[c] > 0) end = std::max(end, L.a.tfirst[c] + L.a.ncls[c] * L.a.grp[c]);
        L.a.cwarps = (end + 31) / 32;
    }
    // cost of one unit per (frame, band) group: latent rows plus packed tile rows
    std::vector<long long> gcost;
    for (int f = 0; f < F; ++f)
        for (int bi = 0; bi < L.a.nbands; ++bi) {
            const int hb0 = row0 + bi * L.a.band_rows, hb1 = std::min(row1, hb0 + L.a.band_rows);
            const long long lat = (long long)(hb1 - hb0) * W * (blend ? esz_dst : esz_src);
            const long long runs =
                host_run_rows(p, f, hb0, hb1) * p.prefix[2][p.num_tiles[2]] * (blend ? esz_src : esz_dst);
            gcost.push_back(lat + runs);
        }
    // jobs: their CTAs, the shared scratch after the ring, and their cost
    std::memset(&L.jb, 0, sizeof(L.jb));
    L.jb.kind = jobs.kind;
    L.jb.B = jobs.B;
    L.jb.K1 = jobs.K1;
    L.jb.p = p;
    std::vector<long long> reserve(L.grid, 0);
    if (jobs.kind == kJobExtent) {
        L.jb.off_job = round_up(L.smem, 16);
        L.smem = L.jb.off_job + round_up(jobs.scratch, 16);
        if (L.smem > kStreamSmemMax) return TDP_ERR_UNSUPPORTED;
        // chunk q on CTA i when ceil(i Q / G) <= q < ceil((i + 1) Q / G)
        const long long Q = (long long)p.total_tiles * jobs.B * jobs.K1, G = L.grid;
        if (Q > INT_MAX) return TDP_ERR_UNSUPPORTED;
        for (int i = 0; i <= L.grid; ++i) L.jb.start[i] = static_cast<int>((i * Q + G - 1) / G);
        for (int i = 0; i < L.grid; ++i)
            for (int q = L.jb.start[i]; q < L.jb.start[i + 1]; ++q) {
                int i_f, i_h, i_w;
                tdp::tile_coords(p, q / jobs.K1 / jobs.B, i_f, i_h, i_w);
                const long long tokens =
                    (long long)tdp::tile_size(p, 0, i_f) * tdp::tile_size(p, 1, i_h) * tdp::tile_size(p, 2, i_w);
                reserve[i] += (tokens + jobs.K1 - 1) / jobs.K1 * kExtentCostPerToken;
            }
    }
    stream_split(gcost, BC, L.grid, L.sp, jobs.kind != kJobNone ? &reserve : nullptr);
    return TDP_OK;
}

// Shapes the streaming kernels take: 16-byte latent rows, at most two
// covering tiles per frame and row; for extract, column tiles at least one
// 16-byte chunk wide (so that an 8-byte group spans at most two tile rows)
// and span indices exact in fp32; for blend, at most two covering column
// tiles, one chunk column per compute thread and at most three column
// tiles per chunk (*kt).  Plans whose tables or stages do not fit are left
// to the general kernels by stream_geometry.
inline bool stream_eligible(const tdp_plan_t& p, bool blend, int esz_src, int esz_dst, int* kt) {
    const int H = p.dims[1], W = p.dims[2];
    const int lat_esz = blend ? esz_dst : esz_src;
    *kt = 0;
    if ((W * lat_esz) % 16 != 0) return false;
    if (p.max_cover[0] > 2 || p.max_cover[1] > 2) return false;
    if (!blend) {
        int min_sw = INT_MAX, max_sw = 0;
        for (int i = 0; i < p.num_tiles[2]; ++i) {
            min_sw = std::min(min_sw, tdp::tile_size(p, 2, i));
            max_sw = std::max(max_sw, tdp::tile_size(p, 2, i));
        }
        if (min_sw < 16 / esz_src) return false;
        if ((long long)H * max_sw >= (1LL << 21)) return false;
        return true;
    }
    if (p.max_cover[2] > 2) return false;
    if (W * esz_dst / 16 > 32 * kStreamBlendWarps) return false;
    *kt = host_col_terms(p, 16 / esz_dst);
    return *kt <= 3;
}

// Geometry of a launch on the current device, and the kernel's opt-in to
// its dynamic shared memory.
template <typename K>
tdp_status stream_prepare(K kernel, const tdp_plan_t& p, bool blend, int BC, int esz_src, int esz_dst, StreamLaunch& L,
                          const StreamJobPlan& jobs = StreamJobPlan{}, int row0 = 0, int row1 = -1) {
    tdp_status st = stream_geometry(p, blend, BC, esz_src, esz_dst, sm_count(), L, jobs, row0, row1);
    if (st != TDP_OK) return st;
    return cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem));
}

// The streaming extract, if it takes the plan (*taken); with `gen`, also
// the partial extents of every (tile, batch) pair's K1 token chunks (B
// batches) into `partials` in the same launch.
template <typename E>
tdp_status launch_extract_stream(const tdp_plan_t& p, int BC, const void* latent, void* tiles, cudaStream_t stream,
                                 bool* taken, const int* gen = nullptr, int B = 0, int K1 = 0,
                                 int* partials = nullptr, const StreamZero& zero = StreamZero{}) {
    constexpr int esz = static_cast<int>(sizeof(E));
    *taken = false;
    int kt = 0;
    if (!stream_eligible(p, false, esz, esz, &kt)) return TDP_OK;
    static thread_local StreamLaunch L;   // 13 KB: kept off the caller's stack
    StreamJobPlan jobs;
    if (gen) {
        // scratch: the reduction's ints, then one chunk's tokens (3 int2 each)
        int nmax = 1;
        for (int t = 0; t < p.total_tiles; ++t) {
            int i_f, i_h, i_w;
            tdp::tile_coords(p, t, i_f, i_h, i_w);
            nmax = std::max(nmax, tdp::tile_size(p, 0, i_f) * tdp::tile_size(p, 1, i_h) * tdp::tile_size(p, 2, i_w));
        }
        jobs.kind = kJobExtent;
        jobs.B = B;
        jobs.K1 = K1;
        jobs.scratch = 4 * kChunkShInts + 24 * ((nmax + K1 - 1) / K1);
    }
    tdp_status st = gen ? stream_prepare(extract_stream_kernel<E, StreamJobs>, p, false, BC, esz, esz, L, jobs)
                        : stream_prepare(extract_stream_kernel<E, NoJobs>, p, false, BC, esz, esz, L, jobs);
    if (st == TDP_ERR_UNSUPPORTED) return TDP_OK;
    if (st != TDP_OK) return st;
    L.a.src = latent;
    L.a.dst = tiles;
    L.a.src_bytes = (long long)BC * p.dims[0] * p.dims[1] * p.dims[2] * esz;
    L.a.dst_bytes = (long long)BC * tdp::total_volume(p) * esz;
    L.jb.gen = gen;
    L.jb.partials = partials;
    L.jb.zero_a = zero.a;
    L.jb.nzero_a = zero.a ? zero.na : 0;
    L.jb.zero_b = zero.b;
    L.jb.nzero_b = zero.b ? zero.nb : 0;
    *taken = true;
    if (!gen)
        return launch(extract_stream_kernel<E, NoJobs>, L.grid, kStreamExtractThreads, L.smem, stream, 1, L.a, L.sp, L.tb,
                      NoJobs{});
    return launch(extract_stream_kernel<E, StreamJobs>, L.grid, kStreamExtractThreads, L.smem, stream, 1, L.a, L.sp, L.tb,
                  L.jb);
}

// The streaming blend of output rows [row0, row1) (out: [BC, F, row1 - row0,
// W]), if it takes the plan (*taken).
template <typename Tin, typename Tout>
tdp_status launch_blend_stream(const tdp_plan_t& p, int BC, const void* tiles, long long tiles_numel, void* out,
                               cudaStream_t stream, bool* taken, int row0, int row1) {
    constexpr int isz = static_cast<int>(sizeof(Tin)), osz = static_cast<int>(sizeof(Tout));
    *taken = false;
    int kt = 0;
    if (!stream_eligible(p, true, isz, osz, &kt)) return TDP_OK;
    auto go = [&](auto kernel) -> tdp_status {
        static thread_local StreamLaunch L;   // 13 KB: kept off the caller's stack
        tdp_status st = stream_prepare(kernel, p, true, BC, isz, osz, L, StreamJobPlan{}, row0, row1);
        if (st == TDP_ERR_UNSUPPORTED) return TDP_OK;
        if (st != TDP_OK) return st;
        L.a.src = tiles;
        L.a.dst = out;
        L.a.src_bytes = tiles_numel * isz;
        L.a.dst_bytes = (long long)BC * p.dims[0] * (row1 - row0) * p.dims[2] * osz;
        *taken = true;
        return launch(kernel, L.grid, kStreamBlendThreads, L.smem, stream, 1, L.a, L.sp, L.tb);
    };
    if (row0 != 0 || row1 != p.dims[1]) {
        if (kt == 1) return go(blend_stream_kernel<Tin, Tout, 1, true>);
        if (kt == 2) return go(blend_stream_kernel<Tin, Tout, 2, true>);
        return go(blend_stream_kernel<Tin, Tout, 3, true>);
    }
    if (kt == 1) return go(blend_stream_kernel<Tin, Tout, 1, false>);
    if (kt == 2) return go(blend_stream_kernel<Tin, Tout, 2, false>);
    return go(blend_stream_kernel<Tin, Tout, 3, false>);
}
