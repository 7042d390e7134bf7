/*
 * tdp.h -- C ABI of the tiled-latent extract / trapezoid overlap-add path
 * (libtdp.so, CUDA for sm_103a).
 *
 * The method is LTX-2's Tiled Data Parallelism ("Tiled Data Parallelism
 * (TDP)", LTX-2 multi-GPU docs, section "What it is"): the patchified
 * (frames, height, width) latent is split into overlapping tiles by count
 * per axis, each tile is processed on its own, and the per-tile results are
 * recombined with separable trapezoidal masks that sum to 1.  The interval
 * split and the window are the ones that the mold issue #673 ("A bug found
 * while porting") measures for upstream's split_by_count / blend.
 *
 * Conventions shared by every call
 *   - Latent X is [B, C, F, H, W], contiguous, W fastest.
 *   - Tiles are numbered frames-major: t = (i_f * n_h + i_h) * n_w + i_w.
 *   - Packed tiles: tile after tile, each [B, C, f_t, h_t, w_t] contiguous;
 *     tile t starts at element tdp_tile_offset(plan, t, B, C).  Tile shapes
 *     may differ (the last tile of an axis absorbs the remainder).
 *   - Generated token n of the latent grid is n = (f * H + h) * W + w;
 *     positions are int32 [start, end) pairs, layout [B, 3, N, 2] with
 *     axis 0 = time (frames), 1 = height, 2 = width.
 *   - Device pointers are owned by the caller.  The library allocates no
 *     device memory, never synchronises the stream and keeps no state
 *     between calls apart from one diagnostic word (tdp_device_error).
 *     Every device pointer must be 16-byte aligned (else
 *     TDP_ERR_ALIGNMENT); buffers must not overlap unless stated.
 *   - Every call validates its arguments on the host (including that the
 *     plan is exactly what tdp_plan returns for its own dims, counts,
 *     overlaps and flags) and returns before any launch when they are
 *     wrong.  Kernels never trap.  A failed launch or runtime call returns
 *     TDP_ERR_CUDA; tdp_last_cuda_error gives its cudaError_t code.
 *   - B or C (or M) equal to 0 is an empty batch: the call validates the
 *     plan and returns TDP_OK without launching.
 */
#ifndef TDP_H_
#define TDP_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TDP_MAX_PER_AXIS 64          /* tiles per axis */
#define TDP_PLAN_UPSTREAM_COMPAT 1u  /* accept overlap*(n+1) > dim (windows then sum above 1) */

/* DimensionTilingConfig(num_tiles, overlap): a tile COUNT and an overlap in
 * latent grid units ("Tiled Data Parallelism (TDP)", section API, Tiling
 * config).  The page's default is {1, 0}. */
typedef struct {
    int32_t num_tiles;
    int32_t overlap;
} tdp_dim_cfg;

/* TileCountConfig(frames, height, width): counts, not sizes (same section). */
typedef struct {
    tdp_dim_cfg frames;
    tdp_dim_cfg height;
    tdp_dim_cfg width;
} tdp_tile_count_cfg;

typedef enum {
    TDP_OK = 0,
    TDP_ERR_INVALID_ARG = 1,     /* bad size, count, pointer or dtype */
    TDP_ERR_GUARD = 2,           /* overlap*(n+1) > dim without TDP_PLAN_UPSTREAM_COMPAT */
    TDP_ERR_TOO_MANY_TILES = 3,  /* num_tiles > TDP_MAX_PER_AXIS */
    TDP_ERR_ALIGNMENT = 4,       /* a device pointer is not 16-byte aligned */
    TDP_ERR_CUDA = 5,            /* a CUDA launch or runtime call failed */
    TDP_ERR_UNSUPPORTED = 6      /* a shape the kernels cannot stage (see each call) */
} tdp_status;

typedef enum { TDP_F32 = 0, TDP_BF16 = 1 } tdp_dtype;

/* Host-side plan.  Plain data: filled by tdp_plan, read by every other call
 * (it is copied by value into the kernels, so it may be reused or freed as
 * soon as a call returns). */
typedef struct {
    int32_t dims[3];                               /* F, H, W */
    int32_t num_tiles[3];                          /* n per axis */
    int32_t overlap[3];                            /* overlap per axis */
    int32_t stride[3];                             /* floor((dim - overlap) / n) */
    int32_t start[3][TDP_MAX_PER_AXIS];            /* tile i covers [start, end) */
    int32_t end[3][TDP_MAX_PER_AXIS];
    int32_t prefix[3][TDP_MAX_PER_AXIS + 1];       /* sum of sizes of tiles < i */
    int32_t max_cover[3];                          /* most tiles covering one index */
    int32_t total_tiles;                           /* T = n_f * n_h * n_w */
    uint32_t flags;
} tdp_plan_t;

/*
 * tdp_plan -- step 1, interval planning per axis.
 *
 * Source: the mold issue #673 ("A bug found while porting") describes
 * split_by_count and the guard overlap <= dim/(n+1) that keeps the windows
 * a partition of unity; "Tiled Data Parallelism (TDP)" (API) gives the
 * count/overlap configuration.  The split formula is not printed on the
 * pages; the one used here -- stride s = floor((dim - overlap)/n), tile i =
 * [i*s, i*s + s + overlap), last tile stretched to end at dim -- is the
 * simple split that reproduces the mold issue's measured window sums.
 *
 * dims_fhw: host array {F, H, W}, each >= 1.
 * cfg:      host pointer; per axis num_tiles in [1, TDP_MAX_PER_AXIS],
 *           overlap >= 0, overlap == 0 when num_tiles == 1, stride >= 1.
 * flags:    0 (guard enforced) or TDP_PLAN_UPSTREAM_COMPAT.
 * out:      host pointer, written only on TDP_OK.
 * Errors: TDP_ERR_INVALID_ARG, TDP_ERR_TOO_MANY_TILES, TDP_ERR_GUARD.
 * Host only; touches no GPU.
 */
tdp_status tdp_plan(const int32_t dims_fhw[3], const tdp_tile_count_cfg* cfg, uint32_t flags,
                    tdp_plan_t* out);

/* Element offset of tile t in the packed tile buffer, and the total number
 * of packed elements (sum over tiles of B*C*f_t*h_t*w_t).  Host only;
 * return -1 on a bad argument. */
int64_t tdp_tile_offset(const tdp_plan_t* plan, int32_t t, int32_t B, int32_t C);
int64_t tdp_tiles_numel(const tdp_plan_t* plan, int32_t B, int32_t C);

/* Start and size of tile t per axis (host arrays of 3). */
tdp_status tdp_tile_box(const tdp_plan_t* plan, int32_t t, int32_t start[3], int32_t size[3]);

/*
 * tdp_plan_stats -- layout statistics of a plan (host only).
 *
 * Source: DistVAE docs "Choosing a tile window" (decoded area, seams,
 * per-tile activations, heaviest-rank imbalance) and "Tiled Data
 * Parallelism (TDP)" (tiles assigned to ranks round-robin, t mod ranks).
 *   decoded_area   = prod_d (sum of tile sizes on d) / dim_d
 *   seams          = sum_a (n_a - 1) * prod_{b != a} n_b
 *   tile_fraction  = largest tile volume / latent volume
 *   imbalance      = heaviest rank's volume / (total / ranks) - 1
 *   max_window_sum = max over the grid of sum_t w_t (exact rational
 *                    arithmetic, rounded once to double)
 * Any output pointer may be NULL.  ranks >= 1.
 */
tdp_status tdp_plan_stats(const tdp_plan_t* plan, int32_t ranks, double* decoded_area,
                          int32_t* seams, double* tile_fraction, double* imbalance,
                          double* max_window_sum);

/*
 * tdp_balanced_tile_split -- height x width tile counts for a rank count.
 *
 * Source: "Tiled Data Parallelism (TDP)", Usage: balanced_tile_split(world
 * size) gives the balanced 2-D spatial grid of the upscale stage.  The rule
 * is not printed; the one used here is the factor pair of `ranks` closest to
 * a square, with the smaller count on height (the latents are wider than
 * tall).  ranks >= 1; h_tiles, w_tiles: host pointers.  Host only.
 */
tdp_status tdp_balanced_tile_split(int32_t ranks, int32_t* h_tiles, int32_t* w_tiles);

#define TDP_SEARCH_NO_LIMITS 2u   /* tdp_search_layouts: skip the DistVAE window limits */

typedef enum {
    TDP_ROLE_DOMINATED = 0,   /* another candidate is no worse on every criterion and better on one */
    TDP_ROLE_FRONTIER = 1,    /* on the frontier, not selected */
    TDP_ROLE_COARSE = 2,      /* the frontier's largest window */
    TDP_ROLE_FINE = 3,        /* the smallest window among the rest */
    TDP_ROLE_BALANCED = 4     /* the least worst normalised score among the rest */
} tdp_layout_role;

typedef struct {
    int32_t num_tiles[3];           /* n_f, n_h, n_w */
    int32_t overlap[3];
    int64_t window_volume;          /* largest tile, f*h*w latent units (window area) */
    int64_t decoded_volume;         /* sum of tile volumes (decoded area) */
    int64_t heaviest_rank_volume;   /* round-robin, tile t on rank t mod ranks */
    int32_t seams;                  /* sum_a (n_a - 1) * prod_{b != a} n_b */
    int32_t role;                   /* tdp_layout_role */
} tdp_layout_candidate;

/*
 * tdp_search_layouts -- layout search over tile counts (host only).
 *
 * Source: DistVAE docs "Choosing a tile window", Benchmark plan selection,
 * applied to TDP tile counts:
 *   - candidates: every (n_h, n_w) with max(2, ranks) <= n_f*n_h*n_w <=
 *     4*ranks whose plan tdp_plan accepts (the frame axis keeps `frames`;
 *     a tiled spatial axis takes overlap_h / overlap_w, an untiled one 0);
 *   - unless TDP_SEARCH_NO_LIMITS: no candidate at all when the latent's
 *     narrow spatial axis has fewer than max(16, ranks) units, and none
 *     whose overlap on a tiled spatial axis is below a quarter of the
 *     window (stride + overlap) -- the page's conservative limits;
 *   - roles: dominated / frontier on window area, decoded area, rank
 *     imbalance (heaviest / total) and tile columns; among the frontier,
 *     coarse = largest window, fine = smallest window among the rest,
 *     balanced = least max(window / top window, decoded / top decoded,
 *     imbalance / top imbalance) among the rest (tops over the frontier);
 *     ties go to less decoded area, less imbalance, fewer columns, fewer rows.
 * flags: TDP_PLAN_UPSTREAM_COMPAT (plans without the guard) and/or
 *        TDP_SEARCH_NO_LIMITS.
 * out:   host array of `capacity` entries (NULL allowed when capacity is 0).
 * count: receives the number of candidates; when it exceeds `capacity`
 *        only the first `capacity` are written.  Order: n_h, then n_w.
 */
tdp_status tdp_search_layouts(const int32_t dims_fhw[3], int32_t ranks, const tdp_dim_cfg* frames,
                              int32_t overlap_h, int32_t overlap_w, uint32_t flags,
                              tdp_layout_candidate* out, int32_t capacity, int32_t* count);

/*
 * tdp_extract -- step 2, tile extract (K1).
 *
 * Source: "Tiled Data Parallelism (TDP)", What it is (each tile is the
 * latent's sub-box); mold issue #673, Scope (per-tile latent slice).
 *   tiles[t][b, c, k, y, x] = latent[b, c, f0_t + k, h0_t + y, w0_t + x]
 * latent: device, [B, C, F, H, W] of `dtype`.
 * tiles:  device, packed (tdp_tiles_numel elements of `dtype`).
 * Bit-exact copy.  Asynchronous on `stream`.
 */
tdp_status tdp_extract(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype,
                       const void* latent, void* tiles, cudaStream_t stream);

/*
 * tdp_positions -- step 3, per-tile position grids (K4).
 *
 * Source: "Tiled Data Parallelism (TDP)", Position normalization: the
 * tile's positions are shifted by the minimum start of its generated
 * tokens, per (batch, axis), so they start at zero; interval widths are
 * unchanged.
 * gen_pos:   device int32 [B, 3, N, 2], N = F*H*W.
 * normalize: nonzero -> subtract the offset from start and end.
 * tile_pos:  device int32, packed [T][B, 3, N_t, 2], N_t = f_t*h_t*w_t,
 *            tokens in tile row-major order; tile t starts at element
 *            6 * B * (sum of N_t' for t' < t).
 * offsets:   device int32 [T, B, 3], min start of tile t's generated tokens
 *            (written whether or not `normalize` is set).
 * Bit-exact.  Asynchronous on `stream`.
 */
tdp_status tdp_positions(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos,
                         int32_t normalize, int32_t* tile_pos, int32_t* offsets,
                         cudaStream_t stream);

/*
 * tdp_cond_select -- step 4, conditioning-token selection (K5).
 *
 * Source: "Tiled Data Parallelism (TDP)", Shared negative (reference)
 * positions: a tile keeps a conditioning token whose [start, end) overlaps
 * the tile in all three axes, or whose time start is negative; a token
 * kept by k tiles has blend weight 1/k.  Kept tokens go after the tile's
 * generated tokens, so they are shifted by the same offset (Position
 * normalization).
 *   extent[t,b,d] = [TS, TE): min start / max end of tile t's generated
 *                   tokens on axis d (before any shift).
 *   keep[t,b,m]   = cond_t_start < 0  or  for all d: cs_d < TE_d and ce_d > TS_d
 *   count[b,m]    = sum_t keep[t,b,m];  weight = count ? 1.0f/count : 0 (IEEE fp32)
 * gen_pos:       device int32 [B, 3, N, 2].
 * cond_pos:      device int32 [B, 3, M, 2] (M >= 0).
 * normalize:     nonzero -> tile_cond_pos is shifted by TS.
 * tile_extent:   device int32 [T, B, 3, 2] (required).
 * keep:          device uint8 [T, B, M] (required, 0/1).
 * count:         device int32 [B, M] (required).
 * weight:        device float [B, M] (required).
 * kept_idx:      device int32 [T, B, M] or NULL: indices of kept tokens in
 *                their original order, -1 after the last one.
 * num_kept:      device int32 [T, B] or NULL.
 * tile_cond_pos: device int32 [T, B, 3, M, 2] or NULL: positions of the
 *                kept tokens in kept order, zero after the last one.
 * Bit-exact.  Asynchronous on `stream`.
 */
tdp_status tdp_cond_select(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos,
                           int32_t M, const int32_t* cond_pos, int32_t normalize,
                           int32_t* tile_extent, uint8_t* keep, int32_t* count, float* weight,
                           int32_t* kept_idx, int32_t* num_kept, int32_t* tile_cond_pos,
                           cudaStream_t stream);

/*
 * tdp_tokens -- steps 3 and 4 in one launch: tdp_positions and
 * tdp_cond_select over the same tiles, sharing one pass over the generated
 * positions (the tile extent is reduced once and serves both).
 *
 * Source: "Tiled Data Parallelism (TDP)", Position normalization and
 * Shared negative (reference) positions, as for the two calls above.
 * Arguments mean what they mean there.  tile_pos NULL skips the positions
 * (offsets may then be NULL too); M == 0 skips the conditioning tokens
 * (cond_pos, keep, count and weight may then be NULL); tile_extent, when
 * not NULL, receives [TS, TE) per tile, batch and axis (required when
 * M > 0).  slot_of, when not NULL, receives int32 [T, B, M]: the token's
 * position in tile t's kept list, or -1 (the index tdp_cond_combine
 * gathers by).  Every result equals what the separate calls write.
 * Bit-exact.  Asynchronous on `stream`.
 */
tdp_status tdp_tokens(const tdp_plan_t* plan, int32_t B, const int32_t* gen_pos,
                      int32_t normalize, int32_t* tile_pos, int32_t* offsets, int32_t M,
                      const int32_t* cond_pos, int32_t* tile_extent, uint8_t* keep,
                      int32_t* count, float* weight, int32_t* kept_idx, int32_t* num_kept,
                      int32_t* tile_cond_pos, int32_t* slot_of, cudaStream_t stream);

/*
 * tdp_extract_and_tokens -- steps 2, 3 and 4 and the window maximum of
 * step 6 in two launches: everything tdp_extract, tdp_tokens and
 * tdp_window_sum (maximum only) write.
 *
 * Source: "Tiled Data Parallelism (TDP)", What it is (each tile is the
 * latent's sub-box; masks that sum to 1), Position normalization and
 * Shared negative (reference) positions, as for those three calls.
 * Arguments mean what they mean there: B, C, dtype, latent and tiles as
 * for tdp_extract; gen_pos through slot_of as for tdp_tokens (M > 0
 * requires cond_pos, tile_extent, keep, count and weight; tile_pos NULL
 * skips the positions); max_abs_dev as for tdp_window_sum (NULL: no
 * maximum).  C == 0 leaves the tiles alone and still does the rest.
 * workspace: device memory of at least tdp_extract_and_tokens_workspace
 *            (plan, B) bytes, owned by the caller and free for the call's
 *            duration (calls that run at the same time need their own);
 *            its contents on entry do not matter.
 * When the streaming extract takes the plan (and the workspace is large
 * enough), the extract launch also reduces the partial extents of every
 * (tile, batch) pair's token chunks, spread over its CTAs, into the
 * workspace, and a second, short launch combines them and writes the
 * positions, keep flags, kept lists, counts, weights and the maximum.
 * Otherwise the separate kernels run in turn (workspace unused; it may be
 * NULL).  Every result equals what the separate calls write, bit for bit.
 * Asynchronous on `stream`.  Errors: as the separate calls
 * (TDP_ERR_ALIGNMENT for any pointer not 16-byte aligned).
 */
int64_t tdp_extract_and_tokens_workspace(const tdp_plan_t* plan, int32_t B);   /* bytes; -1 if invalid */
tdp_status tdp_extract_and_tokens(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype,
                                  const void* latent, void* tiles, const int32_t* gen_pos,
                                  int32_t normalize, int32_t* tile_pos, int32_t* offsets, int32_t M,
                                  const int32_t* cond_pos, int32_t* tile_extent, uint8_t* keep,
                                  int32_t* count, float* weight, int32_t* kept_idx, int32_t* num_kept,
                                  int32_t* tile_cond_pos, int32_t* slot_of, float* max_abs_dev,
                                  void* workspace, int64_t workspace_bytes, cudaStream_t stream);

/*
 * tdp_extract_and_tokens_no_alloc -- tdp_extract_and_tokens with the
 * library's own scratch instead of a caller's workspace: a file-scope
 * device array of 64 KiB (one instance per device, found with
 * cudaGetSymbolAddress on the current device); nothing is allocated.
 * Arguments, results and errors as tdp_extract_and_tokens; a plan and
 * batch whose tdp_extract_and_tokens_workspace exceeds 64 KiB give
 * TDP_ERR_UNSUPPORTED.  Calls that overlap on one device (other streams,
 * other host threads) share the scratch and race: run them one after
 * another.  Nothing is claimed for CUDA graph capture.
 */
tdp_status tdp_extract_and_tokens_no_alloc(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype,
                                           const void* latent, void* tiles, const int32_t* gen_pos,
                                           int32_t normalize, int32_t* tile_pos, int32_t* offsets, int32_t M,
                                           const int32_t* cond_pos, int32_t* tile_extent, uint8_t* keep,
                                           int32_t* count, float* weight, int32_t* kept_idx, int32_t* num_kept,
                                           int32_t* tile_cond_pos, int32_t* slot_of, float* max_abs_dev,
                                           cudaStream_t stream);

/*
 * tdp_cond_combine -- the blend of the conditioning tokens' per-tile
 * outputs (the step after tdp_cond_select).
 *
 * Source: "Tiled Data Parallelism (TDP)", Shared negative (reference)
 * positions: a token kept by several tiles is not counted twice; its blend
 * weight is 1 / (number of tiles that kept it).
 *   out[b,m,:] = sum over tiles t with slot_of[t,b,m] >= 0, in increasing t,
 *                of weight[b,m] * tile_cond_out[t,b,slot_of[t,b,m],:]
 * accumulated in fp32 (fmaf) and stored once in `out_dtype` (round to
 * nearest even for bf16); a token kept by no tile gets zeros.
 * tile_cond_out: device [T, B, M, D] in `in_dtype`: tile t's outputs for
 *                its kept tokens in kept order (rows past the tile's kept
 *                count are not read).
 * slot_of:       device int32 [T, B, M] from tdp_tokens: the token's
 *                position in tile t's kept list, or -1.
 * weight:        device float [B, M] from tdp_cond_select / tdp_tokens.
 * out:           device [B, M, D] in `out_dtype`.
 * B, M or D == 0: nothing to do.  Asynchronous on `stream`.
 */
tdp_status tdp_cond_combine(const tdp_plan_t* plan, int32_t B, int32_t M, int32_t D,
                            tdp_dtype in_dtype, const void* tile_cond_out, const int32_t* slot_of,
                            const float* weight, tdp_dtype out_dtype, void* out,
                            cudaStream_t stream);

/*
 * tdp_blend -- step 5, fused separable trapezoid window + overlap-add (K2).
 *
 * Source: "Tiled Data Parallelism (TDP)", What it is (overlapping regions
 * blended with trapezoidal masks that sum to 1); mold issue #673 (a
 * separable trapezoidal window; blend has no normalisation pass).
 *   out[b,c,f,h,w] = sum over tiles t covering (f,h,w) of
 *                    r_f(f) * r_h(h) * r_w(w) * tiles[t][b,c,f-f0,h-h0,w-w0]
 * with, on each axis for tile i of n over [a, e) and overlap o,
 *   r(x) = up * down,  up = (i > 0) ? min(1, (x-a+1)/(o+1)) : 1,
 *                      down = (i < n-1) ? min(1, (e-x)/(o+1)) : 1.
 * The weights are formed in fp32 registers, the sum is accumulated in fp32
 * and written once in `out_dtype` (round to nearest even for bf16); there
 * is no zero-fill pass and no atomics.  Every element of `out` is written.
 * tiles: device, packed, `in_dtype`.  out: device [B, C, F, H, W].
 * Asynchronous on `stream`.
 */
tdp_status tdp_blend(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype in_dtype,
                     const void* tiles, tdp_dtype out_dtype, void* out, cudaStream_t stream);

/*
 * tdp_shard_plan -- the sharded blend's layout for one of `ranks` ranks
 * (host only).
 *
 * Source: "Tiled Data Parallelism (TDP)", What it is (tiles go to ranks
 * round robin, tile t to rank t mod R, and one all_reduce sums the ranks'
 * blended full-size buffers).  Reading: the same sum is formed without a
 * reduction over full-size buffers -- the latent's rows are split into R
 * disjoint output slabs, rank r blends its slab alone (tdp_blend_slab) from
 * every tile that meets it, and the tiles it needs but does not own (its
 * halo) come from their owners; the slabs concatenated along H are the
 * blend, bit for bit.
 *   row0, row1: rank `rank`'s slab, rows [row0, row1) of H, with
 *               row_r = floor(r * H / ranks) (empty when ranks > H)
 *   owned[t]:   1 iff t mod ranks == rank
 *   needed[t]:  1 iff tile t's rows [start_h, end_h) meet [row0, row1)
 * owned and needed: host uint8 arrays of plan->total_tiles entries, or
 * NULL.  ranks >= 1 and 0 <= rank < ranks, else TDP_ERR_INVALID_ARG.
 */
tdp_status tdp_shard_plan(const tdp_plan_t* plan, int32_t ranks, int32_t rank, int32_t* row0,
                          int32_t* row1, uint8_t* owned, uint8_t* needed);

/*
 * tdp_blend_slab -- step 5 restricted to output rows [row0, row1).
 *
 * Source: as tdp_blend; the slab split is the reading of tdp_shard_plan.
 *   out[b, c, f, h - row0, w] = the tdp_blend sum at (b, c, f, h, w),
 *                               row0 <= h < row1
 * with the same fp32 weights, grouping and order as tdp_blend, so that the
 * slab equals those rows of tdp_blend bit for bit.
 * tiles: device, packed as for tdp_blend (tdp_tiles_numel elements of
 *        `in_dtype`); only the tiles whose rows meet [row0, row1) are read,
 *        the others may hold anything.
 * out:   device [B, C, F, row1 - row0, W] of `out_dtype`, every element
 *        written.
 * 0 <= row0 <= row1 <= H, else TDP_ERR_INVALID_ARG; row0 == row1 is a
 * no-op.  Asynchronous on `stream`.
 */
tdp_status tdp_blend_slab(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype in_dtype,
                          const void* tiles, int32_t row0, int32_t row1, tdp_dtype out_dtype, void* out,
                          cudaStream_t stream);

/*
 * tdp_extract_tokens -- step 2 into token-major tiles.
 *
 * Source: "Tiled Data Parallelism (TDP)", What it is and When to use it
 * (every tile goes through the transformer on its own, as the sequence of
 * its N_t = f_t*h_t*w_t tokens) and Position normalization (a tile's
 * generated tokens are its sub-grid of the latent's token grid, in the
 * grid's row-major order).
 *   tokens[t][b, n, c] = latent[b, c, f0_t + k, h0_t + y, w0_t + x],
 *   n = (k * h_t + y) * w_t + x
 * latent: device, [B, C, F, H, W] of `dtype`.
 * tokens: device, packed tile after tile like tdp_extract (tile t starts at
 *         element tdp_tile_offset(plan, t, B, C)), each tile [B, N_t, C]
 *         with C fastest; tdp_tiles_numel elements of `dtype`.
 * C * sizeof(dtype) must be a multiple of 16 bytes and at most 16 KiB
 * (else TDP_ERR_UNSUPPORTED).  Bit-exact copy.  Asynchronous on `stream`.
 */
tdp_status tdp_extract_tokens(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype dtype,
                              const void* latent, void* tokens, cudaStream_t stream);

/*
 * tdp_blend_tokens -- step 5 from token-major tiles.
 *
 * Source: as tdp_blend, with the tiles in the layout of tdp_extract_tokens.
 *   out[b,c,f,h,w] = sum over tiles t covering (f,h,w) of
 *                    r_f(f) * r_h(h) * r_w(w) * tokens[t][b, n_t(f,h,w), c]
 * with n_t(f,h,w) = ((f-f0)*h_t + (h-h0))*w_t + (w-w0) and the same fp32
 * windows as tdp_blend.  fp32 accumulation, one store per element in
 * `out_dtype` (round to nearest even for bf16); every element of `out` is
 * written.  tokens: device, packed token-major, `in_dtype`.
 * out: device [B, C, F, H, W].  C * sizeof(in_dtype) must be a multiple of
 * 16 bytes and at most 16 KiB -- 8 KiB when C * sizeof(in_dtype) / 16 is not
 * a multiple of 4, 4 KiB when it is odd (else TDP_ERR_UNSUPPORTED).
 * Asynchronous on `stream`.
 */
tdp_status tdp_blend_tokens(const tdp_plan_t* plan, int32_t B, int32_t C, tdp_dtype in_dtype,
                            const void* tokens, tdp_dtype out_dtype, void* out, cudaStream_t stream);

/*
 * tdp_window_sum -- window-sum check (K3).
 *
 * Source: "Tiled Data Parallelism (TDP)", What it is (masks sum to 1
 * globally) and mold issue #673 (the sum exceeds 1 when the guard is
 * violated: up to 1.074 for (21,3,8), 1.161 for (21,4,8)).
 *   S(f,h,w) = sum_t r_f * r_h * r_w (fp32, the weights tdp_blend applies)
 * max_abs_dev: device float, receives max |S - 1| (required).
 * sum_out:     device float [F, H, W] or NULL, receives S.
 * Asynchronous on `stream`.
 */
tdp_status tdp_window_sum(const tdp_plan_t* plan, float* max_abs_dev, float* sum_out,
                          cudaStream_t stream);

/*
 * tdp_launch_geometry -- how tdp_extract (blend == 0) or tdp_blend
 * (blend == 1; tdp_blend_slab for output rows [row0, row1) other than
 * [0, H)) lays out a call with these sizes on a GPU with `sm_count`
 * SMs.  Extract takes row0 = 0, row1 = H; 0 <= row0 < row1 <= H, else
 * TDP_ERR_INVALID_ARG.  Host only; touches no GPU.  It describes a launch, not a step of
 * the method: it lets the kernels' index arithmetic be checked on the CPU
 * and a benchmark report the launch configuration.
 *   streaming       1 when the 16-byte streaming kernel takes the call (each
 *                   output 16-byte chunk is written by one thread with one
 *                   store); 0 when the general kernel does, and then every
 *                   other field is 0
 *   band_rows       latent rows per unit of work; nbands units per
 *                   (b, c, frame) plane
 *   units           B*C*F*nbands; unit u = (f * nbands + band) * B*C + b*C + c
 *   grid            CTAs; CTA i takes units [cta_start[i], cta_start[i+1])
 *   stages, stage_bytes  the shared-memory ring of staged units (each stage
 *                   holds its data between two 32-byte guards); one producer
 *                   warp fills it with bulk copies ahead of the compute warps
 *   max_runs        blend: staged tile-row runs per stage at most (a stage
 *                   holds one covering frame tile's runs of a band; a unit
 *                   of a frame two tiles cover takes two stages)
 *   shared_bytes    dynamic shared memory per CTA
 *   off_hdr, off_data  shared offsets of the run-base entries and the ring
 *   chunks_per_row  blend: 16-byte output chunks per latent row
 *   column_terms    blend: most column tiles touching one output chunk
 *   rows_per_thread blend: most band rows one thread computes in one unit
 *   class_first[c], row_groups[c], row_step[c]  blend, per chunk class c
 *                   (0: one term of weight 1 over the whole chunk; 1: one
 *                   term otherwise; 2, 3: two, three terms): its first
 *                   compute thread (a warp boundary where the classes fit
 *                   in whole warps) and G = row_groups[c] threads per chunk
 *                   entry (0 without entries).  Thread class_first[c] + l,
 *                   l < n_c * G (n_c the class's entries, in chunk-table
 *                   order), takes entry l mod n_c and group g = l / n_c,
 *                   which computes band rows g', g' + G, ... of the CTA's
 *                   k-th unit, g' = (g + k * row_step[c]) mod G
 *   threads         compute threads of a CTA (the launch adds one producer
 *                   warp)
 *   run_slot        blend: shared bytes of each staged run's slot (run r of
 *                   a unit sits at r * run_slot in its stage)
 * For extract, in_dtype is the latent's type and out_dtype must equal it.
 * cta_start: host int32 array of cta_start_len entries, or NULL; filled
 *            with grid + 1 entries when cta_start_len > grid.
 * tables:    host buffer of tables_bytes bytes, or NULL; receives the plan
 *            tables passed with the launch (table_bytes of them, at most
 *            tables_bytes) and, in table_offsets (7 int32, or NULL), the
 *            16-byte word offsets of its sections: bands, frames, rows,
 *            frame-tile constants, column-tile constants, runs, chunks.
 */
typedef struct {
    int32_t streaming;
    int32_t band_rows, nbands, units, grid, stages, stage_bytes, max_runs, shared_bytes;
    int32_t off_hdr, off_data, chunks_per_row, column_terms, rows_per_thread, threads, run_slot;
    int32_t table_bytes;
    int32_t class_first[4], row_groups[4], row_step[4];
} tdp_launch_geometry_t;

tdp_status tdp_launch_geometry(const tdp_plan_t* plan, int32_t B, int32_t C, int32_t blend, tdp_dtype in_dtype,
                               tdp_dtype out_dtype, int32_t sm_count, tdp_launch_geometry_t* geometry,
                               int32_t* cta_start, int32_t cta_start_len, void* tables, int32_t tables_bytes,
                               int32_t* table_offsets, int32_t row0, int32_t row1);

/* Diagnostic word of the current device, an OR of
 *   1  an extract kernel gave up waiting for its staged copies (bounded
 *      wait, about 1 s) and skipped its work: its output is incomplete;
 *   2  a blend kernel gave up likewise;
 *   4  after such a give-up, copies the kernel had issued did not land
 *      within a second bounded wait before it exited: they may still write
 *      into shared memory that a later kernel owns, so no later output on
 *      the device can be trusted;
 *   8  (debug builds only, TDP_DEBUG_CHECKS) an index check of a global or
 *      shared access failed; the access was skipped.
 * Reads it synchronously into *code and, when `clear` is nonzero, resets
 * it.  Returns TDP_ERR_CUDA if the read fails. */
tdp_status tdp_device_error(uint32_t* code, int32_t clear);

const char* tdp_status_str(tdp_status status);

/* cudaError_t code of the most recent TDP_ERR_CUDA on the calling thread
 * (0 if none). */
int32_t tdp_last_cuda_error(void);

/* sizeof(tdp_plan_t), so that bindings can check their mirror of it. */
size_t tdp_plan_struct_size(void);

#ifdef __cplusplus
}
#endif

#endif /* TDP_H_ */
