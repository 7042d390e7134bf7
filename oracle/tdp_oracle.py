"""CPU oracle for the tiled-latent overlap-add path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the test-suite, the package smoke check and the benchmark's CPU-baseline
leg may.  It shares no code with the CUDA library (no kernels, headers,
tables or helpers); the two meet only through the seeded inputs that the
tests feed to both.

It is deliberately plain: NumPy slicing and float64 (the pages fix no
precision for the windows), one tile at a time, no blocking or fusion.

Method sources (the pages are documentation, not code):

* "Tiled Data Parallelism (TDP)", LTX-2 multi-GPU docs,
  §What it is -- tiles of the patchified (frames, height, width) latent,
  overlapping regions blended with trapezoidal masks that sum to 1;
  §Position normalization -- per-(batch, dim) minimum start of the
  generated tokens is subtracted from every position, widths unchanged;
  §Shared negative (reference) positions -- conditioning-token keep rule
  and the 1/(number of tiles that kept it) weight;
  §API -- TileCountConfig / DimensionTilingConfig(num_tiles, overlap):
  counts per axis, overlap in latent grid units.
* mold issue #673 (porting LTX-2's tiled stage 2), §A bug found while
  porting -- split_by_count, the separable trapezoidal window, the measured
  window-sum table for splits (21,2,8), (21,3,8), (21,4,8) and the guard
  overlap <= dim/(n+1).
* DistVAE docs "Choosing a tile window" -- decoded area, seams and per-rank
  imbalance of a tile layout (used for plan statistics only).

Readings taken where the pages are silent (each is listed in the design
notes of the repository):

* split_by_count: stride s = floor((dim - overlap) / n); tile i covers
  [i*s, i*s + s + overlap); the last tile is stretched to end at dim.  This
  is the one simple family that reproduces the mold window-sum table
  exactly (1, 29/27, 94/81).
* 1-D window of tile i over [a, e): product of a rising ramp
  min(1, (x - a + 1)/(overlap + 1)) and a falling ramp
  min(1, (e - x)/(overlap + 1)); the rising ramp is 1 for the first tile,
  the falling ramp is 1 for the last tile (no ramp at the latent border).
* Tiles are enumerated frames-major: t = (i_f * n_h + i_h) * n_w + i_w.
* Generated token n of a (F, H, W) grid is n = (f*H + h)*W + w.
* A conditioning interval [cs, ce) overlaps the tile's interval [TS, TE)
  when cs < TE and ce > TS; [TS, TE) is the minimum start / maximum end of
  the tile's generated tokens; "negative time coordinate" is start_t < 0.
* 1/count is an IEEE float32 division; a token kept by no tile gets
  count 0 and weight 0.
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction
from typing import List, Sequence, Tuple

import numpy as np

AXES = ("frames", "height", "width")


class GuardError(ValueError):
    """overlap * (n + 1) > dim: the windows no longer sum to 1."""


# ---------------------------------------------------------------------------
# Step 1: interval planning (mold issue #673 §A bug found while porting;
# TDP docs §API for the count/overlap configuration).
# ---------------------------------------------------------------------------
def split_by_count(dim: int, num_tiles: int, overlap: int, compat: bool = False
                   ) -> List[Tuple[int, int]]:
    """Half-open intervals of `num_tiles` tiles over an axis of length `dim`.

    Consecutive tiles share `overlap` units.  With `compat=False` the
    partition-of-unity guard overlap <= dim/(n+1) (written overlap*(n+1) <=
    dim) is enforced, as the mold port does; `compat=True` reproduces the
    unguarded upstream behaviour whose excess the mold table measures.
    """
    if dim < 1 or num_tiles < 1 or overlap < 0:
        raise ValueError("dim and num_tiles must be >= 1, overlap >= 0")
    if num_tiles == 1:
        if overlap != 0:
            raise ValueError("a single tile cannot overlap anything")
        return [(0, dim)]
    stride = (dim - overlap) // num_tiles
    if stride < 1:
        raise ValueError("stride (dim - overlap) // num_tiles must be >= 1")
    if not compat and overlap * (num_tiles + 1) > dim:
        raise GuardError(f"overlap {overlap} > dim/(n+1) for dim {dim}, n {num_tiles}")
    intervals = []
    for i in range(num_tiles):
        start = i * stride
        end = start + stride + overlap
        intervals.append((start, end))
    intervals[-1] = (intervals[-1][0], dim)
    return intervals


def ramp_exact(intervals: Sequence[Tuple[int, int]], overlap: int, i: int, x: int) -> Fraction:
    """1-D trapezoid weight of tile i at coordinate x, as an exact fraction."""
    a, e = intervals[i]
    if not (a <= x < e):
        return Fraction(0)
    n = len(intervals)
    up = Fraction(1) if i == 0 else min(Fraction(1), Fraction(x - a + 1, overlap + 1))
    down = Fraction(1) if i == n - 1 else min(Fraction(1), Fraction(e - x, overlap + 1))
    return up * down


def ramp_1d(intervals: Sequence[Tuple[int, int]], overlap: int, i: int) -> np.ndarray:
    """float64 weights of tile i over its own local coordinates 0..size-1."""
    a, e = intervals[i]
    n = len(intervals)
    x = np.arange(a, e, dtype=np.float64)
    up = np.ones_like(x) if i == 0 else np.minimum(1.0, (x - a + 1.0) / (overlap + 1.0))
    down = np.ones_like(x) if i == n - 1 else np.minimum(1.0, (e - x) / (overlap + 1.0))
    return up * down


@dataclass
class Plan:
    dims: Tuple[int, int, int]                 # (F, H, W)
    counts: Tuple[int, int, int]               # tiles per axis
    overlaps: Tuple[int, int, int]
    intervals: Tuple[List[Tuple[int, int]], ...]  # per axis

    @property
    def num_tiles(self) -> int:
        return self.counts[0] * self.counts[1] * self.counts[2]

    def tile_index(self, t: int) -> Tuple[int, int, int]:
        """(i_f, i_h, i_w) of tile t, frames-major order."""
        i_w = t % self.counts[2]
        i_h = (t // self.counts[2]) % self.counts[1]
        i_f = t // (self.counts[2] * self.counts[1])
        return i_f, i_h, i_w

    def box(self, t: int) -> Tuple[Tuple[int, int], Tuple[int, int], Tuple[int, int]]:
        i = self.tile_index(t)
        return tuple(self.intervals[d][i[d]] for d in range(3))

    def shape(self, t: int) -> Tuple[int, int, int]:
        return tuple(e - s for (s, e) in self.box(t))


def make_plan(dims: Sequence[int], cfg: Sequence[Tuple[int, int]], compat: bool = False) -> Plan:
    """dims = (F, H, W); cfg = ((n_f, o_f), (n_h, o_h), (n_w, o_w)) as in
    TileCountConfig(frames, height, width) of DimensionTilingConfig(num_tiles, overlap)."""
    ivs = tuple(split_by_count(int(dims[d]), int(cfg[d][0]), int(cfg[d][1]), compat)
                for d in range(3))
    return Plan(tuple(int(v) for v in dims), tuple(int(c[0]) for c in cfg),
                tuple(int(c[1]) for c in cfg), ivs)


def tile_window(plan: Plan, t: int) -> np.ndarray:
    """Separable trapezoid of tile t: outer product of the three 1-D ramps."""
    i = plan.tile_index(t)
    rf, rh, rw = (ramp_1d(plan.intervals[d], plan.overlaps[d], i[d]) for d in range(3))
    return rf[:, None, None] * rh[None, :, None] * rw[None, None, :]


# ---------------------------------------------------------------------------
# Step 2: tile extract.  tiles[t][b, c, k, y, x] = X[b, c, f0+k, h0+y, w0+x].
# ---------------------------------------------------------------------------
def extract(plan: Plan, latent: np.ndarray) -> List[np.ndarray]:
    assert latent.ndim == 5 and tuple(latent.shape[2:]) == plan.dims
    out = []
    for t in range(plan.num_tiles):
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        out.append(np.array(latent[:, :, f0:f1, h0:h1, w0:w1], copy=True))
    return out


def pack(tiles: Sequence[np.ndarray]) -> np.ndarray:
    """Packed layout: tile after tile, each [B, C, f_t, h_t, w_t] row-major."""
    return np.concatenate([np.ascontiguousarray(x).reshape(-1) for x in tiles])


def unpack(plan: Plan, B: int, C: int, flat: np.ndarray) -> List[np.ndarray]:
    out, pos = [], 0
    for t in range(plan.num_tiles):
        shp = (B, C) + plan.shape(t)
        n = int(np.prod(shp))
        out.append(flat[pos:pos + n].reshape(shp))
        pos += n
    assert pos == flat.size
    return out


# ---------------------------------------------------------------------------
# Token-major tiles (TDP docs §What it is and §When to use it: every tile is
# run through the transformer on its own, as a sequence of its N_t tokens;
# §Position normalization: a tile's generated tokens are its sub-grid of the
# latent's token grid, in the same row-major order).  Reading: token n of a
# tile with shape (f_t, h_t, w_t) is local (k, y, x) with
# n = (k*h_t + y)*w_t + x, and each token carries all C channels.
# ---------------------------------------------------------------------------
def extract_tokens(plan: Plan, latent: np.ndarray) -> List[np.ndarray]:
    """tokens[t][b, n, c] = X[b, c, f0+k, h0+y, w0+x], n = (k*h_t + y)*w_t + x."""
    assert latent.ndim == 5 and tuple(latent.shape[2:]) == plan.dims
    B, C = latent.shape[:2]
    out = []
    for t in range(plan.num_tiles):
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        sub = latent[:, :, f0:f1, h0:h1, w0:w1]            # [B, C, f_t, h_t, w_t]
        out.append(np.ascontiguousarray(sub.reshape(B, C, -1).transpose(0, 2, 1)))
    return out


def unpack_tokens(plan: Plan, B: int, C: int, flat: np.ndarray) -> List[np.ndarray]:
    """Packed token-major buffer -> per-tile [B, N_t, C] views (tile after
    tile, the same tile offsets as the channel-first packing)."""
    out, pos = [], 0
    for t in range(plan.num_tiles):
        n_t = int(np.prod(plan.shape(t)))
        out.append(flat[pos:pos + B * n_t * C].reshape(B, n_t, C))
        pos += B * n_t * C
    assert pos == flat.size
    return out


def blend_tokens(plan: Plan, tiles_tok: Sequence[np.ndarray]) -> np.ndarray:
    """Overlap-add of token-major tile outputs: the token (k, y, x) of tile t
    lands on latent point (f0+k, h0+y, w0+x) of every channel, weighted by
    the tile's separable trapezoid there.  float64 accumulation."""
    B, _, C = tiles_tok[0].shape
    acc = np.zeros((B, C) + plan.dims, dtype=np.float64)
    for t in range(plan.num_tiles):
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        ft, ht, wt = plan.shape(t)
        grid = tiles_tok[t].astype(np.float64).transpose(0, 2, 1).reshape(B, C, ft, ht, wt)
        acc[:, :, f0:f1, h0:h1, w0:w1] += tile_window(plan, t)[None, None] * grid
    return acc


# ---------------------------------------------------------------------------
# Step 5: window and overlap-add (TDP docs §What it is; mold §A bug found
# while porting: blend has no normalisation pass).
# ---------------------------------------------------------------------------
def blend(plan: Plan, tiles: Sequence[np.ndarray]) -> np.ndarray:
    """Y = sum_t w_t * tile_t, accumulated in float64."""
    B, C = tiles[0].shape[:2]
    acc = np.zeros((B, C) + plan.dims, dtype=np.float64)
    for t in range(plan.num_tiles):
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        acc[:, :, f0:f1, h0:h1, w0:w1] += tile_window(plan, t)[None, None] * tiles[t].astype(np.float64)
    return acc


def blend_abs(plan: Plan, tiles: Sequence[np.ndarray]) -> np.ndarray:
    """sum_t w_t * |tile_t|: the magnitude that rounding error scales with."""
    return blend(plan, [np.abs(x.astype(np.float64)) for x in tiles])


def window_sum(plan: Plan) -> np.ndarray:
    """S(f, h, w) = sum over tiles covering the point of the 3-D window."""
    S = np.zeros(plan.dims, dtype=np.float64)
    for t in range(plan.num_tiles):
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        S[f0:f1, h0:h1, w0:w1] += tile_window(plan, t)
    return S


def window_sum_1d_exact(intervals: Sequence[Tuple[int, int]], overlap: int, dim: int) -> List[Fraction]:
    return [sum((ramp_exact(intervals, overlap, i, x) for i in range(len(intervals))), Fraction(0))
            for x in range(dim)]


def max_abs_deviation(plan: Plan) -> float:
    return float(np.max(np.abs(window_sum(plan) - 1.0)))


# ---------------------------------------------------------------------------
# Step 3: per-tile positions (TDP docs §Position normalization).
# gen_pos[b, d, n, :] = [start, end) of generated token n on axis d.
# ---------------------------------------------------------------------------
def tile_token_indices(plan: Plan, t: int) -> np.ndarray:
    """Global token indices n = (f*H + h)*W + w of tile t, in tile row-major order."""
    F, H, W = plan.dims
    (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
    f = np.arange(f0, f1)[:, None, None]
    h = np.arange(h0, h1)[None, :, None]
    w = np.arange(w0, w1)[None, None, :]
    return ((f * H + h) * W + w).reshape(-1)


def positions(plan: Plan, gen_pos: np.ndarray, normalize: bool = True
              ) -> Tuple[List[np.ndarray], np.ndarray]:
    """Per tile: its generated tokens' positions [B, 3, N_t, 2], shifted by the
    per-(batch, dim) minimum start when `normalize`; and that minimum, [T, B, 3]."""
    B = gen_pos.shape[0]
    out, offsets = [], np.zeros((plan.num_tiles, B, 3), dtype=np.int64)
    for t in range(plan.num_tiles):
        p = gen_pos[:, :, tile_token_indices(plan, t), :].astype(np.int64)
        off = p[..., 0].min(axis=2)                 # min start per (batch, dim)
        offsets[t] = off
        if normalize:
            p = p - off[:, :, None, None]          # start and end move together
        out.append(p)
    return out, offsets


# ---------------------------------------------------------------------------
# Step 4: conditioning-token selection (TDP docs §Shared negative (reference)
# positions).  cond_pos[b, d, m, :] = [start, end) of conditioning token m.
# ---------------------------------------------------------------------------
@dataclass
class CondSelection:
    extent: np.ndarray          # [T, B, 3, 2]  [min start, max end) of the tile's generated tokens
    keep: np.ndarray            # [T, B, M] bool
    count: np.ndarray           # [B, M] int
    weight: np.ndarray          # [B, M] float32
    kept: List[List[np.ndarray]]        # kept[t][b] = kept token indices, original order
    tile_cond_pos: List[List[np.ndarray]]  # [t][b] -> [3, K, 2] positions of kept tokens


def cond_select(plan: Plan, gen_pos: np.ndarray, cond_pos: np.ndarray, normalize: bool = True
                ) -> CondSelection:
    B, _, M, _ = cond_pos.shape
    T = plan.num_tiles
    cond = cond_pos.astype(np.int64)
    extent = np.zeros((T, B, 3, 2), dtype=np.int64)
    keep = np.zeros((T, B, M), dtype=bool)
    for t in range(T):
        p = gen_pos[:, :, tile_token_indices(plan, t), :].astype(np.int64)
        TS = p[..., 0].min(axis=2)                  # [B, 3]
        TE = p[..., 1].max(axis=2)
        extent[t, :, :, 0], extent[t, :, :, 1] = TS, TE
        overlaps = (cond[..., 0] < TE[:, :, None]) & (cond[..., 1] > TS[:, :, None])  # [B, 3, M]
        negative_time = cond[:, 0, :, 0] < 0
        keep[t] = overlaps.all(axis=1) | negative_time
    count = keep.sum(axis=0).astype(np.int64)
    weight = np.zeros((B, M), dtype=np.float32)
    nz = count > 0
    weight[nz] = np.float32(1.0) / count[nz].astype(np.float32)
    kept, tcp = [], []
    for t in range(T):
        kept.append([np.nonzero(keep[t, b])[0] for b in range(B)])
        rows = []
        for b in range(B):
            sel = cond[b][:, kept[t][b], :]         # [3, K, 2]
            if normalize:
                sel = sel - extent[t, b, :, 0][:, None, None]
            rows.append(sel)
        tcp.append(rows)
    return CondSelection(extent, keep, count, weight, kept, tcp)


def cond_combine(sel: CondSelection, tile_cond_out: np.ndarray) -> np.ndarray:
    """Blend of the conditioning tokens' per-tile outputs (TDP §Shared negative
    (reference) positions: a token kept by k tiles has blend weight 1/k).
    tile_cond_out[t, b, j] is tile t's output for its j-th kept token of batch
    b (kept order = original order); rows past a tile's kept count are ignored.
    Returns out[b, m] = sum over the tiles t keeping m of (1/k) *
    tile_cond_out[t, b, j_t(m)], in float64 (a token kept by no tile gives 0)."""
    T, B, M = sel.keep.shape
    D = tile_cond_out.shape[-1]
    out = np.zeros((B, M, D), dtype=np.float64)
    for b in range(B):
        for m in range(M):
            k = int(sel.count[b, m])
            if k == 0:
                continue
            for t in range(T):
                hits = np.nonzero(sel.kept[t][b] == m)[0]
                if len(hits):
                    out[b, m] += tile_cond_out[t, b, int(hits[0])].astype(np.float64) / k
    return out


def cond_slots(sel: CondSelection) -> np.ndarray:
    """slot[t, b, m] = the position of token m in tile t's kept list, or -1."""
    T, B, M = sel.keep.shape
    slot = np.full((T, B, M), -1, dtype=np.int64)
    for t in range(T):
        for b in range(B):
            for j, m in enumerate(sel.kept[t][b]):
                slot[t, b, m] = j
    return slot


# ---------------------------------------------------------------------------
# Plan statistics (DistVAE "Choosing a tile window": decoded area, seams,
# per-tile activations, heaviest-rank imbalance; TDP §What it is: tiles go to
# ranks round-robin).
# ---------------------------------------------------------------------------
@dataclass
class LayoutStats:
    decoded_area: float         # sum of tile volumes / latent volume
    seams: int                  # internal tile boundaries: sum_a (n_a - 1) * prod_{b != a} n_b
    tile_fraction: float        # largest tile volume / latent volume
    imbalance: float            # heaviest rank / even split - 1, round-robin assignment


def layout_stats(axis_intervals: Sequence[Sequence[Tuple[int, int]]], dims: Sequence[int],
                 ranks: int) -> LayoutStats:
    """Statistics of any separable layout given by its per-axis intervals."""
    sizes = [[e - s for (s, e) in iv] for iv in axis_intervals]
    counts = [len(s) for s in sizes]
    latent = float(np.prod(dims))
    area = 1.0
    for d in range(len(dims)):
        area *= sum(sizes[d]) / dims[d]
    seams = 0
    for a in range(len(counts)):
        others = 1
        for b in range(len(counts)):
            if b != a:
                others *= counts[b]
        seams += (counts[a] - 1) * others
    vols = []
    for idx in np.ndindex(*counts):              # frames-major / row-major tile order
        v = 1
        for d in range(len(dims)):
            v *= sizes[d][idx[d]]
        vols.append(v)
    per_rank = [0] * ranks
    for t, v in enumerate(vols):
        per_rank[t % ranks] += v
    even = sum(vols) / ranks
    return LayoutStats(area, seams, max(vols) / latent, max(per_rank) / even - 1.0)


# ---------------------------------------------------------------------------
# Layout planning (TDP docs §Usage: a balanced height x width tile grid from
# the rank count; DistVAE "Choosing a tile window" §Benchmark plan selection:
# search grids of max(2, ranks)..4*ranks tiles, drop unsupported windows,
# keep the candidates no other one beats on window area, decoded area, rank
# imbalance and tile columns, and name coarse / fine / balanced among them).
# ---------------------------------------------------------------------------
def balanced_tile_split(ranks: int) -> Tuple[int, int]:
    """(height tiles, width tiles): the factor pair of `ranks` closest to a
    square, the smaller count on height (the latents here are wider than
    tall).  Reading: the pages print only the call, not the rule."""
    if ranks < 1:
        raise ValueError("ranks must be >= 1")
    h = max(d for d in range(1, int(np.sqrt(ranks)) + 2) if d * d <= ranks and ranks % d == 0)
    return h, ranks // h


@dataclass
class LayoutCandidate:
    counts: Tuple[int, int, int]       # (n_f, n_h, n_w)
    overlaps: Tuple[int, int, int]
    window_volume: int                 # largest tile's f*h*w (window area, frames fixed)
    decoded_volume: int                # sum of tile volumes (decoded area)
    heaviest_rank_volume: int          # round-robin assignment, tile t -> rank t mod ranks
    seams: int
    role: str = ""                     # "coarse", "fine", "balanced", "frontier" or "dominated"

    @property
    def columns(self) -> int:
        return self.counts[2]

    def imbalance(self, ranks: int) -> float:
        return self.heaviest_rank_volume * ranks / self.decoded_volume - 1.0


def _beats(a: LayoutCandidate, b: LayoutCandidate) -> bool:
    """a is no worse than b on every criterion and better on one (imbalance
    compared as heaviest/total, cross-multiplied to stay exact)."""
    ia = a.heaviest_rank_volume * b.decoded_volume
    ib = b.heaviest_rank_volume * a.decoded_volume
    le = (a.window_volume <= b.window_volume and a.decoded_volume <= b.decoded_volume
          and ia <= ib and a.columns <= b.columns)
    lt = (a.window_volume < b.window_volume or a.decoded_volume < b.decoded_volume
          or ia < ib or a.columns < b.columns)
    return le and lt


def search_layouts(dims: Sequence[int], ranks: int, frames: Tuple[int, int], overlap_h: int, overlap_w: int,
                   compat: bool = False, limits: bool = True) -> List[LayoutCandidate]:
    """Every supported (n_h, n_w) grid with max(2, ranks) <= n_f*n_h*n_w <=
    4*ranks, each marked with its role.  With `limits`, the DistVAE limits
    apply: the latent's narrow spatial axis holds >= 16 units and >= one
    unit per rank (else no candidate), and every tiled spatial axis has
    overlap >= a quarter of its window (stride + overlap).  An untiled axis
    takes overlap 0."""
    F, H, W = (int(v) for v in dims)
    if ranks < 1:
        raise ValueError("ranks must be >= 1")
    if limits and min(H, W) < max(16, ranks):
        return []
    lo, hi = max(2, ranks), 4 * ranks
    out = []
    for n_h in range(1, H + 1):
        for n_w in range(1, W + 1):
            if not lo <= frames[0] * n_h * n_w <= hi:
                continue
            oh = overlap_h if n_h > 1 else 0
            ow = overlap_w if n_w > 1 else 0
            try:
                plan = make_plan((F, H, W), (frames, (n_h, oh), (n_w, ow)), compat=compat)
            except ValueError:
                continue                                   # unsupported window (incl. the guard)
            if limits:
                windows = [(plan.intervals[d][0][1] - plan.intervals[d][0][0], plan.overlaps[d])
                           for d in (1, 2) if plan.counts[d] > 1]
                if any(4 * o < win for win, o in windows):
                    continue
            vols = [int(np.prod(plan.shape(t))) for t in range(plan.num_tiles)]
            per_rank = [0] * ranks
            for t, v in enumerate(vols):
                per_rank[t % ranks] += v
            stats = layout_stats(plan.intervals, plan.dims, ranks)
            out.append(LayoutCandidate(plan.counts, plan.overlaps, max(vols), sum(vols), max(per_rank),
                                       stats.seams))
    frontier = [c for c in out if not any(_beats(d, c) for d in out)]
    for c in out:
        c.role = "frontier" if c in frontier else "dominated"
    if not frontier:
        return out

    def ties(c):   # fixed order among equals: less decoded, less imbalance, fewer columns, fewer rows
        return (c.decoded_volume, Fraction(c.heaviest_rank_volume, c.decoded_volume), c.columns, c.counts[1])

    coarse = min(frontier, key=lambda c: (-c.window_volume,) + ties(c))
    coarse.role = "coarse"
    rest = [c for c in frontier if c is not coarse]
    if rest:
        fine = min(rest, key=lambda c: (c.window_volume,) + ties(c))
        fine.role = "fine"
        rest = [c for c in rest if c is not fine]
    if rest:
        # worst of the three scores, each divided by its largest value on the frontier
        top_w = max(c.window_volume for c in frontier)
        top_d = max(c.decoded_volume for c in frontier)
        top_i = max(c.imbalance(ranks) for c in frontier)

        def score(c):
            s_i = c.imbalance(ranks) / top_i if top_i > 0 else 0.0
            return max(c.window_volume / top_w, c.decoded_volume / top_d, s_i)

        balanced = min(rest, key=lambda c: (score(c),) + ties(c))
        balanced.role = "balanced"
    return out
