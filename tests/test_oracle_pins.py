"""Pins for the CPU oracle: page-printed values, closed forms, invariants and
brute force on tiny inputs -- never the oracle checked against itself."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import tdp_oracle as O
from overlap_add_blending_gb300 import inputs
from overlap_add_blending_gb300.workloads import WORKLOADS

from conftest import read_golden_rows

# ---------------------------------------------------------------- planning
def test_mold_window_sum_table():
    """mold issue #673 table: max window sum of (21,2,8), (21,3,8), (21,4,8)."""
    rows = read_golden_rows("mold_window_sum_table.txt")
    assert len(rows) == 3
    for dim, n, ov, printed in rows:
        dim, n, ov, printed = int(dim), int(n), int(ov), float(printed)
        iv = O.split_by_count(dim, n, ov, compat=True)
        s_exact = max(O.window_sum_1d_exact(iv, ov, dim))
        # 3-D float path through a (1, 1, dim) plan gives the same number
        plan = O.make_plan((1, 1, dim), ((1, 0), (1, 0), (n, ov)), compat=True)
        s_float = float(O.window_sum(plan).max())
        assert abs(s_float - float(s_exact)) < 1e-12
        # the table rounds to 3 decimals; 1.16049 is printed as 1.161 (a
        # double rounding through 1.1605), so allow 6e-4
        assert abs(float(s_exact) - printed) <= 6e-4, (dim, n, ov, s_exact)
    # the two-tile split sums to exactly one everywhere
    iv2 = O.split_by_count(21, 2, 8, compat=True)
    assert all(v == 1 for v in O.window_sum_1d_exact(iv2, 8, 21))
    # the prose gives the largest excess to two decimals
    iv4 = O.split_by_count(21, 4, 8, compat=True)
    assert round(float(max(O.window_sum_1d_exact(iv4, 8, 21))), 2) == 1.16


def test_guard_rejects_in_strict_mode():
    for dim, n, ov in ((21, 2, 8), (21, 3, 8), (21, 4, 8)):
        with pytest.raises(O.GuardError):
            O.split_by_count(dim, n, ov)
    O.split_by_count(24, 2, 8)             # 8 * 3 <= 24: allowed


@pytest.mark.parametrize("n", [3, 4, 5])
def test_guard_iff_partition_of_unity(n):
    """tile_size >= 2*overlap  <=>  overlap <= dim/(n+1) (mold issue #673):
    for n >= 3 the guard holds exactly when the windows sum to one."""
    for dim in range(n, 25):
        for ov in range(0, dim):
            if (dim - ov) // n < 1:
                continue
            iv = O.split_by_count(dim, n, ov, compat=True)
            unity = all(v == 1 for v in O.window_sum_1d_exact(iv, ov, dim))
            assert unity == (ov * (n + 1) <= dim), (dim, n, ov)


def test_two_tiles_never_triple_overlap():
    for dim in range(2, 40):
        for ov in range(0, dim):
            if (dim - ov) // 2 < 1:
                continue
            iv = O.split_by_count(dim, 2, ov, compat=True)
            cover = [sum(1 for (s, e) in iv if s <= x < e) for x in range(dim)]
            assert max(cover) <= 2
            assert all(v == 1 for v in O.window_sum_1d_exact(iv, ov, dim))


def test_interval_structure():
    """Every tile but the last has length stride+overlap, neighbours share
    exactly `overlap` units and the tiles cover [0, dim)."""
    for dim, n, ov in itertools.product(range(1, 30), range(1, 6), range(0, 10)):
        try:
            iv = O.split_by_count(dim, n, ov)
        except ValueError:
            continue
        s = (dim - ov) // n
        assert iv[0][0] == 0 and iv[-1][1] == dim
        for i in range(n - 1):
            assert iv[i][1] - iv[i][0] == s + ov
            assert iv[i][1] - iv[i + 1][0] == ov
        covered = set()
        for a, e in iv:
            covered.update(range(a, e))
        assert covered == set(range(dim))


def test_invalid_configurations():
    with pytest.raises(ValueError):
        O.split_by_count(16, 1, 2)          # one tile, nonzero overlap
    with pytest.raises(ValueError):
        O.split_by_count(3, 4, 0)           # more tiles than units
    with pytest.raises(ValueError):
        O.split_by_count(0, 1, 0)


def test_workload_intervals():
    """Hand-derived intervals of the named workloads (floor stride, last tile to the end)."""
    p = O.make_plan((16, 68, 120), ((2, 2), (4, 8), (4, 12)))
    assert p.intervals[0] == [(0, 9), (7, 16)]
    assert p.intervals[1] == [(0, 23), (15, 38), (30, 53), (45, 68)]
    assert p.intervals[2] == [(0, 39), (27, 66), (54, 93), (81, 120)]
    p = O.make_plan((16, 32, 48), ((1, 0), (2, 8), (2, 12)))
    assert p.intervals == ([(0, 16)], [(0, 20), (12, 32)], [(0, 30), (18, 48)])
    p = O.make_plan((1, 128, 128), ((1, 0), (3, 8), (5, 8)))
    assert p.intervals[1] == [(0, 48), (40, 88), (80, 128)]
    assert p.intervals[2] == [(0, 32), (24, 56), (48, 80), (72, 104), (96, 128)]
    assert p.num_tiles == 15


# ---------------------------------------------------------------- extract
def test_extract_bruteforce():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((2, 3, 5, 9, 11))
    plan = O.make_plan((5, 9, 11), ((2, 1), (3, 2), (2, 3)))
    tiles = O.extract(plan, X)
    for t in range(plan.num_tiles):
        i_w = t % 2
        i_h = (t // 2) % 3
        i_f = t // 6
        f0 = plan.intervals[0][i_f][0]
        h0 = plan.intervals[1][i_h][0]
        w0 = plan.intervals[2][i_w][0]
        shp = tiles[t].shape
        for b, c, k, y, x in itertools.product(*(range(s) for s in shp)):
            assert tiles[t][b, c, k, y, x] == X[b, c, f0 + k, h0 + y, w0 + x]


def test_extract_coordinate_latent_and_packing():
    F, H, W = 4, 16, 16
    f, h, w = np.meshgrid(np.arange(F), np.arange(H), np.arange(W), indexing="ij")
    X = ((f * 1000 + h * 100 + w)[None, None]).astype(np.float64).repeat(2, axis=1)
    plan = O.make_plan((F, H, W), ((1, 0), (2, 4), (2, 4)))
    tiles = O.extract(plan, X)
    for t in range(plan.num_tiles):
        (f0, _), (h0, _), (w0, _) = plan.box(t)
        v = tiles[t][0, 1]
        assert v[0, 0, 0] == f0 * 1000 + h0 * 100 + w0
        assert np.all(np.diff(v, axis=2) == 1) and np.all(np.diff(v, axis=1) == 100)
    flat = O.pack(tiles)
    assert flat.size == sum(x.size for x in tiles)
    back = O.unpack(plan, 1, 2, flat)
    assert all(np.array_equal(a, b) for a, b in zip(back, tiles))


# ---------------------------------------------------------------- blend
@pytest.mark.parametrize("name", ["tiny", "stage1", "strips", "grid"])
def test_blend_identity_reproduces_input(name):
    wl = WORKLOADS[name]
    C = min(wl.C, 4)
    X = inputs.latent((wl.B, C) + wl.dims, seed=0).astype(np.float64)
    plan = O.make_plan(wl.dims, wl.tiling)
    Y = O.blend(plan, O.extract(plan, X))
    assert np.max(np.abs(Y - X)) < 1e-12


def test_blend_shared_affine_is_affine():
    """All tiles get the same a*x+b: windows summing to one give a*X+b."""
    X = inputs.latent((1, 4, 16, 68, 120), seed=0).astype(np.float64)
    plan = O.make_plan((16, 68, 120), ((2, 2), (4, 8), (4, 12)))
    Y = O.blend(plan, [1.25 * t - 0.5 for t in O.extract(plan, X)])
    assert np.max(np.abs(Y - (1.25 * X - 0.5))) < 1e-12


def test_blend_of_ones_shows_table_excess():
    """A constant latent through a guard-violating split is brightened by the
    window-sum excess of the mold table."""
    for dim, n, ov, printed in read_golden_rows("mold_window_sum_table.txt"):
        dim, n, ov, printed = int(dim), int(n), int(ov), float(printed)
        plan = O.make_plan((1, 1, dim), ((1, 0), (1, 0), (n, ov)), compat=True)
        Y = O.blend(plan, O.extract(plan, np.ones((1, 1, 1, 1, dim))))
        assert abs(Y.max() - printed) <= 6e-4
        assert Y.min() >= 1.0 - 1e-12


def test_blend_hard_cut_without_overlap():
    """Overlap 0: every point belongs to one tile with weight 1."""
    rng = np.random.default_rng(3)
    plan = O.make_plan((3, 10, 13), ((3, 0), (2, 0), (4, 0)))
    X = rng.standard_normal((1, 2, 3, 10, 13))
    tiles = [rng.standard_normal(t.shape) for t in O.extract(plan, X)]
    Y = O.blend(plan, tiles)
    for t in range(plan.num_tiles):
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        assert np.array_equal(Y[:, :, f0:f1, h0:h1, w0:w1], tiles[t])


def test_single_tile_is_identity_copy():
    X = inputs.latent((1, 3, 4, 5, 6), seed=4).astype(np.float64)
    plan = O.make_plan((4, 5, 6), ((1, 0), (1, 0), (1, 0)))
    tiles = O.extract(plan, X)
    assert len(tiles) == 1 and np.array_equal(tiles[0], X)
    assert np.array_equal(O.blend(plan, tiles), X)


def test_blend_per_tile_affine_closed_form():
    """Y = x * sum_t w_t a_t + sum_t w_t b_t for y_t = a_t x + b_t."""
    plan = O.make_plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    X = inputs.latent((1, 8, 4, 16, 16), seed=0).astype(np.float64)
    a, b = (v.astype(np.float64) for v in inputs.affine_params(plan.num_tiles, seed=1))
    Y = O.blend(plan, [a[t] * x + b[t] for t, x in enumerate(O.extract(plan, X))])
    # per-axis exact weights, assembled point by point
    A = np.zeros(plan.dims)
    Bc = np.zeros(plan.dims)
    for f, h, w in itertools.product(*(range(d) for d in plan.dims)):
        for t in range(plan.num_tiles):
            i = plan.tile_index(t)
            wt = 1.0
            for d, x in enumerate((f, h, w)):
                wt *= float(O.ramp_exact(plan.intervals[d], plan.overlaps[d], i[d], x))
            A[f, h, w] += wt * a[t]
            Bc[f, h, w] += wt * b[t]
    assert np.max(np.abs(Y - (X * A + Bc))) < 1e-12


# ---------------------------------------------------------------- window sum
@pytest.mark.parametrize("cfg", [((2, 2), (4, 8), (4, 12)), ((3, 3), (3, 9), (5, 11))])
def test_window_sum_is_separable(cfg):
    dims = (16, 68, 120)
    plan = O.make_plan(dims, cfg, compat=True)
    S = O.window_sum(plan)
    Sd = [np.array([float(v) for v in O.window_sum_1d_exact(plan.intervals[d], plan.overlaps[d], dims[d])])
          for d in range(3)]
    assert np.max(np.abs(S - Sd[0][:, None, None] * Sd[1][None, :, None] * Sd[2][None, None, :])) < 1e-12


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_window_sum_is_one_under_guard(name):
    wl = WORKLOADS[name]
    plan = O.make_plan(wl.dims, wl.tiling)
    for d in range(3):
        exact = O.window_sum_1d_exact(plan.intervals[d], plan.overlaps[d], wl.dims[d])
        assert all(v == 1 for v in exact)
    assert O.max_abs_deviation(plan) < 1e-12


# ---------------------------------------------------------------- positions
@pytest.mark.parametrize("name", ["tiny", "stage1", "fullres", "4k"])
def test_normalized_positions_equal_fresh_tile_grid(name):
    """Normalised tile positions equal a position grid built at the tile's own
    shape (mold issue #673: what upstream's normalize_positions achieves)."""
    wl = WORKLOADS[name]
    F, H, W = wl.dims
    gen = inputs.grid_positions(2, F, H, W)
    plan = O.make_plan(wl.dims, wl.tiling)
    tp, off = O.positions(plan, gen, normalize=True)
    for t in range(plan.num_tiles):
        assert np.array_equal(tp[t], inputs.grid_positions(2, *plan.shape(t)))
        (f0, _), (h0, _), (w0, _) = plan.box(t)
        assert np.array_equal(off[t, 0], [f0 * 8, h0 * 32, w0 * 32])


def test_positions_origin_and_widths():
    F, H, W = 3, 7, 9
    gen = inputs.random_positions(2, F * H * W, seed=11)
    plan = O.make_plan((F, H, W), ((2, 1), (2, 2), (3, 2)))
    tp, off = O.positions(plan, gen, normalize=True)
    raw, off2 = O.positions(plan, gen, normalize=False)
    assert np.array_equal(off, off2)
    for t in range(plan.num_tiles):
        assert np.all(tp[t][..., 0].min(axis=2) == 0)
        assert np.array_equal(tp[t][..., 1] - tp[t][..., 0], raw[t][..., 1] - raw[t][..., 0])
        # brute-force gather of the unnormalised positions
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        j = 0
        for f in range(f0, f1):
            for h in range(h0, h1):
                for w in range(w0, w1):
                    n = (f * H + h) * W + w
                    assert np.array_equal(raw[t][:, :, j, :], gen[:, :, n, :])
                    j += 1


# ---------------------------------------------------------------- conditioning
def _cond_fixture():
    F, H, W = 4, 16, 16
    plan = O.make_plan((F, H, W), ((1, 0), (2, 4), (2, 4)))   # h, w tiles [0,10),[6,16)
    gen = inputs.grid_positions(1, F, H, W)
    return plan, gen


def test_cond_negative_time_kept_by_every_tile():
    plan, gen = _cond_fixture()
    cond = np.array([[[[-8, 0]], [[10000, 10032]], [[-500, -400]]]], dtype=np.int32)  # outside in h, w
    sel = O.cond_select(plan, gen, cond)
    assert sel.count[0, 0] == plan.num_tiles
    assert sel.weight[0, 0] == np.float32(1.0) / np.float32(4.0)


def test_cond_hand_cases():
    plan, gen = _cond_fixture()
    # token 0: rows/cols [0,32) in px = latent unit 0 -> only tile 0
    # token 1: latent units 7..8 in h and w ([224, 288) px) -> inside the
    #          overlap on both axes -> all 4 tiles
    # token 2: h unit 7 (overlap), w unit 15 (right only) -> tiles 1 and 3
    # token 3: zero-width time interval at t=0: overlaps nothing
    # token 4: h interval ends exactly where tile 1 starts ([0, 192) px):
    #          half-open, so only tiles 0 and 1 (h tile 0)
    cond = np.zeros((1, 3, 5, 2), dtype=np.int32)
    spans = [((0, 8), (0, 32), (0, 32)),
             ((0, 8), (224, 288), (224, 288)),
             ((0, 8), (224, 256), (480, 512)),
             ((0, 0), (0, 512), (0, 512)),
             ((0, 8), (0, 192), (0, 512))]
    for m, sp in enumerate(spans):
        for d in range(3):
            cond[0, d, m] = sp[d]
    sel = O.cond_select(plan, gen, cond)
    assert sel.keep[:, 0, 0].tolist() == [True, False, False, False]
    assert sel.keep[:, 0, 1].tolist() == [True, True, True, True]
    assert sel.keep[:, 0, 2].tolist() == [False, True, False, True]
    assert sel.keep[:, 0, 3].tolist() == [False] * 4
    assert sel.keep[:, 0, 4].tolist() == [True, True, False, False]
    assert sel.count[0].tolist() == [1, 4, 2, 0, 2]
    assert sel.weight[0].tolist() == [1.0, 0.25, 0.5, 0.0, 0.5]
    # kept tokens keep their original order and are shifted by the tile offset
    assert sel.kept[3][0].tolist() == [1, 2]
    assert sel.tile_cond_pos[3][0][1, 0].tolist() == [224 - 6 * 32, 288 - 6 * 32]   # token 1
    assert sel.tile_cond_pos[3][0][1, 1].tolist() == [224 - 6 * 32, 256 - 6 * 32]   # token 2
    assert sel.tile_cond_pos[3][0][2, 1].tolist() == [480 - 6 * 32, 512 - 6 * 32]


def test_cond_bruteforce_tiny():
    """Keep iff negative time start, or for every axis some generated token of
    the tile overlaps the interval (the grid has no gaps, so this is overlap
    with the tile's extent)."""
    F, H, W = 3, 6, 8
    gen = inputs.grid_positions(2, F, H, W)
    cond = inputs.cond_positions(2, 40, F, H, W, n_negative=6, seed=9)
    plan = O.make_plan((F, H, W), ((1, 0), (2, 2), (3, 2)))
    sel = O.cond_select(plan, gen, cond)
    for t in range(plan.num_tiles):
        toks = O.tile_token_indices(plan, t)
        for b in range(2):
            for m in range(40):
                keep = cond[b, 0, m, 0] < 0
                if not keep:
                    keep = all(any(gen[b, d, n, 0] < cond[b, d, m, 1] and gen[b, d, n, 1] > cond[b, d, m, 0]
                                   for n in toks) for d in range(3))
                assert sel.keep[t, b, m] == keep
    for b in range(2):
        for m in range(40):
            c = int(sel.keep[:, b, m].sum())
            assert sel.count[b, m] == c
            assert sel.weight[b, m] == (np.float32(Fraction(1, c)) if c else np.float32(0))


# ---------------------------------------------------------------- stats
def test_distvae_strip_figures():
    g = {r[0]: r[1:] for r in read_golden_rows("distvae_strips.txt")}
    H, W = int(g["latent_h"][0]), int(g["latent_w"][0])
    rows = [int(v) for v in g["strip_rows"]]
    iv, start = [], 0
    for r in rows:
        iv.append((start, start + r))
        start += 32                         # stride 32 = 43 - overlap 11
    assert iv[-1][1] == H
    st = O.layout_stats([[(0, 1)], iv, [(0, W)]], (1, H, W), ranks=int(g["ranks"][0]))
    assert round(st.decoded_area, 2) == float(g["decoded_area"][0])
    assert round(st.tile_fraction, 2) == float(g["tile_fraction"][0])
    assert round(st.imbalance, 3) == float(g["imbalance"][0])
    assert st.seams == int(g["seams"][0])
    grid = O.make_plan((1, 128, 128), ((1, 0), (int(g["grid_rows"][0]), 8), (int(g["grid_cols"][0]), 8)))
    assert O.layout_stats(grid.intervals, grid.dims, 4).seams == int(g["grid_seams"][0])


# --------------------------------------------------------------------------
# Conditioning-token combine (TDP §Shared negative (reference) positions: a
# token kept by k tiles has blend weight 1/k).
def _cond_case(seed=0, D=5):
    dims, cfg = (5, 37, 53), ((2, 1), (3, 5), (4, 6))
    plan = O.make_plan(dims, cfg)
    gen = inputs.grid_positions(2, *dims)
    cond = inputs.cond_positions(2, 60, *dims, n_negative=9, seed=seed)
    sel = O.cond_select(plan, gen, cond)
    rng = np.random.default_rng(seed)
    T, B, M = sel.keep.shape
    tile_out = rng.standard_normal((T, B, M, D))
    return sel, tile_out


def test_cond_combine_matches_cumsum_slots():
    # independent slot derivation: slot = (number of kept tokens up to m) - 1
    sel, x = _cond_case(3)
    T, B, M = sel.keep.shape
    slot = np.cumsum(sel.keep, axis=2) - 1
    ref = np.zeros((B, M, x.shape[-1]))
    for t in range(T):
        k = sel.keep[t]                                   # [B, M]
        gathered = np.take_along_axis(x[t], np.where(k, slot[t], 0)[..., None], axis=1)
        ref += np.where(k[..., None], gathered / np.maximum(sel.count, 1)[..., None], 0.0)
    assert np.array_equal(O.cond_slots(sel), np.where(sel.keep, slot, -1))
    assert np.allclose(O.cond_combine(sel, x), ref, rtol=0, atol=1e-12)


def test_cond_combine_single_keeper_is_a_copy_and_unkept_is_zero():
    sel, x = _cond_case(4)
    out = O.cond_combine(sel, x)
    slot = O.cond_slots(sel)
    one = sel.count == 1
    none = sel.count == 0
    assert one.any() and none.any()
    for b, m in zip(*np.nonzero(one)):
        t = int(np.nonzero(sel.keep[:, b, m])[0][0])
        assert np.array_equal(out[b, m], x[t, b, slot[t, b, m]])   # weight exactly 1
    assert np.all(out[none] == 0.0)


def test_cond_combine_partition_of_unity_and_reference_tokens():
    sel, _ = _cond_case(5)
    T, B, M = sel.keep.shape
    rng = np.random.default_rng(9)
    v = rng.standard_normal((B, M, 3))
    slot = O.cond_slots(sel)
    x = np.zeros((T, B, M, 3))
    for t in range(T):
        for b in range(B):
            for m in range(M):
                if slot[t, b, m] >= 0:
                    x[t, b, slot[t, b, m]] = v[b, m]       # every keeper returns the same value
    out = O.cond_combine(sel, x)
    kept = sel.count > 0
    assert np.allclose(out[kept], v[kept], rtol=1e-12, atol=1e-12)
    # reference (negative time) tokens are kept by every tile, weight 1/T each
    cond_neg = sel.keep.all(axis=0)
    assert cond_neg.any() and np.all(sel.count[cond_neg] == T)


# ---------------------------------------------------------------- token-major tiles
def test_extract_tokens_bruteforce_order():
    """Each token of each tile, found by walking the tile's box in (f, h, w)
    order with a running counter, holds that point's C channels."""
    rng = np.random.default_rng(7)
    X = rng.standard_normal((2, 5, 5, 9, 11))
    plan = O.make_plan((5, 9, 11), ((2, 1), (3, 2), (2, 3)))
    tok = O.extract_tokens(plan, X)
    for t in range(plan.num_tiles):
        (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
        assert tok[t].shape == (2, (f1 - f0) * (h1 - h0) * (w1 - w0), 5)
        n = 0
        for f in range(f0, f1):
            for h in range(h0, h1):
                for w in range(w0, w1):
                    for b in range(2):
                        for c in range(5):
                            assert tok[t][b, n, c] == X[b, c, f, h, w]
                    n += 1
        assert n == tok[t].shape[1]


def test_extract_tokens_carry_their_positions():
    """Token n of tile t sits at the point whose generated-token position is
    the n-th entry of the tile's (unnormalised) position list: the value
    latent encodes each point's grid position, so the two layouts agree."""
    F, H, W = 4, 16, 16
    plan = O.make_plan((F, H, W), ((2, 1), (2, 4), (2, 4)))
    gen = inputs.grid_positions(1, F, H, W)
    f, h, w = np.meshgrid(np.arange(F), np.arange(H), np.arange(W), indexing="ij")
    X = np.stack([f * 8, h * 32, w * 32]).astype(np.float64)[None]      # [1, 3, F, H, W]
    tok = O.extract_tokens(plan, X)
    raw, _ = O.positions(plan, gen, normalize=False)
    for t in range(plan.num_tiles):
        assert np.array_equal(tok[t][0].T, raw[t][0, :, :, 0])           # [3, N_t] starts


def test_extract_tokens_single_tile_is_patchify():
    """One tile: the token sequence is the latent flattened over (F, H, W)
    and transposed to channel-last."""
    X = inputs.latent((2, 3, 4, 5, 6), seed=4).astype(np.float64)
    plan = O.make_plan((4, 5, 6), ((1, 0), (1, 0), (1, 0)))
    tok = O.extract_tokens(plan, X)
    assert len(tok) == 1
    assert np.array_equal(tok[0], np.moveaxis(X.reshape(2, 3, 120), 1, 2))
    assert np.array_equal(O.blend_tokens(plan, tok), X)


@pytest.mark.parametrize("name", ["tiny", "stage1", "strips", "grid"])
def test_blend_tokens_identity_reproduces_input(name):
    wl = WORKLOADS[name]
    X = inputs.latent((wl.B, min(wl.C, 4)) + wl.dims, seed=0).astype(np.float64)
    plan = O.make_plan(wl.dims, wl.tiling)
    assert np.max(np.abs(O.blend_tokens(plan, O.extract_tokens(plan, X)) - X)) < 1e-12


def test_blend_tokens_bruteforce_exact_weights():
    """Per-tile, per-channel random token outputs, summed point by point with
    the exact rational window of each tile (no reshape, no window array)."""
    rng = np.random.default_rng(9)
    dims = (3, 7, 9)
    plan = O.make_plan(dims, ((2, 1), (2, 2), (3, 2)), compat=True)
    C = 3
    tok = [rng.standard_normal((1, int(np.prod(plan.shape(t))), C)) for t in range(plan.num_tiles)]
    Y = O.blend_tokens(plan, tok)
    for f, h, w in itertools.product(*(range(d) for d in dims)):
        want = np.zeros(C)
        for t in range(plan.num_tiles):
            (f0, f1), (h0, h1), (w0, w1) = plan.box(t)
            if not (f0 <= f < f1 and h0 <= h < h1 and w0 <= w < w1):
                continue
            i = plan.tile_index(t)
            wt = Fraction(1)
            for d, x in enumerate((f, h, w)):
                wt *= O.ramp_exact(plan.intervals[d], plan.overlaps[d], i[d], x)
            n = ((f - f0) * (h1 - h0) + (h - h0)) * (w1 - w0) + (w - w0)
            want += float(wt) * tok[t][0, n]
        assert np.max(np.abs(Y[0, :, f, h, w] - want)) < 1e-12


def test_blend_tokens_agrees_with_channel_first_blend():
    """The same per-tile outputs in either layout blend to the same latent."""
    rng = np.random.default_rng(12)
    plan = O.make_plan((16, 68, 120), ((2, 2), (4, 8), (4, 12)))
    B, C = 1, 2
    tiles = [rng.standard_normal((B, C) + plan.shape(t)) for t in range(plan.num_tiles)]
    tok = [np.moveaxis(x.reshape(B, C, -1), 1, 2) for x in tiles]
    assert np.max(np.abs(O.blend_tokens(plan, tok) - O.blend(plan, tiles))) < 1e-12


def test_tokens_packing_uses_channel_first_offsets():
    plan = O.make_plan((5, 9, 11), ((2, 1), (3, 2), (2, 3)))
    X = np.random.default_rng(2).standard_normal((2, 4, 5, 9, 11))
    tok = O.extract_tokens(plan, X)
    flat = O.pack(tok)
    assert flat.size == O.pack(O.extract(plan, X)).size
    back = O.unpack_tokens(plan, 2, 4, flat)
    assert all(np.array_equal(a, b) for a, b in zip(back, tok))


# ---------------------------------------------------------------- layout planning
def test_balanced_tile_split_is_the_squarest_factor_pair():
    assert [O.balanced_tile_split(r) for r in (1, 2, 4, 6, 8, 12, 16, 7)] == \
        [(1, 1), (1, 2), (2, 2), (2, 3), (2, 4), (3, 4), (4, 4), (1, 7)]
    for r in range(1, 300):
        h, w = O.balanced_tile_split(r)
        pairs = [(a, r // a) for a in range(1, r + 1) if r % a == 0]
        assert h * w == r and h <= w
        assert w - h == min(abs(b - a) for a, b in pairs)


@pytest.mark.parametrize("ranks", [2, 3])
def test_search_layouts_hand_worked_cases(golden_rows, ranks):
    got = {(c.counts, c.window_volume, c.decoded_volume, c.heaviest_rank_volume, c.seams, c.role)
           for c in O.search_layouts((1, 32, 32), ranks, (1, 0), 4, 4)}
    want = {((int(r[0]), int(r[1]), int(r[2])), int(r[3]), int(r[4]), int(r[5]), int(r[6]), r[7])
            for r in golden_rows(f"plan_search_32x32_r{ranks}.txt")}
    assert got == want


def test_dominance_compares_imbalance_as_a_share():
    """Less decoded work does not beat a layout whose heaviest rank carries a
    smaller share of its (larger) total: 60/100 of the work against 100/200."""
    a = O.LayoutCandidate((1, 2, 1), (0, 4, 0), 10, 100, 60, 1)
    b = O.LayoutCandidate((1, 2, 1), (0, 4, 0), 10, 200, 100, 1)
    assert not O._beats(a, b) and not O._beats(b, a)
    c = O.LayoutCandidate((1, 2, 1), (0, 4, 0), 10, 100, 50, 1)
    assert O._beats(c, b) and not O._beats(b, c)
    d = O.LayoutCandidate((1, 1, 2), (0, 0, 4), 10, 100, 50, 2)    # same, one more tile column
    assert O._beats(c, d) and not O._beats(d, c)


@pytest.mark.parametrize("dims,ranks,frames,oh,ow,limits", [
    ((16, 68, 120), 8, (2, 2), 8, 12, True),
    ((16, 68, 120), 4, (1, 0), 8, 12, True),
    ((1, 128, 128), 4, (1, 0), 8, 8, True),
    ((16, 32, 48), 2, (1, 0), 8, 12, False),
    ((16, 16, 24), 4, (1, 0), 4, 6, False),
])
def test_search_layouts_frontier_properties(dims, ranks, frames, oh, ow, limits):
    cands = O.search_layouts(dims, ranks, frames, oh, ow, limits=limits)
    assert cands
    front = [c for c in cands if c.role != "dominated"]
    for c in cands:
        T = c.counts[0] * c.counts[1] * c.counts[2]
        assert max(2, ranks) <= T <= 4 * ranks
        beaten = any(O._beats(d, c) for d in cands)
        assert beaten == (c.role == "dominated")
        if beaten:     # beaten by the frontier itself (the relation is transitive)
            assert any(O._beats(d, c) for d in front)
    roles = [c.role for c in front]
    assert roles.count("coarse") == 1 and roles.count("fine") == (len(front) > 1)
    assert roles.count("balanced") == (len(front) > 2)
    coarse = next(c for c in front if c.role == "coarse")
    assert coarse.window_volume == max(c.window_volume for c in front)
    if len(front) > 1:
        fine = next(c for c in front if c.role == "fine")
        assert fine.window_volume == min(c.window_volume for c in front if c is not coarse)


def test_search_layouts_contains_the_4k_workload_tiling():
    """The bench's 4k tiling (2x4x4, overlaps 2/8/12) is a supported grid
    for 8 ranks; its window is one tile of 9x23x39 tokens."""
    cands = O.search_layouts((16, 68, 120), 8, (2, 2), 8, 12)
    c = next(c for c in cands if c.counts == (2, 4, 4))
    assert c.window_volume == 9 * 23 * 39
    assert c.decoded_volume == 32 * 9 * 23 * 39
    assert c.heaviest_rank_volume * 8 == c.decoded_volume   # 32 equal tiles over 8 ranks


def test_search_layouts_limits():
    # a latent narrower than 16 units, or than one unit per rank, has no candidate
    assert O.search_layouts((1, 15, 64), 2, (1, 0), 4, 4) == []
    assert O.search_layouts((1, 20, 64), 24, (1, 0), 4, 4) == []
    # without the limits the quarter-window rule no longer drops wide windows
    with_l = {c.counts for c in O.search_layouts((1, 32, 32), 2, (1, 0), 4, 4)}
    without = {c.counts for c in O.search_layouts((1, 32, 32), 2, (1, 0), 4, 4, limits=False)}
    assert (1, 2, 1) in without - with_l
