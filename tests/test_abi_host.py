"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/tdp.h declares, and its host planner / statistics match the oracle
bit for bit.  Device entry points are only called on argument errors that
return before any CUDA call."""
import ctypes as C
import itertools
import os
import re

import numpy as np
import pytest

from oracle import tdp_oracle as O
from overlap_add_blending_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def T():
    from overlap_add_blending_gb300 import build
    build.build()
    from overlap_add_blending_gb300 import tdp
    return tdp


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tdp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tdp_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(T):
    names = declared_functions()
    assert len(names) >= 12
    lib = C.CDLL(T.library_path())
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(T.EXPORTS)


def _oracle_plan_or_error(dims, cfg, compat):
    try:
        return O.make_plan(dims, cfg, compat=compat)
    except O.GuardError:
        return "guard"
    except ValueError:
        return "invalid"


def test_plan_matches_oracle_exhaustive_small(T):
    seen_guard = seen_ok = 0
    for D, n, o in itertools.product(range(1, 26), range(1, 7), range(0, 9)):
        for compat in (False, True):
            dims, cfg = (1, 3, D), ((1, 0), (1, 0), (n, o))
            ref = _oracle_plan_or_error(dims, cfg, compat)
            if isinstance(ref, str):
                with pytest.raises(T.TdpError) as e:
                    T.plan(dims, cfg, compat=compat)
                assert e.value.status == (2 if ref == "guard" else 1)
                seen_guard += ref == "guard"
                continue
            p = T.plan(dims, cfg, compat=compat)
            assert p.intervals(2) == ref.intervals[2]
            seen_ok += 1
    assert seen_guard > 50 and seen_ok > 300


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_plans_and_offsets(T, name):
    wl = WORKLOADS[name]
    p = T.plan(wl.dims, wl.tiling)
    ref = O.make_plan(wl.dims, wl.tiling)
    assert p.T == ref.num_tiles
    for d in range(3):
        assert p.intervals(d) == ref.intervals[d]
    # packed offsets are the running sum of tile sizes in tile order
    B, Cc = 2, 3
    run = 0
    for t in range(p.T):
        start, size = p.box(t)
        box = ref.box(t)
        assert start == tuple(b[0] for b in box) and size == ref.shape(t)
        assert p.tile_offset(t, B, Cc) == run
        run += B * Cc * int(np.prod(size))
    assert p.tiles_numel(B, Cc) == run


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("ranks", [1, 2, 3, 4, 8])
def test_plan_stats_match_oracle(T, name, ranks):
    wl = WORKLOADS[name]
    p = T.plan(wl.dims, wl.tiling)
    ref = O.make_plan(wl.dims, wl.tiling)
    st = T.plan_stats(p, ranks)
    rs = O.layout_stats(ref.intervals, ref.dims, ranks)
    assert st.seams == rs.seams
    assert abs(st.decoded_area - rs.decoded_area) < 1e-12
    assert abs(st.tile_fraction - rs.tile_fraction) < 1e-12
    assert abs(st.imbalance - rs.imbalance) < 1e-12
    assert abs(st.max_window_sum - float(O.window_sum(ref).max())) < 1e-12


def test_plan_stats_guard_violating_splits(T):
    for dim, n, ov, printed in [(21, 2, 8, 1.000), (21, 3, 8, 1.074), (21, 4, 8, 1.161)]:
        p = T.plan((1, 1, dim), ((1, 0), (1, 0), (n, ov)), compat=True)
        ref = O.make_plan((1, 1, dim), ((1, 0), (1, 0), (n, ov)), compat=True)
        mw = T.plan_stats(p).max_window_sum
        assert abs(mw - float(O.window_sum(ref).max())) < 1e-12
        assert abs(mw - printed) <= 6e-4


def test_plan_rejections(T):
    with pytest.raises(T.TdpError) as e:
        T.plan((16, 68, 120), ((2, 2), (4, 8), (65, 1)))
    assert e.value.status == 3
    for bad in [((1, 2), (1, 0), (1, 0)),        # one tile with overlap
                ((1, 0), (1, 0), (200, 0)),      # more tiles than columns
                ((0, 0), (1, 0), (1, 0))]:
        with pytest.raises(T.TdpError):
            T.plan((16, 68, 120), bad)
    with pytest.raises(T.TdpError):
        T.plan((0, 4, 4), ((1, 0), (1, 0), (1, 0)))


def test_device_calls_reject_bad_arguments_before_launch(T):
    lib = C.CDLL(T.library_path())
    lib.tdp_extract.argtypes = T._lib.tdp_extract.argtypes
    lib.tdp_blend.argtypes = T._lib.tdp_blend.argtypes
    lib.tdp_window_sum.argtypes = T._lib.tdp_window_sum.argtypes
    p = T.plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    P = C.byref(p)
    good, odd = 0x10000, 0x10004
    assert lib.tdp_extract(P, 1, 8, 0, None, C.c_void_p(good), None) == 1       # null latent
    assert lib.tdp_extract(P, 1, 8, 0, C.c_void_p(odd), C.c_void_p(good), None) == 4
    assert lib.tdp_extract(P, 1, 8, 7, C.c_void_p(good), C.c_void_p(good), None) == 1   # bad dtype
    assert lib.tdp_extract(P, -1, 8, 0, C.c_void_p(good), C.c_void_p(good), None) == 1
    assert lib.tdp_extract(P, 0, 8, 0, None, None, None) == 0                   # empty batch
    assert lib.tdp_blend(P, 1, 8, 0, C.c_void_p(good), 1, C.c_void_p(odd), None) == 4
    assert lib.tdp_window_sum(P, None, None, None) == 1
    # a hand-edited plan is refused
    q = T.Plan.from_buffer_copy(p)
    q.end[1][0] += 1
    assert lib.tdp_extract(C.byref(q), 1, 8, 0, C.c_void_p(good), C.c_void_p(good), None) == 1
    assert lib.tdp_plan_stats(C.byref(q), 1, None, None, None, None, None) == 1


# ----------------------------------------------------------------- layout planner (host)
def test_balanced_tile_split_matches_oracle(T):
    for r in range(1, 300):
        assert T.balanced_tile_split(r) == O.balanced_tile_split(r)
    with pytest.raises(T.TdpError):
        T.balanced_tile_split(0)


@pytest.mark.parametrize("dims,ranks,frames,oh,ow,compat,limits", [
    ((1, 32, 32), 2, (1, 0), 4, 4, False, True),
    ((1, 32, 32), 3, (1, 0), 4, 4, False, True),
    ((16, 68, 120), 1, (2, 2), 8, 12, False, True),
    ((16, 68, 120), 2, (2, 2), 8, 12, False, True),
    ((16, 68, 120), 4, (2, 2), 8, 12, False, True),
    ((16, 68, 120), 8, (2, 2), 8, 12, False, True),
    ((16, 68, 120), 16, (2, 2), 8, 12, False, True),
    ((16, 68, 120), 8, (1, 0), 5, 5, False, False),
    ((1, 128, 128), 4, (1, 0), 8, 8, False, True),
    ((1, 128, 128), 8, (1, 0), 8, 8, False, False),
    ((16, 16, 24), 4, (1, 0), 4, 6, False, False),
    ((16, 32, 48), 2, (1, 0), 8, 12, False, False),
    ((1, 21, 21), 4, (1, 0), 8, 8, True, False),
    ((1, 15, 64), 2, (1, 0), 4, 4, False, True),      # narrow axis below 16: no candidate
])
def test_search_layouts_matches_oracle(T, dims, ranks, frames, oh, ow, compat, limits):
    got = T.search_layouts(dims, ranks, frames, oh, ow, compat=compat, limits=limits)
    want = O.search_layouts(dims, ranks, frames, oh, ow, compat=compat, limits=limits)
    assert [(c["counts"], c["overlaps"], c["window_volume"], c["decoded_volume"], c["heaviest_rank_volume"],
             c["seams"], c["role"]) for c in got] == \
        [(c.counts, c.overlaps, c.window_volume, c.decoded_volume, c.heaviest_rank_volume, c.seams, c.role)
         for c in want]


def test_search_layouts_random_shapes_match_oracle(T):
    rng = np.random.default_rng(21)
    for _ in range(60):
        dims = (int(rng.integers(1, 5)), int(rng.integers(8, 90)), int(rng.integers(8, 130)))
        ranks = int(rng.integers(1, 13))
        frames = (1, 0) if dims[0] < 4 or rng.random() < 0.5 else (2, 1)
        oh, ow = int(rng.integers(0, 12)), int(rng.integers(0, 12))
        limits = bool(rng.random() < 0.5)
        got = T.search_layouts(dims, ranks, frames, oh, ow, limits=limits)
        want = O.search_layouts(dims, ranks, frames, oh, ow, limits=limits)
        assert [(c["counts"], c["heaviest_rank_volume"], c["role"]) for c in got] == \
            [(c.counts, c.heaviest_rank_volume, c.role) for c in want], (dims, ranks, frames, oh, ow, limits)


def test_search_layouts_capacity_and_errors(T):
    import ctypes as C_
    d = (C_.c_int32 * 3)(1, 32, 32)
    fr = T.DimCfg(1, 0)
    n = C_.c_int32()
    lib = T._lib
    assert lib.tdp_search_layouts(C_.byref(d), 3, C_.byref(fr), 4, 4, 0, None, 0, C_.byref(n)) == 0
    assert n.value == 13
    buf = (T.LayoutCandidate * 4)()
    assert lib.tdp_search_layouts(C_.byref(d), 3, C_.byref(fr), 4, 4, 0, buf, 4, C_.byref(n)) == 0
    assert n.value == 13 and tuple(buf[3].num_tiles) == (1, 1, 6)
    assert lib.tdp_search_layouts(C_.byref(d), 0, C_.byref(fr), 4, 4, 0, None, 0, C_.byref(n)) == 1
    assert lib.tdp_search_layouts(C_.byref(d), 3, C_.byref(fr), 4, 4, 8, None, 0, C_.byref(n)) == 1
    assert lib.tdp_search_layouts(C_.byref(d), 3, C_.byref(fr), 4, 4, 0, None, 2, C_.byref(n)) == 1


def test_token_major_calls_reject_before_any_cuda_call(T):
    """Argument errors of tdp_extract_tokens / tdp_blend_tokens return before
    the library touches CUDA (fake, never dereferenced 16-byte-aligned pointers)."""
    import ctypes as C_
    lib = T._lib
    p = T.plan((2, 4, 6), ((1, 0), (1, 0), (1, 0)))
    ok, bad = C_.c_void_p(4096), C_.c_void_p(4104)   # 16-byte aligned / 8-byte aligned
    BF16, F32 = T.BF16, T.F32
    ex, bl = lib.tdp_extract_tokens, lib.tdp_blend_tokens
    assert ex(C_.byref(p), 1, 3, BF16, ok, ok, None) == 6          # 6-byte tokens
    assert bl(C_.byref(p), 1, 3, BF16, ok, BF16, ok, None) == 6
    assert bl(C_.byref(p), 1, 2056, BF16, ok, BF16, ok, None) == 6  # 257 chunks per token, odd
    assert ex(C_.byref(p), 1, 8208, BF16, ok, ok, None) == 6        # past 16 KiB per token
    assert ex(C_.byref(p), 1, 8, BF16, bad, ok, None) == 4          # alignment
    assert bl(C_.byref(p), 1, 8, BF16, ok, F32, bad, None) == 4
    assert ex(C_.byref(p), 1, 8, BF16, None, ok, None) == 1         # null pointer
    assert ex(C_.byref(p), 1, 8, 7, ok, ok, None) == 1              # unknown dtype
    assert ex(C_.byref(p), 0, 8, BF16, None, None, None) == 0       # empty batch: nothing to do
    assert bl(C_.byref(p), 1, 0, BF16, None, BF16, None, None) == 0
    q = T.Plan()
    C_.memmove(C_.byref(q), C_.byref(p), C_.sizeof(p))
    q.stride[2] += 1                                                # not what tdp_plan produces
    assert ex(C_.byref(q), 1, 8, BF16, ok, ok, None) == 1


def test_bench_algorithmic_bytes_of_the_4k_workload(T):
    """Extract reads the latent and writes the tiles; blend reads the tiles
    and writes the latent.  On the 4k workload the tile sizes per axis are
    9 + 9 frames, 4 x 23 rows and 4 x 39 columns, so the tiles hold
    18 * 92 * 156 tokens of 128 bf16 channels."""
    import bench
    wl = WORKLOADS["4k"]
    p = T.plan(wl.dims, wl.tiling)
    latent = 16 * 68 * 120 * 128
    tiles = 18 * 92 * 156 * 128
    assert p.tiles_numel(1, 128) == tiles
    ab = bench.algorithmic_bytes(wl, tiles)
    assert ab["extract"] == ab["blend"] == 2 * (latent + tiles) == 99_557_376
    assert ab["total"] == 199_114_752
    assert round(ab["overlap_factor"], 5) == 1.97868


def test_extract_and_tokens_workspace_size(T):
    """tdp_extract_and_tokens_workspace (host only): per (tile, batch) pair,
    6 int32 for each of its K1 token chunks -- K1 = the most of ceil(tile
    tokens / 3072) and 256 CTAs // pairs -- then one int32 per batch, rounded
    up to 16 bytes; 0 for no batch; a negative batch is rejected."""
    wl = WORKLOADS["4k"]
    p = T.plan(wl.dims, wl.tiling)   # 32 tiles of 9 x 23 x 39 = 8073 tokens: 3 chunks of 3072 at least
    r16 = lambda n: -(-n // 16) * 16
    for B in (1, 2, 3, 6, 9):
        pairs = 32 * B
        K1 = max(3, 256 // pairs)
        assert T.extract_and_tokens_workspace(p, B) == r16((pairs * K1 * 6 + B) * 4), B
    assert T.extract_and_tokens_workspace(p, 0) == 0
    with pytest.raises(ValueError):
        T.extract_and_tokens_workspace(p, -1)
