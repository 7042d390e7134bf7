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
