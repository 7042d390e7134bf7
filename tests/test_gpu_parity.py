"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Integer outputs (tiles as bit copies, positions, keep masks, counts, kept
lists, 1/count weights) must match exactly; blended floats must be within
max-abs 1e-5 (fp32 output) or 8e-3 relative (bf16 output) of the oracle,
which accumulates in float64."""
import numpy as np
import pytest
import torch

from oracle import tdp_oracle as O
from overlap_add_blending_gb300 import inputs
from overlap_add_blending_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def T():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from overlap_add_blending_gb300 import tdp
    return tdp


def _dev(x_np, dtype):
    return torch.from_numpy(np.ascontiguousarray(x_np)).to(dtype).cuda()


def _np64(t):
    return t.detach().cpu().double().numpy()


def apply_affine(T, p, tiles, B, C, a, b):
    """The per-tile op between extract and blend (the caller's work, here a_t*x + b_t)."""
    out = torch.empty_like(tiles)
    for t in range(p.T):
        _, size = p.box(t)
        n = B * C * size[0] * size[1] * size[2]
        o = p.tile_offset(t, B, C)
        out[o:o + n] = (tiles[o:o + n].float() * float(a[t]) + float(b[t])).to(tiles.dtype)
    return out


def check_blend(Y, ref, ref_abs, out_dtype):
    Y = _np64(Y)
    if out_dtype == torch.float32:
        err = np.max(np.abs(Y - ref)) if Y.size else 0.0
        assert err <= 1e-5, err
    else:
        bound = 8e-3 * np.abs(ref) + 1e-5 * ref_abs + 1e-30
        bad = np.abs(Y - ref) > bound
        assert not bad.any(), (np.abs(Y - ref)[bad][:5], ref[bad][:5])


def run_path(T, dims, tiling, B, C, dtype, op="affine", compat=False, out_dtype=None, seed=0):
    p = T.plan(dims, tiling, compat=compat)
    ref_plan = O.make_plan(dims, tiling, compat=compat)
    Xf = inputs.latent((B, C) + tuple(dims), seed=seed)
    X = _dev(Xf, dtype)
    tiles = T.extract(p, X)
    # extract is a bit copy
    ref_tiles = O.pack(O.extract(ref_plan, _np64(X)))
    assert torch.equal(tiles.cpu(), torch.from_numpy(ref_tiles).to(dtype)), "extract mismatch"
    if op == "affine":
        a, b = inputs.affine_params(p.T, seed=1)
        tiles = apply_affine(T, p, tiles, B, C, a, b)
    Y = T.blend(p, tiles, B, C, out_dtype=out_dtype or dtype)
    torch.cuda.synchronize()
    tl = O.unpack(ref_plan, B, C, _np64(tiles))
    check_blend(Y, O.blend(ref_plan, tl), O.blend_abs(ref_plan, tl), out_dtype or dtype)
    assert T.device_error() == 0
    return p, X, Y


# ----------------------------------------------------------------- named workloads
@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("op", ["identity", "affine"])
def test_extract_blend_workloads(T, name, op):
    wl = WORKLOADS[name]
    p, X, Y = run_path(T, wl.dims, wl.tiling, wl.B, wl.C, TORCH_DT[wl.dtype], op=op)
    if op == "identity":
        # windows sum to one: blend(extract(X)) reproduces X -- exactly in
        # bf16 (the fp32 sum is within a few fp32 ulp of x, far inside half a
        # bf16 ulp), within weight rounding in fp32
        if wl.dtype == "bf16":
            assert torch.equal(Y, X)
        else:
            assert (Y - X).abs().max().item() <= 1e-5


def test_4k_identity_roundtrip_is_near_exact(T):
    wl = WORKLOADS["4k"]
    p, X, Y = run_path(T, wl.dims, wl.tiling, wl.B, wl.C, torch.bfloat16, op="identity", out_dtype=torch.float32)
    # fp32 output of a bf16 identity round trip: only weight rounding remains
    assert (Y - X.float()).abs().max().item() <= 2e-6 * X.float().abs().max().item() + 1e-7


def test_4k_two_batches(T):
    # the 4k tiling with B = 2, C = 64: batch offsets in every kernel and
    # 128 items per (frame, band) group split by cost across the blend's CTAs
    wl = WORKLOADS["4k"]
    run_path(T, wl.dims, wl.tiling, 2, 64, torch.bfloat16, seed=5)


# ----------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_odd_shapes(T, dtype):
    # remainders on every axis, odd W (single-column stores), odd tile starts
    run_path(T, (5, 37, 53), ((2, 1), (3, 5), (4, 6)), 2, 3, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_row_bands(T, dtype):
    # planes larger than the shared-memory budget are cut into row bands
    run_path(T, (2, 300, 200), ((1, 0), (3, 20), (2, 16)), 1, 2, dtype)


@pytest.mark.parametrize("in_dt,out_dt", [(torch.bfloat16, torch.float32), (torch.float32, torch.bfloat16)])
def test_mixed_dtypes(T, in_dt, out_dt):
    run_path(T, (4, 16, 24), ((1, 0), (2, 4), (2, 6)), 1, 16, in_dt, out_dtype=out_dt)


def test_single_tile_identity_copy(T):
    p, X, Y = run_path(T, (3, 9, 10), ((1, 0), (1, 0), (1, 0)), 2, 2, torch.float32, op="identity")
    assert torch.equal(X, Y)


def test_hard_cut_overlap_zero(T):
    p, X, Y = run_path(T, (3, 10, 14), ((3, 0), (2, 0), (4, 0)), 1, 4, torch.float32, op="identity")
    assert torch.equal(X, Y)


@pytest.mark.parametrize("n", [2, 3, 4])
def test_guard_violating_splits_brighten(T, n):
    dims, tiling = (1, 1, 21), ((1, 0), (1, 0), (n, 8))
    p = T.plan(dims, tiling, compat=True)
    X = torch.ones((1, 2) + dims, dtype=torch.float32, device="cuda")
    Y = T.blend(p, T.extract(p, X), 1, 2)
    rp = O.make_plan(dims, tiling, compat=True)
    ref = O.blend(rp, O.extract(rp, np.ones((1, 2) + dims)))
    check_blend(Y, ref, ref, torch.float32)
    printed = {2: 1.000, 3: 1.074, 4: 1.161}[n]
    assert abs(Y.max().item() - printed) <= 6e-4


def test_blend_cost_split_leaves_a_cta_without_items(T):
    # 3 items (B*C = 1, 3 frames, the middle one in both frame tiles) on 3
    # CTAs: the cost split gives the middle CTA an empty range
    run_path(T, (3, 16, 16), ((2, 1), (2, 4), (2, 4)), 1, 1, torch.float32)


def test_blend_many_frame_groups_use_the_count_split(T):
    # 70 frames: more (frame, band) groups than the blend's cost table holds
    run_path(T, (70, 12, 16), ((4, 3), (2, 2), (2, 4)), 1, 2, torch.bfloat16)


def test_compat_3d_triple_cover(T):
    run_path(T, (6, 21, 21), ((3, 2), (4, 8), (3, 8)), 1, 3, torch.float32, compat=True)


def test_empty_batch(T):
    p = T.plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    x = torch.empty((0, 8, 4, 16, 16), device="cuda")
    tiles = T.extract(p, x)
    assert tiles.numel() == 0
    assert T.blend(p, tiles, 0, 8).numel() == 0


# ----------------------------------------------------------------- window sum
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_window_sum_workloads(T, name):
    wl = WORKLOADS[name]
    p = T.plan(wl.dims, wl.tiling)
    dev, S = T.window_sum(p, want_sum=True)
    ref = O.window_sum(O.make_plan(wl.dims, wl.tiling))
    torch.cuda.synchronize()
    assert np.max(np.abs(_np64(S) - ref)) <= 1e-6
    assert abs(dev.item() - np.max(np.abs(ref - 1))) <= 1e-6
    assert dev.item() <= 4 * 2.0 ** -23


def test_window_sum_equals_blend_of_ones(T):
    dims, tiling = (6, 21, 21), ((3, 2), (4, 8), (3, 8))
    p = T.plan(dims, tiling, compat=True)
    _, S = T.window_sum(p, want_sum=True)
    ones = torch.ones(p.tiles_numel(1, 1), dtype=torch.float32, device="cuda")
    Y = T.blend(p, ones, 1, 1)
    assert torch.equal(Y[0, 0], S)           # same weights, products and order


@pytest.mark.parametrize("n", [2, 3, 4])
def test_window_sum_mold_table(T, n):
    p = T.plan((1, 1, 21), ((1, 0), (1, 0), (n, 8)), compat=True)
    dev, S = T.window_sum(p, want_sum=True)
    printed = {2: 1.000, 3: 1.074, 4: 1.161}[n]
    assert abs(S.max().item() - printed) <= 6e-4
    assert abs(dev.item() - (S.max().item() - 1.0)) <= 1e-7


# ----------------------------------------------------------------- positions
@pytest.mark.parametrize("name", ["tiny", "stage1", "fullres", "4k"])
@pytest.mark.parametrize("normalize", [True, False])
def test_positions_grid(T, name, normalize):
    wl = WORKLOADS[name]
    B = 2
    gen = inputs.grid_positions(B, *wl.dims)
    p = T.plan(wl.dims, wl.tiling)
    tp, off = T.positions(p, _dev(gen, torch.int32), normalize=normalize)
    ref_tp, ref_off = O.positions(O.make_plan(wl.dims, wl.tiling), gen, normalize=normalize)
    assert np.array_equal(off.cpu().numpy(), ref_off)
    assert np.array_equal(tp.cpu().numpy(), np.concatenate([x.reshape(-1) for x in ref_tp]))


def test_positions_random_intervals(T):
    dims, tiling = (5, 37, 53), ((2, 1), (3, 5), (4, 6))
    gen = inputs.random_positions(3, int(np.prod(dims)), seed=7)
    p = T.plan(dims, tiling)
    tp, off = T.positions(p, _dev(gen, torch.int32))
    ref_tp, ref_off = O.positions(O.make_plan(dims, tiling), gen)
    assert np.array_equal(off.cpu().numpy(), ref_off)
    for t in range(p.T):
        assert np.array_equal(T.tile_positions_view(p, tp, 3, t).cpu().numpy(), ref_tp[t])


# ----------------------------------------------------------------- conditioning
def check_cond(T, dims, tiling, gen, cond, normalize=True, compat=False):
    p = T.plan(dims, tiling, compat=compat)
    o = T.cond_select(p, _dev(gen, torch.int32), _dev(cond, torch.int32), normalize=normalize)
    ref = O.cond_select(O.make_plan(dims, tiling, compat=compat), gen, cond, normalize=normalize)
    torch.cuda.synchronize()
    B, M = cond.shape[0], cond.shape[2]
    assert np.array_equal(o["extent"].cpu().numpy(), ref.extent)
    assert np.array_equal(o["keep"].cpu().numpy(), ref.keep.astype(np.uint8))
    assert np.array_equal(o["count"].cpu().numpy(), ref.count)
    assert np.array_equal(o["weight"].cpu().numpy().view(np.uint32), ref.weight.view(np.uint32))
    kept, nk, tcp = o["kept_idx"].cpu().numpy(), o["num_kept"].cpu().numpy(), o["tile_cond_pos"].cpu().numpy()
    for t in range(p.T):
        for b in range(B):
            k = len(ref.kept[t][b])
            assert nk[t, b] == k
            assert np.array_equal(kept[t, b, :k], ref.kept[t][b]) and np.all(kept[t, b, k:] == -1)
            assert np.array_equal(tcp[t, b, :, :k, :], ref.tile_cond_pos[t][b]) and np.all(tcp[t, b, :, k:, :] == 0)
    return o, ref


@pytest.mark.parametrize("name", ["tiny", "stage1", "fullres", "4k"])
def test_cond_select_workloads(T, name):
    wl = WORKLOADS[name]
    gen = inputs.grid_positions(wl.B, *wl.dims)
    cond = inputs.cond_positions(wl.B, wl.num_cond, *wl.dims, n_negative=wl.num_cond_negative, seed=2)
    o, ref = check_cond(T, wl.dims, wl.tiling, gen, cond)
    neg = cond[:, 0, :, 0] < 0
    assert np.all(ref.count[neg] == WORKLOADS[name].tiling[0][0] * wl.tiling[1][0] * wl.tiling[2][0])


@pytest.mark.parametrize("M", [0, 1, 37, 1000, 3000])   # 3000: chunks over the cluster's CTAs
@pytest.mark.parametrize("normalize", [True, False])
def test_cond_select_sizes(T, M, normalize):
    dims, tiling = (5, 37, 53), ((2, 1), (3, 5), (4, 6))
    gen = inputs.grid_positions(2, *dims)
    cond = inputs.cond_positions(2, M, *dims, n_negative=M // 5, seed=3)
    check_cond(T, dims, tiling, gen, cond, normalize=normalize)


def test_cond_select_random_gen_positions(T):
    dims, tiling = (3, 10, 12), ((1, 0), (2, 3), (3, 3))
    gen = inputs.random_positions(2, int(np.prod(dims)), seed=4, lo=-100, hi=400)
    cond = inputs.random_positions(2, 300, seed=5, lo=-150, hi=450)
    check_cond(T, dims, tiling, gen, cond)


# ----------------------------------------------------------------- positions + conditioning in one launch
@pytest.mark.parametrize("case", ["4k", "4k_b3", "ragged", "random", "no_cond", "big_chunks"])
def test_tokens_matches_separate_calls_and_oracle(T, case):
    if case in ("4k", "4k_b3", "no_cond"):
        wl = WORKLOADS["4k"]
        dims, tiling, B = wl.dims, wl.tiling, 3 if case == "4k_b3" else 2
        gen = inputs.grid_positions(B, *dims)
        M = 0 if case == "no_cond" else wl.num_cond
        cond = inputs.cond_positions(B, M, *dims, n_negative=M // 4, seed=2)
    elif case == "ragged":
        dims, tiling, B = (5, 37, 53), ((2, 1), (3, 5), (4, 6)), 3
        gen = inputs.grid_positions(B, *dims)
        cond = inputs.cond_positions(B, 37, *dims, n_negative=7, seed=3)
    elif case == "random":
        dims, tiling, B = (3, 10, 12), ((1, 0), (2, 3), (3, 3)), 2
        gen = inputs.random_positions(B, int(np.prod(dims)), seed=4, lo=-100, hi=400)
        cond = inputs.random_positions(B, 300, seed=5, lo=-150, hi=450)
    else:   # tiles whose chunks exceed the per-thread register cache (read twice)
        dims, tiling, B = (8, 160, 160), ((1, 0), (2, 8), (2, 8)), 1
        gen = inputs.grid_positions(B, *dims)
        cond = inputs.cond_positions(B, 64, *dims, n_negative=8, seed=6)
    p = T.plan(dims, tiling)
    rp = O.make_plan(dims, tiling)
    o = T.tokens(p, _dev(gen, torch.int32), _dev(cond, torch.int32))
    tp, off = T.positions(p, _dev(gen, torch.int32))
    torch.cuda.synchronize()
    ref_tp, ref_off = O.positions(rp, gen)
    assert np.array_equal(o["offsets"].cpu().numpy(), ref_off)
    assert np.array_equal(o["tile_pos"].cpu().numpy(), np.concatenate([x.reshape(-1) for x in ref_tp]))
    assert torch.equal(o["tile_pos"], tp) and torch.equal(o["offsets"], off)
    M = cond.shape[2]
    if M:
        ref = O.cond_select(rp, gen, cond)
        assert np.array_equal(o["extent"].cpu().numpy(), ref.extent)
        assert np.array_equal(o["keep"].cpu().numpy(), ref.keep.astype(np.uint8))
        assert np.array_equal(o["count"].cpu().numpy(), ref.count)
        assert np.array_equal(o["weight"].cpu().numpy().view(np.uint32), ref.weight.view(np.uint32))
        sep = T.cond_select(p, _dev(gen, torch.int32), _dev(cond, torch.int32))
        for k in ("extent", "keep", "count", "weight", "kept_idx", "num_kept", "tile_cond_pos"):
            assert torch.equal(o[k], sep[k]), k
    assert T.device_error() == 0


# ----------------------------------------------------------------- window maximum without the per-element sums
@pytest.mark.parametrize("case", list(WORKLOADS) + ["mold3", "mold4", "triple", "ragged"])
def test_window_max_alone_equals_full_sum(T, case):
    if case in WORKLOADS:
        wl = WORKLOADS[case]
        dims, tiling, compat = wl.dims, wl.tiling, False
    else:
        dims, tiling, compat = {"mold3": ((1, 1, 21), ((1, 0), (1, 0), (3, 8)), True),
                                "mold4": ((1, 1, 21), ((1, 0), (1, 0), (4, 8)), True),
                                "triple": ((6, 21, 21), ((3, 2), (4, 8), (3, 8)), True),
                                "ragged": ((5, 37, 53), ((2, 1), (3, 5), (4, 6)), False)}[case]
    p = T.plan(dims, tiling, compat=compat)
    dev_full, S = T.window_sum(p, want_sum=True)
    full = dev_full.item()
    dev_alone, none = T.window_sum(p)             # no per-element output: the one-CTA path
    assert none is None
    assert dev_alone.item() == full               # bit-identical maximum
    assert abs(full - float(np.max(np.abs(_np64(S) - 1.0)))) == 0.0


# ----------------------------------------------------------------- conditioning combine
@pytest.mark.parametrize("case", ["4k", "ragged_f32", "ragged_bf16_to_f32", "many_tiles", "d_odd", "no_cond"])
def test_cond_combine(T, case):
    if case == "4k":
        wl = WORKLOADS["4k"]
        dims, tiling, B, M, D, dt, odt = wl.dims, wl.tiling, 1, wl.num_cond, 128, torch.bfloat16, torch.bfloat16
    elif case.startswith("ragged"):
        dims, tiling, B, M, D = (5, 37, 53), ((2, 1), (3, 5), (4, 6)), 2, 60, 33
        dt = torch.float32 if case == "ragged_f32" else torch.bfloat16
        odt = torch.float32
    elif case == "many_tiles":     # 64 tiles: two 32-lane slot passes per token
        dims, tiling, B, M, D, dt, odt = (12, 40, 40), ((4, 1), (4, 2), (4, 2)), 1, 90, 64, torch.float32, torch.bfloat16
    elif case == "d_odd":
        dims, tiling, B, M, D, dt, odt = (3, 10, 12), ((1, 0), (2, 3), (3, 3)), 2, 300, 7, torch.bfloat16, torch.bfloat16
    else:
        dims, tiling, B, M, D, dt, odt = (5, 37, 53), ((2, 1), (3, 5), (4, 6)), 1, 0, 16, torch.float32, torch.float32
    p = T.plan(dims, tiling)
    rp = O.make_plan(dims, tiling)
    gen = inputs.grid_positions(B, *dims)
    cond = inputs.cond_positions(B, M, *dims, n_negative=M // 5, seed=11)
    o = T.tokens(p, _dev(gen, torch.int32), _dev(cond, torch.int32))
    rng = np.random.default_rng(12)
    x = rng.standard_normal((p.T, B, M, D)).astype(np.float32)
    xd = _dev(x, dt)
    Y = T.cond_combine(p, xd, o["slot_of"], o["weight"], out_dtype=odt)
    torch.cuda.synchronize()
    assert Y.shape == (B, M, D) and Y.dtype == odt
    if M == 0:
        return
    sel = O.cond_select(rp, gen, cond)
    assert np.array_equal(o["slot_of"].cpu().numpy(), O.cond_slots(sel))
    ref = O.cond_combine(sel, _np64(xd))          # the same (rounded) inputs, float64 sums, weight 1/k
    Yn = _np64(Y)
    if odt == torch.float32:
        assert np.max(np.abs(Yn - ref)) <= 1e-5
    else:
        assert np.all(np.abs(Yn - ref) <= 8e-3 * np.abs(ref) + 1e-5)
    assert np.all(Yn[sel.count == 0] == 0.0)
    assert T.device_error() == 0
