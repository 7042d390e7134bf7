"""Parity of tdp_extract_and_tokens (the tiles, the token steps and the
window maximum in two launches) with the CPU oracle and with the separate
calls, through the C ABI.

The call reduces the partial extents of every (tile, batch) pair's token
chunks inside the streaming extract launch and finishes the token steps in
a second launch; every output must equal the oracle's (integers and the
IEEE 1/count weights bit for bit) and the separate calls' bit for bit."""
import numpy as np
import pytest
import torch

from oracle import tdp_oracle as O
from overlap_add_blending_gb300 import inputs
from overlap_add_blending_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from overlap_add_blending_gb300 import tdp
    return tdp


def _dev(x_np, dtype):
    return torch.from_numpy(np.ascontiguousarray(x_np)).to(dtype).cuda()


def _case(name):
    """(dims, tiling, B, C, dtype, gen, cond, fused): fused says whether the
    streaming kernels take the plan (one launch per call)."""
    wl = WORKLOADS["4k"]
    if name == "4k":              # the bench workload: 32 token jobs over the grid
        dims, tiling, B, C, dt, M = wl.dims, wl.tiling, 1, 128, torch.bfloat16, wl.num_cond
    elif name == "4k_b3":         # 96 token jobs
        dims, tiling, B, C, dt, M = wl.dims, wl.tiling, 3, 16, torch.bfloat16, wl.num_cond
    elif name == "4k_b6":         # 192 token jobs: some CTAs take two
        dims, tiling, B, C, dt, M = wl.dims, wl.tiling, 6, 4, torch.bfloat16, 40
    elif name == "random_f32":    # random intervals (negative starts, empty overlaps) on an fp32 latent
        dims, tiling, B, C, dt, M = (3, 10, 12), ((1, 0), (2, 3), (3, 3)), 2, 8, torch.float32, 300
    elif name == "many_cond":     # more conditioning tokens than a CTA's compute threads: several scan rounds
        dims, tiling, B, C, dt, M = (4, 24, 40), ((2, 1), (2, 4), (2, 8)), 2, 16, torch.bfloat16, 2000
    elif name == "no_cond":
        dims, tiling, B, C, dt, M = wl.dims, wl.tiling, 1, 32, torch.bfloat16, 0
    elif name == "ragged":        # W * 2 bytes not a multiple of 16: the separate kernels in turn
        dims, tiling, B, C, dt, M = (5, 37, 53), ((2, 1), (3, 5), (4, 6)), 2, 8, torch.bfloat16, 37
    else:
        raise KeyError(name)
    if name == "random_f32":
        gen = inputs.random_positions(B, int(np.prod(dims)), seed=4, lo=-100, hi=400)
        cond = inputs.random_positions(B, M, seed=5, lo=-150, hi=450)
    else:
        gen = inputs.grid_positions(B, *dims)
        cond = inputs.cond_positions(B, M, *dims, n_negative=M // 4, seed=2)
    return dims, tiling, B, C, dt, gen, cond, name != "ragged"


CASES = ["4k", "4k_b3", "4k_b6", "random_f32", "many_cond", "no_cond", "ragged"]


@pytest.mark.parametrize("name", CASES)
def test_extract_and_tokens(T, name):
    dims, tiling, B, C, dt, gen, cond, fused = _case(name)
    p = T.plan(dims, tiling)
    rp = O.make_plan(dims, tiling)
    geo, _ = T.launch_geometry(p, B, C, False, dt, dt, torch.cuda.get_device_properties(0).multi_processor_count)
    assert bool(geo["streaming"]) == fused
    X = inputs.latent((B, C) + tuple(dims), seed=1)
    Xd = _dev(X, dt)
    g, c = _dev(gen, torch.int32), _dev(cond, torch.int32)
    M = cond.shape[2]
    tok = T.token_outputs(p, B, M, Xd.device)
    for v in tok.values():
        v.fill_(-3)   # stale contents must not leak into the results
    ws = torch.full((T.extract_and_tokens_workspace(p, B) + 16,), 0x5A, dtype=torch.uint8, device=Xd.device)
    tiles, tok, dev = T.extract_and_tokens(p, Xd, g, c, tok=tok, workspace=ws)
    torch.cuda.synchronize()
    assert T.device_error() == 0
    # the separate calls
    assert torch.equal(tiles, T.extract(p, Xd))
    sep = T.tokens(p, g, c)
    sep_dev, _ = T.window_sum(p)
    torch.cuda.synchronize()
    assert dev.item() == sep_dev.item()
    for k in ("tile_pos", "offsets"):
        assert torch.equal(tok[k], sep[k]), k
    if M:
        for k in ("extent", "keep", "count", "weight", "kept_idx", "num_kept", "tile_cond_pos", "slot_of"):
            assert torch.equal(tok[k], sep[k]), k
    # the oracle
    ref_tiles = O.pack(O.extract(rp, np.asarray(Xd.float().cpu().numpy(), dtype=np.float64)))
    assert np.array_equal(tiles.float().cpu().numpy().astype(np.float64), ref_tiles)
    ref_tp, ref_off = O.positions(rp, gen)
    assert np.array_equal(tok["offsets"].cpu().numpy(), ref_off)
    assert np.array_equal(tok["tile_pos"].cpu().numpy(), np.concatenate([x.reshape(-1) for x in ref_tp]))
    assert abs(dev.item() - O.max_abs_deviation(rp)) <= 1e-6
    if M:
        ref = O.cond_select(rp, gen, cond)
        assert np.array_equal(tok["extent"].cpu().numpy(), ref.extent)
        assert np.array_equal(tok["keep"].cpu().numpy(), ref.keep.astype(np.uint8))
        assert np.array_equal(tok["count"].cpu().numpy(), ref.count)
        assert np.array_equal(tok["weight"].cpu().numpy().view(np.uint32), ref.weight.view(np.uint32))
        kept, nk, tcp = tok["kept_idx"].cpu().numpy(), tok["num_kept"].cpu().numpy(), tok["tile_cond_pos"].cpu().numpy()
        for t in range(p.T):
            for b in range(B):
                k = len(ref.kept[t][b])
                assert nk[t, b] == k
                assert np.array_equal(kept[t, b, :k], ref.kept[t][b]) and np.all(kept[t, b, k:] == -1)
                assert np.array_equal(tcp[t, b, :, :k, :], ref.tile_cond_pos[t][b]) and np.all(tcp[t, b, :, k:, :] == 0)
        assert np.array_equal(tok["slot_of"].cpu().numpy(), O.cond_slots(ref))


@pytest.mark.parametrize("name", ["4k", "random_f32"])
def test_step_round_trip_and_partial_outputs(T, name):
    """Two calls in a row on one stream with their blends, the second without
    kept lists, positions or window maximum and with no workspace (the
    separate kernels): the same tiles, extents, keep flags, counts and
    weights, and the bf16 identity round trip is exact."""
    dims, tiling, B, C, dt, gen, cond, _ = _case(name)
    p = T.plan(dims, tiling)
    g, c = _dev(gen, torch.int32), _dev(cond, torch.int32)
    Xd = _dev(inputs.latent((B, C) + tuple(dims), seed=3), dt)
    M = cond.shape[2]
    tiles1, tok1, _ = T.extract_and_tokens(p, Xd, g, c)
    Y1 = T.blend(p, tiles1, B, C)
    tok2 = {k: v for k, v in T.token_outputs(p, B, M, Xd.device).items()
            if k in ("extent", "keep", "count", "weight")}
    tiles2, _, none = T.extract_and_tokens(p, Xd, g, c, tok=tok2, window_max=False,
                                           workspace=torch.empty(16, dtype=torch.uint8, device=Xd.device))
    Y2 = T.blend(p, tiles2, B, C)
    torch.cuda.synchronize()
    assert none is None and T.device_error() == 0
    assert torch.equal(tiles1, tiles2) and torch.equal(Y1, Y2)
    for k in ("extent", "keep", "count", "weight"):
        assert torch.equal(tok1[k], tok2[k]), k
    if dt == torch.bfloat16:
        assert torch.equal(Y1, Xd)  # identity per-tile op: the bf16 round trip is exact


def test_workspace_size(T):
    wl = WORKLOADS["4k"]
    p = T.plan(wl.dims, wl.tiling)
    # per pair, 6 int32 for each of max(3 chunks of at most 3072 tokens of an
    # 8073-token tile, 256 CTAs // pairs) chunks, then one int32 per batch,
    # rounded up to 16 bytes
    r16 = lambda n: -(-n // 16) * 16
    assert T.extract_and_tokens_workspace(p, 1) == r16((32 * 8 * 6 + 1) * 4)
    assert T.extract_and_tokens_workspace(p, 3) == r16((96 * 3 * 6 + 3) * 4)
    assert T.extract_and_tokens_workspace(p, 0) == 0


def test_fused_argument_checks(T):
    import ctypes as C
    p = T.plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    L = T._lib

    def call(B, Cc, latent, tiles, gen, M, cond, extent, keep, count, weight, dev=None, ws=None, wsb=0):
        return L.tdp_extract_and_tokens(C.byref(p), B, Cc, 1, latent, tiles, gen, 1, None, None, M, cond, extent,
                                        keep, count, weight, None, None, None, None, dev, ws, wsb, None)
    assert call(1, 0, None, None, 16, 5, 16, 16, None, 16, 16) == 1      # M > 0 without keep
    assert call(1, 0, None, None, 16, 5, 16, 16, 16, None, 16) == 1      # M > 0 without count
    assert call(1, 2, 16, None, 16, 0, None, None, None, None, None) == 1   # a latent without its tiles
    assert call(1, 0, None, None, None, 0, None, None, None, None, None) == 1  # no generated positions
    assert call(1, 0, None, None, 20, 0, None, None, None, None, None) == 4    # misaligned pointer
    assert call(1, 0, None, None, 16, 0, None, None, None, None, None, dev=24) == 4
    assert call(1, 0, None, None, 16, 0, None, None, None, None, None, ws=16, wsb=-1) == 1
    with pytest.raises(ValueError):
        T.extract_and_tokens_workspace(p, -1)
