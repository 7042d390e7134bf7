"""The sharded blend on one GPU: R slab blends (tdp_blend_slab, one per
rank of tdp_shard_plan) concatenated along H equal tdp_blend bit for bit,
and a slab reads only the tiles that meet its rows.

Source: "Tiled Data Parallelism (TDP)", What it is (tiles round robin over
ranks; the ranks' blends summed); the slab split is this library's reading.
The ranks here are emulated on one GPU by blending each rank's slab from a
buffer in which every tile the slab does not need is poisoned with NaN."""
import numpy as np
import pytest
import torch

from overlap_add_blending_gb300 import inputs, tdp
from overlap_add_blending_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

CASES = {
    "4k": (WORKLOADS["4k"].dims, WORKLOADS["4k"].tiling, False, 1, 16, torch.bfloat16, torch.bfloat16),
    "4k_f32_out": (WORKLOADS["4k"].dims, WORKLOADS["4k"].tiling, False, 1, 8, torch.bfloat16, torch.float32),
    "ragged": ((5, 37, 53), ((2, 1), (3, 5), (4, 6)), False, 2, 3, torch.float32, torch.float32),
    "triple": ((1, 21, 21), ((1, 0), (4, 8), (3, 8)), True, 1, 4, torch.float32, torch.bfloat16),
    "tiny": (WORKLOADS["tiny"].dims, WORKLOADS["tiny"].tiling, False, 1, 8, torch.float32, torch.float32),
}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch.device("cuda", 0)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("R", [1, 2, 3, 4, 7])
def test_slabs_reassemble_the_blend(dev, name, R):
    dims, tiling, compat, B, C, tin, tout = CASES[name]
    p = tdp.plan(dims, tiling, compat)
    n = p.tiles_numel(B, C)
    tiles = torch.from_numpy(np.random.default_rng(5).standard_normal(n).astype(np.float32)).to(tin).to(dev)
    full = tdp.blend(p, tiles, B, C, out_dtype=tout)
    slabs = []
    for r in range(R):
        sh = tdp.shard_plan(p, R, r)
        mine = tiles.clone()
        for t in range(p.T):
            if t not in sh.needed:   # what this rank never receives
                off = p.tile_offset(t, B, C)
                (_, size) = p.box(t)
                mine[off:off + B * C * size[0] * size[1] * size[2]] = float("nan")
        slabs.append(tdp.blend_slab(p, mine, B, C, sh.row0, sh.row1, out_dtype=tout))
    torch.cuda.synchronize()
    got = torch.cat(slabs, dim=3)
    assert got.shape == full.shape
    assert torch.equal(got, full), "the slabs differ from the single-GPU blend"
    assert tdp.device_error() == 0


def test_slab_identity_round_trip_at_4k(dev):
    wl = WORKLOADS["4k"]
    p = tdp.plan(wl.dims, wl.tiling)
    X = torch.from_numpy(inputs.latent((1, 32) + wl.dims, seed=0)).to(torch.bfloat16).to(dev)
    tiles = tdp.extract(p, X)
    sh = tdp.shard_plan(p, 4, 2)
    slab = tdp.blend_slab(p, tiles, 1, 32, sh.row0, sh.row1)
    torch.cuda.synchronize()
    assert torch.equal(slab, X[:, :, :, sh.row0:sh.row1, :])


def test_slab_argument_checks(dev):
    import ctypes
    p = tdp.plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    tiles = torch.zeros(p.tiles_numel(1, 2), device=dev)
    out = torch.empty((1, 2, 4, 16, 16), device=dev)
    for r0, r1 in ((-1, 3), (5, 4), (0, 17)):
        st = tdp._lib.tdp_blend_slab(ctypes.byref(p), 1, 2, 0, tiles.data_ptr(), r0, r1, 0, out.data_ptr(), None)
        assert st == 1, (r0, r1, st)   # TDP_ERR_INVALID_ARG, before any launch
    empty = tdp.blend_slab(p, tiles, 1, 2, 3, 3)
    assert empty.shape == (1, 2, 4, 0, 16)
