"""tdp_extract_and_tokens_no_alloc (the library's own scratch) against
tdp_extract_and_tokens (a caller's workspace): two calls in a row on one
stream, every output equal bit for bit.  The file sorts last, so in a full
run it also runs after every other test; it runs alone as well."""
import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("B", [1, 3])
def test_no_alloc_matches_workspace_call_twice(T, B):
    wl = WORKLOADS["4k"]
    p = T.plan(wl.dims, wl.tiling)
    C = 16
    M = wl.num_cond
    g = _dev(inputs.grid_positions(B, *wl.dims), torch.int32)
    c = _dev(inputs.cond_positions(B, M, *wl.dims, n_negative=M // 4, seed=2), torch.int32)
    for call in range(2):
        X = _dev(inputs.latent((B, C) + wl.dims, seed=10 + call), torch.bfloat16)
        ref_tiles, ref, ref_dev = T.extract_and_tokens(p, X, g, c)
        tiles = torch.full_like(ref_tiles, 7)
        tok = T.token_outputs(p, B, M, X.device)
        for v in tok.values():
            v.fill_(-5)
        dev = torch.full((4,), -1.0, dtype=torch.float32, device=X.device)
        T.extract_and_tokens_no_alloc(p, X, g, c, tiles, tok, max_dev=dev)
        torch.cuda.synchronize()
        assert T.device_error() == 0
        assert torch.equal(tiles, ref_tiles)
        for k, v in ref.items():
            assert torch.equal(tok[k], v), (call, k)
        assert dev[0].item() == ref_dev.item()


def test_no_alloc_rejects_oversize(T):
    import ctypes as Cty
    wl = WORKLOADS["4k"]
    p = T.plan(wl.dims, wl.tiling)
    B = 200   # 6400 pairs: partials beyond the 64 KiB scratch
    assert T.extract_and_tokens_workspace(p, B) > 64 * 1024
    st = T._lib.tdp_extract_and_tokens_no_alloc(Cty.byref(p), B, 0, 1, None, None, 16, 1, None, None, 0, None,
                                                None, None, None, None, None, None, None, None, None, None)
    assert st == 6   # TDP_ERR_UNSUPPORTED
