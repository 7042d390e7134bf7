"""Parity of the token-major extract / blend (C ABI) with the CPU oracle.

Token-major tiles are bit copies of the latent (exact match); blended floats
must be within max-abs 1e-5 (fp32 output) or 8e-3 relative (bf16 output) of
the oracle's float64 sums, as for the channel-first path."""
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


def _np64(t):
    return t.detach().cpu().double().numpy()


def check_blend(Y, ref, ref_abs, out_dtype):
    Y = _np64(Y)
    if out_dtype == torch.float32:
        err = np.max(np.abs(Y - ref)) if Y.size else 0.0
        assert err <= 1e-5, err
    else:
        bound = 8e-3 * np.abs(ref) + 1e-5 * ref_abs + 1e-30
        bad = np.abs(Y - ref) > bound
        assert not bad.any(), (np.abs(Y - ref)[bad][:5], ref[bad][:5])


def affine_tokens(T, p, tok, B, C, a, b):
    """The per-tile op between extract and blend (the caller's work): a_t*x + b_t."""
    out = torch.empty_like(tok)
    for t in range(p.T):
        _, size = p.box(t)
        n = B * C * size[0] * size[1] * size[2]
        o = p.tile_offset(t, B, C)
        out[o:o + n] = (tok[o:o + n].float() * float(a[t]) + float(b[t])).to(tok.dtype)
    return out


def run_tokens(T, dims, tiling, B, C, dtype, op="affine", compat=False, out_dtype=None, seed=0):
    p = T.plan(dims, tiling, compat=compat)
    rp = O.make_plan(dims, tiling, compat=compat)
    X = torch.from_numpy(inputs.latent((B, C) + tuple(dims), seed=seed)).to(dtype).cuda()
    tok = T.extract_tokens(p, X)
    want = O.pack(O.extract_tokens(rp, _np64(X)))
    assert torch.equal(tok.cpu(), torch.from_numpy(want).to(dtype)), "extract_tokens mismatch"
    if op == "affine":
        a, b = inputs.affine_params(p.T, seed=1)
        tok = affine_tokens(T, p, tok, B, C, a, b)
    odt = out_dtype or dtype
    Y = T.blend_tokens(p, tok, B, C, out_dtype=odt)
    torch.cuda.synchronize()
    tl = O.unpack_tokens(rp, B, C, _np64(tok))
    check_blend(Y, O.blend_tokens(rp, tl), O.blend_tokens(rp, [np.abs(x) for x in tl]), odt)
    assert T.device_error() == 0
    return p, X, tok, Y


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("op", ["identity", "affine"])
def test_token_major_workloads(T, name, op):
    wl = WORKLOADS[name]
    p, X, tok, Y = run_tokens(T, wl.dims, wl.tiling, wl.B, wl.C, TORCH_DT[wl.dtype], op=op)
    if op == "identity":
        if wl.dtype == "bf16":
            assert torch.equal(Y, X)
        else:
            assert (Y - X).abs().max().item() <= 1e-5


def test_token_major_4k_fp32_output(T):
    wl = WORKLOADS["4k"]
    run_tokens(T, wl.dims, wl.tiling, wl.B, wl.C, torch.bfloat16, out_dtype=torch.float32)


def test_token_major_4k_two_batches(T):
    wl = WORKLOADS["4k"]
    run_tokens(T, wl.dims, wl.tiling, 2, 64, torch.bfloat16, seed=5)


def test_tokens_are_channel_first_tiles_transposed(T):
    """The two extract layouts hold the same values, tile by tile."""
    wl = WORKLOADS["fullres"]
    p = T.plan(wl.dims, wl.tiling)
    B, C = 2, wl.C
    X = torch.from_numpy(inputs.latent((B, C) + wl.dims, seed=3)).to(torch.bfloat16).cuda()
    tiles, tok = T.extract(p, X), T.extract_tokens(p, X)
    for t in range(p.T):
        _, size = p.box(t)
        n_t = size[0] * size[1] * size[2]
        o = p.tile_offset(t, B, C)
        cf = tiles[o:o + B * C * n_t].view(B, C, n_t)
        assert torch.equal(tok[o:o + B * C * n_t].view(B, n_t, C), cf.transpose(1, 2))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_token_major_ragged(T, dtype):
    # remainders on every axis, odd widths, two batches, 16-byte tokens
    run_tokens(T, (5, 37, 53), ((2, 1), (3, 5), (4, 6)), 2, 8, dtype)


@pytest.mark.parametrize("C", [16, 40, 136])
def test_token_major_channel_counts(T, C):
    # 2, 5 and 17 sixteen-byte chunks per bf16 token (swizzle widths 2, 4, 8)
    run_tokens(T, (3, 11, 29), ((2, 1), (2, 3), (3, 4)), 1, C, torch.bfloat16)


def test_token_major_many_column_blocks(T):
    # fp32 C=128: 32 chunks per token, 32 columns per unit -> 10 column blocks
    run_tokens(T, (2, 3, 300), ((1, 0), (1, 0), (4, 20)), 1, 128, torch.float32)


def test_token_major_wide_rows(T):
    run_tokens(T, (2, 5, 1500), ((1, 0), (2, 1), (3, 16)), 1, 8, torch.float32)


@pytest.mark.parametrize("in_dt,out_dt", [(torch.bfloat16, torch.float32), (torch.float32, torch.bfloat16)])
def test_token_major_mixed_dtypes(T, in_dt, out_dt):
    run_tokens(T, (4, 16, 24), ((1, 0), (2, 4), (2, 6)), 1, 16, in_dt, out_dtype=out_dt)


def test_token_major_compat_triple_cover(T):
    run_tokens(T, (6, 21, 21), ((3, 2), (4, 8), (3, 8)), 1, 4, torch.float32, compat=True)


def test_token_major_four_column_tiles_cover_a_column(T):
    # (21, 4, 8): column 10 lies in all four column tiles (past the two kept per item)
    run_tokens(T, (1, 2, 21), ((1, 0), (1, 0), (4, 8)), 1, 16, torch.float32, compat=True)


def test_token_major_single_tile_and_hard_cut(T):
    p, X, tok, Y = run_tokens(T, (3, 9, 10), ((1, 0), (1, 0), (1, 0)), 2, 4, torch.float32, op="identity")
    assert torch.equal(X, Y)
    assert torch.equal(tok.view(2, 270, 4), X.view(2, 4, 270).transpose(1, 2))
    p, X, tok, Y = run_tokens(T, (3, 10, 14), ((3, 0), (2, 0), (4, 0)), 1, 4, torch.float32, op="identity")
    assert torch.equal(X, Y)


def test_token_major_rejects_unaligned_tokens_and_empty_batch(T):
    p = T.plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    X = torch.zeros((1, 3, 4, 16, 16), dtype=torch.bfloat16, device="cuda")     # 6-byte tokens
    with pytest.raises(T.TdpError) as e:
        T.extract_tokens(p, X)
    assert e.value.status == 6
    with pytest.raises(T.TdpError):
        T.blend_tokens(p, torch.zeros(p.tiles_numel(1, 3), dtype=torch.bfloat16, device="cuda"), 1, 3)
    x = torch.empty((0, 8, 4, 16, 16), device="cuda")
    tok = T.extract_tokens(p, x)
    assert tok.numel() == 0
    assert T.blend_tokens(p, tok, 0, 8).numel() == 0
