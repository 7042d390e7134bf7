"""CPU models of the kernels' index arithmetic (no GPU code runs here).

Each model restates, in NumPy over a CTA's 256 threads, how one kernel maps
threads to data: the units a CTA walks, the global and shared addresses of
every load and store, and the shared-memory swizzles.  The tests check that
every access stays inside its buffer, that every output element (and every
shared slot) is written exactly once, that the walks and splits cover every
unit exactly once, and that the modelled data movement reproduces the
oracle.  They guard the layouts of the token-major kernels and the fast
blend's cost split; the kernels themselves are checked against the oracle
by the GPU tests.
"""
import numpy as np
import pytest

from oracle import tdp_oracle as O

THREADS, ITEMS = 256, 4
CHUNKS = THREADS * ITEMS


@pytest.fixture(scope="module")
def T():
    from overlap_add_blending_gb300 import build
    build.build()
    from overlap_add_blending_gb300 import tdp
    return tdp


# ----------------------------------------------------------------- shared helpers
def mask_of(chunks):
    m = 1
    while m * 2 <= min(chunks, 8):
        m *= 2
    return m - 1


def swz(j, x, m, n):
    return np.where((j | m) < n, j ^ (x & m), j)


def swzf(j, x, m, n):
    f = (((x & 1) << 2) | ((x >> 1) & 3)) if m == 7 else (x & m)
    return np.where((j | m) < n, j ^ f, j)


def cover(p, d, x):
    n = p.num_tiles[d]
    h = min(x // p.stride[d], n - 1)
    lo = h
    while lo > 0 and p.end[d][lo - 1] > x:
        lo -= 1
    return lo, h


def size(p, d, i):
    return p.end[d][i] - p.start[d][i]


def prefix_volume(p, i_f, i_h, i_w):
    SH, SW = p.prefix[1][p.num_tiles[1]], p.prefix[2][p.num_tiles[2]]
    return p.prefix[0][i_f] * SH * SW + size(p, 0, i_f) * (p.prefix[1][i_h] * SW + size(p, 1, i_h) * p.prefix[2][i_w])


def tm_args(p, B, C, esz, blend):
    J = C * esz // 16
    ipt = 4 if J % 4 == 0 else (2 if J % 2 == 0 else 1)
    lpt = J // ipt
    W = p.dims[2]
    xb_max = THREADS // lpt if blend else CHUNKS // J
    nxb = -(-W // xb_max)
    xb = -(-W // nxb)
    return dict(J=J, jf=C // 4, pm=mask_of(J), pfm=mask_of(C // 4), ipt=ipt, lpt=lpt, xb=xb, nxb=nxb,
                units=B * p.dims[0] * p.dims[1] * nxb)


def unit_of(p, a, u):
    xb = u % a["nxb"]
    q = u // a["nxb"]
    h = q % p.dims[1]
    q //= p.dims[1]
    f, b = q % p.dims[0], q // p.dims[0]
    x0 = xb * a["xb"]
    return b, f, h, x0, min(a["xb"], p.dims[2] - x0)


def walked_units(p, a, G):
    """Units of every CTA by the kernels' mixed-radix walk with stride G."""
    radix = [a["nxb"], p.dims[1], p.dims[0]]

    def digits(u):
        xb = u % a["nxb"]
        u //= a["nxb"]
        h = u % p.dims[1]
        u //= p.dims[1]
        return [xb, h, u % p.dims[0], u // p.dims[0]]

    seen = []
    for cta in range(G):
        u, w, st = cta, digits(cta), digits(G)
        while u < a["units"]:
            assert ((w[3] * p.dims[0] + w[2]) * p.dims[1] + w[1]) * a["nxb"] + w[0] == u
            seen.append(u)
            c = 0
            for d in range(3):
                w[d] += st[d] + c
                c = int(w[d] >= radix[d])
                if c:
                    w[d] -= radix[d]
            w[3] += st[3] + c
            u += G
    return seen


# ----------------------------------------------------------------- token-major extract
def model_extract_tokens(p, B, C, esz, X):
    a = tm_args(p, B, C, esz, blend=False)
    J, VEC = a["J"], 16 // esz
    F, H, W = p.dims
    fhw = F * H * W
    pair = W % 2 == 0 and a["xb"] % 2 == 0
    Xf = X.reshape(-1)
    total = p.tiles_numel(B, C) * esz // 16
    out = np.full((total, VEC), np.nan)
    written = np.zeros(total, np.int64)
    tid = np.arange(THREADS)

    def sw(j, x):
        return swz(j, (x >> 1) if pair else x, a["pm"], J)

    for u in range(a["units"]):
        b, f, h, x0, xbu = unit_of(p, a, u)
        row = (b * C * F + f) * H * W + h * W + x0
        smem = np.full((CHUNKS, VEC), np.nan)
        count = np.zeros(CHUNKS, np.int64)
        ncol = xbu // 2 if pair else xbu
        x, j = tid % ncol, tid // ncol
        for _ in range(ITEMS // 2 if pair else ITEMS):
            ok = j < J
            for col in ([2 * x, 2 * x + 1] if pair else [x]):
                idx = np.stack([row + (j * VEC + e) * fhw + col for e in range(VEC)], 1)
                assert np.all((idx[ok] >= 0) & (idx[ok] < Xf.size))
                slot = col * J + sw(j, col)
                assert np.all((slot[ok] >= 0) & (slot[ok] < CHUNKS))
                smem[slot[ok]] = Xf[idx[ok]]
                np.add.at(count, slot[ok], 1)
            x, j = x + THREADS % ncol, j + THREADS // ncol
            wrap = x >= ncol
            x, j = np.where(wrap, x - ncol, x), np.where(wrap, j + 1, j)
        xs, js = np.meshgrid(np.arange(xbu), np.arange(J), indexing="ij")
        assert np.all(count[(xs * J + sw(js, xs)).reshape(-1)] == 1) and count.sum() == xbu * J
        flo, fhi = cover(p, 0, f)
        hlo, hhi = cover(p, 1, h)
        wlo, whi = cover(p, 2, x0)[0], cover(p, 2, x0 + xbu - 1)[1]
        for i_f in range(flo, fhi + 1):
            for i_h in range(hlo, hhi + 1):
                for i_w in range(wlo, whi + 1):
                    w0 = p.start[2][i_w]
                    sb = min(p.end[2][i_w], x0 + xbu)
                    base = (B * prefix_volume(p, i_f, i_h, i_w)
                            + ((b * size(p, 0, i_f) + f - p.start[0][i_f]) * size(p, 1, i_h) + h - p.start[1][i_h])
                            * size(p, 2, i_w) - w0)
                    xx, jj = max(w0, x0) + tid // J, tid % J
                    while True:
                        act = xx < sb
                        if not act.any():
                            break
                        xl = xx - x0
                        slot = xl * J + sw(jj, xl)
                        d = (base + xx) * J + jj
                        assert np.all(count[slot[act]] == 1)
                        assert np.all((d[act] >= 0) & (d[act] < total))
                        out[d[act]] = smem[slot[act]]
                        np.add.at(written, d[act], 1)
                        xx, jj = xx + THREADS // J, jj + THREADS % J
                        wr = jj >= J
                        jj, xx = np.where(wr, jj - J, jj), np.where(wr, xx + 1, xx)
    assert np.all(written == 1)
    return out.reshape(-1)


# ----------------------------------------------------------------- token-major blend
def model_blend_tokens(p, B, C, esz, tok_flat):
    a = tm_args(p, B, C, esz, blend=True)
    J, VEC, jf, ipt, lpt = a["J"], 16 // esz, a["jf"], a["ipt"], a["lpt"]
    FCH = VEC // 4
    F, H, W = p.dims
    fhw = F * H * W
    chunks = tok_flat.reshape(-1, VEC)
    out = np.full(B * C * fhw, np.nan)
    written = np.zeros(B * C * fhw, np.int64)
    tid = np.arange(THREADS)
    xcol, lit = tid // lpt, tid % lpt
    ivs = [[(p.start[d][i], p.end[d][i]) for i in range(p.num_tiles[d])] for d in range(3)]
    for u in range(a["units"]):
        b, f, h, x0, xbu = unit_of(p, a, u)
        acc = np.zeros((THREADS, ipt, VEC))
        for i_f in range(cover(p, 0, f)[0], cover(p, 0, f)[1] + 1):
            wf = O.ramp_1d(ivs[0], p.overlap[0], i_f)[f - p.start[0][i_f]]
            for i_h in range(cover(p, 1, h)[0], cover(p, 1, h)[1] + 1):
                wh = O.ramp_1d(ivs[1], p.overlap[1], i_h)[h - p.start[1][i_h]]
                for t_ in np.nonzero(xcol < xbu)[0]:
                    w = x0 + xcol[t_]
                    for i_w in range(cover(p, 2, w)[0], cover(p, 2, w)[1] + 1):
                        tok = (B * prefix_volume(p, i_f, i_h, i_w)
                               + ((b * size(p, 0, i_f) + f - p.start[0][i_f]) * size(p, 1, i_h) + h - p.start[1][i_h])
                               * size(p, 2, i_w) + w - p.start[2][i_w])
                        ww = O.ramp_1d(ivs[2], p.overlap[2], i_w)[w - p.start[2][i_w]]
                        for r in range(ipt):
                            ci = tok * J + lit[t_] + r * lpt
                            assert 0 <= ci < len(chunks)
                            acc[t_, r] += wf * wh * ww * chunks[ci]
        smem = np.full((2 * CHUNKS, 4), np.nan)
        count = np.zeros(2 * CHUNKS, np.int64)
        for t_ in np.nonzero(xcol < xbu)[0]:
            for r in range(ipt):
                for c in range(FCH):
                    si = xcol[t_] * jf + int(swzf(np.array(c * J + lit[t_] + r * lpt), np.array(xcol[t_]),
                                                  a["pfm"], jf))
                    assert 0 <= si < 2 * CHUNKS
                    smem[si] = acc[t_, r, 4 * c:4 * c + 4]
                    count[si] += 1
        assert count.sum() == xbu * jf and np.all(count <= 1)
        row = (b * C * F + f) * H * W + h * W + x0
        xt = min(xbu, THREADS)
        for t_ in range(THREADS):
            if t_ // xt >= THREADS // xt:
                continue
            for x in range(t_ % xt, xbu, xt):
                for qc in range(t_ // xt, jf, THREADS // xt):
                    slot = (qc & 1) * J + (qc >> 1) if FCH == 2 else qc
                    si = x * jf + int(swzf(np.array(slot), np.array(x), a["pfm"], jf))
                    assert count[si] == 1
                    for e in range(4):
                        o = row + (4 * qc + e) * fhw + x
                        out[o] = smem[si, e]
                        written[o] += 1
    assert np.all(written == 1)
    return out.reshape((B, C) + tuple(p.dims))


CASES = [
    ((4, 16, 16), ((1, 0), (2, 4), (2, 4)), 1, 8, 4, False),       # tiny fp32, J = 2, column pairs
    ((16, 16, 24), ((1, 0), (2, 4), (2, 6)), 1, 128, 2, False),    # stage-1 bf16, J = 16
    ((3, 7, 9), ((2, 1), (2, 2), (3, 2)), 2, 40, 2, True),         # J = 5, odd W, compat
    ((5, 9, 11), ((2, 1), (3, 2), (2, 3)), 2, 8, 2, False),        # J = 1
    ((2, 3, 300), ((1, 0), (1, 0), (4, 20)), 1, 128, 4, False),    # fp32 J = 32: 10 column blocks
    ((1, 2, 21), ((1, 0), (1, 0), (4, 8)), 1, 16, 2, True),        # four column tiles over one column
    ((3, 11, 29), ((2, 1), (2, 3), (3, 4)), 1, 136, 2, False),     # J = 17
]


@pytest.mark.parametrize("dims,tiling,B,C,esz,compat", CASES)
def test_token_major_models(T, dims, tiling, B, C, esz, compat):
    p = T.plan(dims, tiling, compat=compat)
    rp = O.make_plan(dims, tiling, compat=compat)
    rng = np.random.default_rng(0)
    X = rng.standard_normal((B, C) + tuple(dims))
    assert np.array_equal(model_extract_tokens(p, B, C, esz, X), O.pack(O.extract_tokens(rp, X)))
    tok = rng.standard_normal(p.tiles_numel(B, C))
    want = O.blend_tokens(rp, O.unpack_tokens(rp, B, C, tok))
    assert np.max(np.abs(model_blend_tokens(p, B, C, esz, tok) - want)) < 1e-12
    for blend in (False, True):
        a = tm_args(p, B, C, esz, blend)
        for G in (1, 7, 304, 456, 760, a["units"]):   # 456 / 760: the 4K launches' grids (3 / 5 CTAs per SM)
            assert sorted(walked_units(p, a, min(G, a["units"]))) == list(range(a["units"]))


def test_token_major_models_random(T):
    """Seeded random plans and channel counts (C * element size a multiple
    of 16 bytes): the token-major extract and blend models equal the oracle,
    and the unit walk covers every unit once for several grids."""
    rng = np.random.default_rng(5150)
    for _ in range(12):
        dims = (int(rng.integers(1, 5)), int(rng.integers(2, 20)), int(rng.integers(2, 40)))
        tiling = []
        for d in dims:
            n = int(rng.integers(1, min(4, d) + 1))
            tiling.append((n, int(rng.integers(0, d // (n + 1) + 1)) if n > 1 else 0))
        esz = int(rng.choice([2, 4]))
        C = (16 // esz) * int(rng.integers(1, 6))
        B = int(rng.integers(1, 3))
        p = T.plan(dims, tuple(tiling))
        rp = O.make_plan(dims, tuple(tiling))
        X = rng.standard_normal((B, C) + dims)
        assert np.array_equal(model_extract_tokens(p, B, C, esz, X), O.pack(O.extract_tokens(rp, X))), (dims, tiling)
        tok = rng.standard_normal(p.tiles_numel(B, C))
        want = O.blend_tokens(rp, O.unpack_tokens(rp, B, C, tok))
        assert np.max(np.abs(model_blend_tokens(p, B, C, esz, tok) - want)) < 1e-12, (dims, tiling)
        for blend in (False, True):
            a = tm_args(p, B, C, esz, blend)
            for G in (1, 5, 456, 760):
                assert sorted(walked_units(p, a, min(G, a["units"]))) == list(range(a["units"]))


def test_token_major_swizzles_are_conflict_free_on_the_4k_layout():
    """bf16, C = 128: 16 sixteen-byte chunks per token, 60 columns per unit."""
    J, jf, m, xbu = 16, 32, 7, 60
    tid = np.arange(THREADS)

    def worst(addr, act):   # most 16-byte accesses of one quarter-warp in one bank group
        w = 1
        for q in range(4):
            groups = {}
            for lane in range(8 * q, 8 * q + 8):
                if act[lane]:
                    groups.setdefault(addr[lane] % 8, set()).add(addr[lane])
            w = max(w, max((len(v) for v in groups.values()), default=0))
        return w

    def warps(addr, act):
        return max(worst(addr[32 * k:32 * k + 32], act[32 * k:32 * k + 32]) for k in range(8))

    ones = np.ones(THREADS, bool)
    # extract, pass 1 with column pairs: lanes take neighbouring pairs of one
    # chunk (2-way only where a quarter-warp wraps from the last pair to the first)
    ncol = xbu // 2
    x, j = tid % ncol, tid // ncol
    for col in (2 * x, 2 * x + 1):
        assert warps(col * J + swz(j, col >> 1, m, J), j < J) <= 2
    # extract, pass 2: lanes take one token's chunks
    xl = tid // J
    assert warps(xl * J + swz(tid % J, xl >> 1, m, J), ones) == 1
    # blend, pass 1: 4 threads per token, chunks lit + 4 r, two fp32 halves
    xc, lit = tid // 4, tid % 4
    for r in range(4):
        for c in range(2):
            assert warps(xc * jf + swzf(c * J + lit + 4 * r, xc, m, jf), xc < xbu) == 1
    # blend, pass 2: lanes take neighbouring columns of one fp32 chunk (2-way only where they wrap)
    x2, q2 = tid % xbu, tid // xbu
    for k in range(8):
        qc = q2 + 4 * k
        assert warps(x2 * jf + swzf((qc & 1) * J + (qc >> 1), x2, m, jf), q2 < 4) <= 2


# ----------------------------------------------------------------- fast blend cost split
def item_costs(p, band_rows, nbands, BC):
    SW, W = p.prefix[2][p.num_tiles[2]], p.dims[2]
    cum = [0]
    for g in range(p.dims[0] * nbands):
        f, hb0 = g // nbands, (g % nbands) * band_rows
        hb1 = min(p.dims[1], hb0 + band_rows)
        lo, hi = cover(p, 0, f)
        rows = sum(max(0, min(hb1, p.end[1][i]) - max(hb0, p.start[1][i])) for i in range(p.num_tiles[1]))
        cum.append(cum[-1] + ((hb1 - hb0) * W + (hi - lo + 1) * rows * SW) * BC)
    return cum


def share_start(cum, BC, n, G, b):
    if b >= G:
        return n
    target = b * cum[-1] // G
    g = 0
    while g + 1 < len(cum) - 1 and cum[g + 1] <= target:
        g += 1
    per = (cum[g + 1] - cum[g]) // BC
    return g * BC + min((target - cum[g] + per - 1) // per, BC)


def test_blend_cost_split_partitions_the_items(T):
    rng = np.random.default_rng(3)
    checked = 0
    while checked < 150:
        dims = (int(rng.integers(1, 20)), int(rng.integers(4, 90)), int(rng.integers(4, 130)))
        tiling = ((2, 1) if dims[0] >= 3 else (1, 0), (int(rng.integers(1, 5)), 2), (int(rng.integers(1, 5)), 3))
        try:
            p = T.plan(dims, tiling)
        except T.TdpError:
            continue
        band_rows = int(rng.integers(1, dims[1] + 1))
        nbands = -(-dims[1] // band_rows)
        BC = int(rng.integers(1, 300))
        n = dims[0] * nbands * BC
        if dims[0] * nbands > 64:
            continue
        cum = item_costs(p, band_rows, nbands, BC)
        G = min(n, int(rng.integers(1, 1300)))
        starts = [share_start(cum, BC, n, G, b) for b in range(G + 1)]
        assert starts[0] == 0 and starts[-1] == n
        assert all(a <= b for a, b in zip(starts, starts[1:]))
        checked += 1
    # the 4k workload: the heaviest CTA's share falls from 184,320 to 112,560
    # elements moved (average 109,164) on the blend's 456 CTAs
    p = T.plan((16, 68, 120), ((2, 2), (4, 8), (4, 12)))
    cum = item_costs(p, 68, 1, 128)
    starts = [share_start(cum, 128, 2048, 456, b) for b in range(457)]
    cost = [(cum[i // 128 + 1] - cum[i // 128]) // 128 for i in range(2048)]
    assert max(sum(cost[starts[b]:starts[b + 1]]) for b in range(456)) == 112560
