"""CPU models of the 16-byte streaming extract and blend kernels (no GPU).

Each model restates, in NumPy, how the kernel maps its CTAs, units, warps
and threads to data, using the launch geometry the library itself computes
(tdp_launch_geometry: band height, ring, shared layout and the per-CTA unit
ranges).  It stages every unit into an emulated shared-memory image whose
unstaged bytes hold NaN patterns, replays every shared read window, bulk
copy and global store, and checks that:
  - every shared load lies inside the CTA's allocation (extract: inside
    the staged band) and every bulk copy inside its stage, and every global
    read inside its buffer;
  - every output element is written exactly once (all CTAs modelled);
  - every element a blend term uses is the packed-tile element the method
    names (byte for byte), so the masking keeps the NaN bytes out;
  - the modelled outputs equal the oracle (extract bit for bit; blend
    within 1e-6, the model summing in float64 with the kernels' fp32
    weights where the oracle uses float64 ones).
"""
import numpy as np
import pytest

from oracle import tdp_oracle as O
from overlap_add_blending_gb300 import inputs

SMS = 152
PAD = 32


@pytest.fixture(scope="module")
def T():
    from overlap_add_blending_gb300 import build
    build.build()
    from overlap_add_blending_gb300 import tdp
    return tdp


# ----------------------------------------------------------------- plan helpers
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


def weight32(p, d, i, x):
    """The kernels' 1-D window in fp32: IEEE division, product rounded."""
    o1 = np.float32(p.overlap[d] + 1)
    up = np.float32(1.0) if i == 0 else min(np.float32(1.0), np.float32(x - p.start[d][i] + 1) / o1)
    dn = np.float32(1.0) if i == p.num_tiles[d] - 1 else min(np.float32(1.0), np.float32(p.end[d][i] - x) / o1)
    return np.float32(up * dn)


def small_div(e, sw):
    """floor(e / sw) as the kernels compute it: (e + 1/2) * fl(1/sw) in fp32, truncated."""
    inv = np.float32(1.0) / np.float32(sw)
    return ((np.asarray(e, dtype=np.float32) + np.float32(0.5)) * inv).astype(np.int64)


def unit_decode(u, BC, nb):
    """u = (f * nbands + band) * BC + bc  ->  (bc, f, band)"""
    g = u // BC
    return u % BC, g // nb, g % nb


def run_geom(p, BC, bc, f, hb0, hb1, i_f, i_h, i_w):
    fs, hs, ws = p.start[0][i_f], p.start[1][i_h], p.start[2][i_w]
    sf, sh, sw = size(p, 0, i_f), size(p, 1, i_h), size(p, 2, i_w)
    r0, r1 = max(hs, hb0), min(p.end[1][i_h], hb1)
    e0 = BC * prefix_volume(p, i_f, i_h, i_w) + bc * sf * sh * sw + ((f - fs) * sh + (r0 - hs)) * sw
    return e0, (r1 - r0) * sw, sw, ws, r0, (r0 - hs) * sw


def check_window(addr, total, nbytes, esz):
    """The words a term's window reads: nbytes from `addr` as 32-bit loads
    (2-byte elements: one extra word from the aligned start)."""
    addr = np.asarray(addr)
    lo = addr & ~3
    hi = lo + nbytes + (4 if esz == 2 else 0)
    assert (lo >= 0).all() and (hi <= total).all(), "a window leaves the shared allocation"


def check_split(starts, units, grid):
    assert len(starts) == grid + 1 and starts[0] == 0 and starts[-1] == units
    assert all(a <= b for a, b in zip(starts, starts[1:]))




# ----------------------------------------------------------------- the launch's plan tables
BAND = np.dtype([("hb0", "<i4"), ("hb1", "<i4"), ("ihlo", "<i4"), ("NHB", "<i4")])
COVER = np.dtype([("lo", "<i4"), ("n", "<i4"), ("w", "<f4", 2)])
FCON = np.dtype([("base", "<i8"), ("sf", "<i4"), ("fs", "<i4")])
WCON = np.dtype([("sw", "<i4"), ("ws", "<i4"), ("dq", "<i4"), ("dr", "<i4"), ("inv_sw", "<f4"), ("pad", "<i4", 3)])
RUN = np.dtype([("A", "<i8"), ("slice", "<i4"), ("vrow", "<i4"), ("len", "<i4"), ("src_rel", "<i4"), ("iw", "<i4"),
                ("r0b", "<i4")])
CHUNK = np.dtype({"names": ["nq", "iw", "swb", "xob", "rw", "inb", "col", "cls"],
                  "formats": ["<i4", ("<i4", 3), ("<i4", 3), ("<i4", 3), ("<f4", (3, 8)), ("<u4", 3), "<i4", "<i4"],
                  "offsets": [0, 4, 16, 28, 40, 136, 148, 152], "itemsize": 160})



def check_tables(p, g, buf, offs, BC, esz_stage, blend, rows=None):
    """Every entry of the launch's tables against an independent reconstruction
    (bands over output rows [r0, r1), the whole H unless a slab)."""
    F, H, W = p.dims
    w0, w1 = rows or (0, H)   # the bands' rows
    nw, br, nb = p.num_tiles[2], g["band_rows"], g["nbands"]
    assert nb == -(-(w1 - w0) // br)
    bands = np.frombuffer(buf, BAND, nb, 16 * offs["band"])
    rpb = max(cover(p, 1, min(w1, w0 + b * br + br) - 1)[1] - cover(p, 1, w0 + b * br)[0] + 1 for b in range(nb)) * nw
    for b in range(nb):
        hb0, hb1 = w0 + b * br, min(w1, w0 + b * br + br)
        lo, hi = cover(p, 1, hb0)[0], cover(p, 1, hb1 - 1)[1]
        assert tuple(bands[b]) == (hb0, hb1, lo, hi - lo + 1)
    frames = np.frombuffer(buf, COVER, F, 16 * offs["frame"])
    for f in range(F):
        lo, hi = cover(p, 0, f)
        assert (frames[f]["lo"], frames[f]["n"]) == (lo, hi - lo + 1)
        assert frames[f]["w"][0] == weight32(p, 0, lo, f)
        assert frames[f]["w"][1] == (weight32(p, 0, lo + 1, f) if hi > lo else 0)
    fcon = np.frombuffer(buf, FCON, p.num_tiles[0], 16 * offs["fcon"])
    SH, SW = p.prefix[1][p.num_tiles[1]], p.prefix[2][nw]
    for i in range(p.num_tiles[0]):
        assert tuple(fcon[i]) == (p.prefix[0][i] * SH * SW, size(p, 0, i), p.start[0][i])
    runs = np.frombuffer(buf, RUN, nb * rpb, 16 * offs["runs"]).reshape(nb, rpb)
    for b in range(nb):
        hb0, hb1 = w0 + b * br, min(w1, w0 + b * br + br)
        lo = cover(p, 1, hb0)[0]
        for rr in range(rpb):
            jh, iw = divmod(rr, nw)
            if jh < bands[b]["NHB"]:
                ih = lo + jh
                hs, sh, sw = p.start[1][ih], size(p, 1, ih), size(p, 2, iw)
                r0, r1 = max(hs, hb0), min(p.end[1][ih], hb1)
                want = (p.prefix[1][ih] * SW + sh * p.prefix[2][iw], sh * sw, (r0 - hs) * sw, (r1 - r0) * sw,
                        ((r0 - hb0) * W + p.start[2][iw]) * esz_stage)
                assert tuple(runs[b, rr])[:5] == want, (b, rr)
                assert runs[b, rr]["iw"] == iw, (b, rr)   # the run's column tile, read instead of rr mod nw
                assert runs[b, rr]["r0b"] == r0 * sw * esz_stage, (b, rr)   # first latent row x tile row bytes
    if not blend:
        wcon = np.frombuffer(buf, WCON, nw, 16 * offs["wcon"])
        for i in range(nw):
            sw = size(p, 2, i)
            step = 32 * (8 // esz_stage)
            assert tuple(wcon[i])[:4] == (sw, p.start[2][i], step // sw, step % sw)
            assert wcon[i]["inv_sw"] == np.float32(1.0) / np.float32(sw)
        return
    rows = np.frombuffer(buf, COVER, H, 16 * offs["row"])
    for h in range(H):
        lo, hi = cover(p, 1, h)
        assert (rows[h]["lo"], rows[h]["n"]) == (lo, hi - lo + 1)
        assert rows[h]["w"][0] == weight32(p, 1, lo, h)
        assert rows[h]["w"][1] == (weight32(p, 1, lo + 1, h) if hi > lo else 0)
    cpr = g["chunks_per_row"]
    E = W // cpr
    chunks = np.frombuffer(buf, CHUNK, cpr, 16 * offs["chunk"])
    # every chunk column once, the entries ordered by class: 0 = one term
    # reaching all E columns with r_w = 1, 1 = one term otherwise, 2 / 3 =
    # two / three terms; within a class in column order
    assert sorted(chunks["col"]) == list(range(cpr))
    assert list(chunks["cls"]) == sorted(chunks["cls"])
    for k in range(cpr):
        c = chunks[k]
        j = int(c["col"])
        terms = col_terms(p, j, E)
        assert c["nq"] == len(terms)
        for q, (iw, sw, xo, inn, rw) in enumerate(terms):
            assert (c["iw"][q], c["swb"][q], c["xob"][q]) == (iw, sw * esz_stage, xo * esz_stage)
            assert np.array_equal(c["rw"][q][:E], rw), (j, q)
            assert c["inb"][q] == sum(1 << m for m in range(E) if inn[m])
        ones = len(terms) == 1 and all(terms[0][3][:E]) and np.all(terms[0][4] == 1.0)
        assert c["cls"] == (0 if ones else min(len(terms), 3)), j
        if k > 0 and chunks[k - 1]["cls"] == c["cls"]:
            assert chunks[k - 1]["col"] < j


# ----------------------------------------------------------------- extract
def model_extract(p, g, starts, B, C, esz, lat_bytes, ctas):
    F, H, W = p.dims
    nw = p.num_tiles[2]
    S, SB, off_data, br, nb = g["stages"], g["stage_bytes"], g["off_data"], g["band_rows"], g["nbands"]
    total = g["shared_bytes"]
    epw = 4 // esz
    BC = B * C
    n_el = p.tiles_numel(B, C)
    out = np.full(n_el * esz, 0xEE, np.uint8)
    count = np.zeros(n_el, np.int64)
    for cta in ctas:
        for k, u in enumerate(range(starts[cta], starts[cta + 1])):
            s = k % S
            bc, f, band = unit_decode(u, BC, nb)
            hb0, hb1 = band * br, min(H, band * br + br)
            data_off = off_data + s * SB + PAD
            nbytes = (hb1 - hb0) * W * esz
            assert data_off % 16 == 0 and nbytes % 16 == 0
            assert data_off + nbytes + PAD <= off_data + (s + 1) * SB <= total
            lat0 = ((bc * F + f) * H + hb0) * W * esz
            assert lat0 % 16 == 0 and lat0 + nbytes <= len(lat_bytes)
            smem = np.full(total, 0xCD, np.uint8)
            smem[data_off:data_off + nbytes] = lat_bytes[lat0:lat0 + nbytes]
            flo, fhi = cover(p, 0, f)
            ihlo, ihhi = cover(p, 1, hb0)[0], cover(p, 1, hb1 - 1)[1]
            for i_f in range(flo, fhi + 1):
                for i_h in range(ihlo, ihhi + 1):
                    for i_w in range(nw):
                        e0, ln, sw, ws, r0, _ = run_geom(p, BC, bc, f, hb0, hb1, i_f, i_h, i_w)
                        src0 = data_off + ((r0 - hb0) * W + ws) * esz
                        epq = 8 // esz
                        hd = ((8 - (e0 * esz) % 8) % 8) // esz          # elements before the first 8-byte boundary
                        nq = (ln - hd) // epq if ln > hd else 0
                        # body groups: the kernel's addressing, element m of a group
                        # past the tile row taken W - w_t columns further on
                        e = hd + epq * np.arange(nq)
                        y = small_div(e, sw)
                        assert np.array_equal(y, e // sw), "fp32 row division is not exact"
                        x = e - y * sw
                        ad = src0 + (y * W + x) * esz
                        k1 = sw - x
                        m = np.arange(epq)
                        srcs = (ad[:, None] + m * esz + np.where(m[None, :] >= k1[:, None], (W - sw) * esz, 0)).ravel()
                        els = (e[:, None] + m).ravel()
                        # head and tail elements, one by one
                        rest = np.concatenate([np.arange(min(hd, ln)), np.arange(hd + epq * nq, ln)])
                        yr = small_div(rest, sw)
                        srcs = np.concatenate([srcs, src0 + (yr * W + (rest - yr * sw)) * esz])
                        els = np.concatenate([els, rest])
                        direct = src0 + ((els // sw) * W + els % sw) * esz
                        assert np.array_equal(srcs, direct), "a group element is read from the wrong place"
                        assert ((srcs >= data_off) & (srcs + esz <= data_off + nbytes)).all(), \
                            "a load leaves the staged band"
                        assert ((els >= 0) & (els < ln)).all()
                        dst = (e0 + els) * esz
                        for bb in range(esz):
                            out[dst + bb] = smem[srcs + bb]
                        np.add.at(count, e0 + els, 1)
    return out, count


# ----------------------------------------------------------------- blend
def col_terms(p, j, E):
    c0 = j * E
    lo = cover(p, 2, c0)[0]
    hi = cover(p, 2, c0 + E - 1)[1]
    terms = []
    for i in range(lo, hi + 1):
        w0, w1 = p.start[2][i], p.end[2][i]
        inn = np.array([w0 <= c0 + m < w1 for m in range(E)])
        rw = np.array([weight32(p, 2, i, c0 + m) if inn[m] else np.float32(0) for m in range(E)], dtype=np.float32)
        terms.append((i, w1 - w0, c0 - w0, inn, rw))
    return terms


def decode(b, esz):
    if esz == 4:
        return b.view(np.float32).astype(np.float64)
    return (b.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def model_blend(p, g, starts, B, C, in_esz, out_esz, tiles_bytes, ctas, rows=None):
    F, H, W = p.dims
    nw = p.num_tiles[2]
    S, SB, off_data, off_hdr = g["stages"], g["stage_bytes"], g["off_data"], g["off_hdr"]
    br, nb, max_runs, total = g["band_rows"], g["nbands"], g["max_runs"], g["shared_bytes"]
    assert S >= 2
    E = 16 // out_esz
    cpr = g["chunks_per_row"]
    assert cpr == W * out_esz // 16 and cpr <= g["threads"]
    BC = B * C
    limit = len(tiles_bytes) & ~15
    terms = [col_terms(p, j, E) for j in range(cpr)]
    assert max(len(t) for t in terms) == g["column_terms"]
    # the row groups of each chunk class (0: one term of weight 1 over the
    # chunk, 1: one term otherwise, 2/3: two/three terms): every class with
    # entries has some, their threads fit the CTA, and the step is band rows
    # mod groups
    def cls_of(t):
        return (0 if t[0][3].all() and (t[0][4] == 1).all() else 1) if len(t) == 1 else len(t)
    ncls = [sum(cls_of(t) == c for t in terms) for c in range(4)]
    G, step, first = g["row_groups"], g["row_step"], g["class_first"]
    assert all((G[c] > 0) == (ncls[c] > 0) and G[c] <= br for c in range(4))
    # the classes' thread ranges follow one another inside the CTA's compute threads, on warp
    # boundaries when they fit in whole warps
    ends = [first[c] + ncls[c] * G[c] for c in range(4)]
    assert all(first[c + 1] >= ends[c] for c in range(3)) and ends[3] <= g["threads"]
    if sum(-(-n // 32) for n in ncls) <= g["threads"] // 32:
        assert all(f % 32 == 0 for f in first)
    assert all(step[c] == (br % G[c] if G[c] else 0) for c in range(4))
    assert g["rows_per_thread"] == max(-(-br // G[c]) for c in range(4) if G[c])
    w0, w1 = rows or (0, H)   # the output rows (a slab's, else all): out is [BC, F, w1 - w0, W]
    HS = w1 - w0
    out = np.full(BC * F * HS * W, np.nan)
    count = np.zeros(BC * F * HS * cpr, np.int64)
    for cta in ctas:
        j = 0   # stages filled so far: one per covering frame tile of a unit
        for k, u in enumerate(range(starts[cta], starts[cta + 1])):
            bc, f, band = unit_decode(u, BC, nb)
            hb0, hb1 = w0 + band * br, min(w1, w0 + band * br + br)
            flo, fhi = cover(p, 0, f)
            ihlo, ihhi = cover(p, 1, hb0)[0], cover(p, 1, hb1 - 1)[1]
            NHB = ihhi - ihlo + 1
            nruns = (fhi - flo + 1) * NHB * nw
            stages = [(j + fa) % S for fa in range(fhi - flo + 1)]
            assert len(stages) <= 2 and len(set(stages)) == len(stages), "a unit's stages collide"
            j += len(stages)
            assert NHB * nw <= max_runs
            for s in stages:
                assert off_hdr + (s + 1) * max_runs * 4 <= off_data
            smem = np.full(total, 0xFF, np.uint8)   # NaN in bf16 and fp32 wherever nothing was staged
            hdr = np.zeros(nruns, np.int64)
            slot = g["run_slot"]
            for r in range(nruns):
                iw, q = r % nw, r // nw
                jh, fa = q % NHB, q // NHB
                s = stages[fa]
                e0, ln, sw, ws, r0, vrow = run_geom(p, BC, bc, f, hb0, hb1, flo + fa, ihlo + jh, iw)
                g0 = e0 * in_esz
                g1 = g0 + ln * in_esz
                lo = g0 & ~15
                up = (g1 + 15) & ~15
                off = off_data + s * SB + PAD + (r - fa * NHB * nw) * slot
                assert off % 16 == 0 and up - lo <= slot, "a run overflows its slot"
                assert off + slot <= off_data + (s + 1) * SB - PAD, "a slot leaves its stage"
                assert 0 <= lo and g1 <= len(tiles_bytes)
                # one bulk copy of whole 16-byte chunks; elements in the tile
                # buffer's last, partial chunk loaded one by one
                hi = up if up <= limit else g1 & ~15
                hi = max(hi, lo)
                smem[off:off + hi - lo] = tiles_bytes[lo:hi]
                t0 = max(hi, g0)
                smem[off + t0 - lo:off + g1 - lo] = tiles_bytes[t0:g1]
                hdr[r] = off + (g0 - lo) - r0 * sw * in_esz   # latent row h of the tile starts at hdr + h * row bytes
            fe = [(i, weight32(p, 0, i, f)) for i in range(flo, fhi + 1)]
            # the k-th unit's rows of each chunk entry: group g takes rows g', g' + G, ... of the band,
            # g' = (g + k * step) mod G; every (entry, row) exactly once
            taken = np.zeros((cpr, hb1 - hb0), np.int64)
            for jc in range(cpr):
                c = cls_of(terms[jc])
                for grp in range(G[c]):
                    taken[jc, (grp + k * step[c]) % G[c]::G[c]] += 1
            assert (taken == 1).all()
            for h in range(hb0, hb1):
                hlo, hhi = cover(p, 1, h)
                acc = np.zeros((cpr, E))
                for fa, (i_f, rf) in enumerate(fe):
                    for ih in range(hlo, hhi + 1):
                        wfh = np.float32(rf * weight32(p, 1, ih, h))
                        base = (fa * NHB + ih - ihlo) * nw
                        yo = h - p.start[1][ih]
                        fs, hs = p.start[0][i_f], p.start[1][ih]
                        sf, sh = size(p, 0, i_f), size(p, 1, ih)
                        for j in range(cpr):
                            inner = np.zeros(E)
                            for (iw, sw, xo, inn, rw) in terms[j]:
                                ad = hdr[base + iw] + (h * sw + xo) * in_esz
                                check_window(ad, total, E * in_esz, in_esz)
                                m = np.arange(E)
                                pos = ad + m * in_esz
                                raw = np.stack([smem[pos + b] for b in range(in_esz)], axis=1).ravel()
                                val = decode(raw, in_esz)
                                e = (BC * prefix_volume(p, i_f, ih, iw) + bc * sf * sh * sw +
                                     ((f - fs) * sh + yo) * sw + xo + m)
                                for mm in np.nonzero(inn)[0]:
                                    want = tiles_bytes[e[mm] * in_esz:(e[mm] + 1) * in_esz]
                                    assert np.array_equal(raw[mm * in_esz:(mm + 1) * in_esz], want), \
                                        "a term reads the wrong tile element"
                                inner += np.where(inn, rw.astype(np.float64) * np.where(inn, val, 0.0), 0.0)
                            acc[j] += np.float64(wfh) * inner
                row = ((bc * F + f) * HS + h - w0) * W
                out[row:row + W] = acc.ravel()
                count[((bc * F + f) * HS + h - w0) * cpr + np.arange(cpr)] += 1
    return out, count


# ----------------------------------------------------------------- cases
def _plan_pair(T, dims, tiling, compat=False):
    return T.plan(dims, tiling, compat=compat), O.make_plan(dims, tiling, compat=compat)


def _latent(B, C, dims, esz, seed=0):
    X = inputs.latent((B, C) + tuple(dims), seed=seed)
    if esz == 2:
        bits = (X.view(np.uint32) + 0x7FFF + ((X.view(np.uint32) >> 16) & 1)) >> 16   # round to nearest even
        Xb = bits.astype(np.uint16)
        return Xb.ravel().view(np.uint8).copy(), (Xb.astype(np.uint32) << 16).view(np.float32)
    return X.ravel().view(np.uint8).copy(), X


CASES = [
    # (dims, tiling, B, C, esz in, esz out, all CTAs)
    ((4, 16, 16), ((1, 0), (2, 4), (2, 4)), 1, 8, 4, 4, True),           # tiny
    ((16, 16, 24), ((1, 0), (2, 4), (2, 6)), 1, 16, 2, 2, True),         # stage-1 shape, fewer channels
    ((16, 32, 48), ((1, 0), (2, 8), (2, 12)), 1, 4, 2, 2, True),         # full-res shape, fewer channels
    ((2, 300, 200), ((1, 0), (3, 20), (2, 16)), 1, 2, 2, 2, True),      # row bands
    ((2, 300, 200), ((1, 0), (3, 20), (2, 16)), 1, 2, 4, 4, True),
    ((4, 16, 24), ((1, 0), (2, 4), (2, 6)), 1, 16, 2, 4, True),         # bf16 tiles -> fp32 latent
    ((4, 16, 24), ((1, 0), (2, 4), (2, 6)), 1, 16, 4, 2, True),         # fp32 tiles -> bf16 latent
    ((3, 16, 16), ((2, 1), (2, 4), (2, 4)), 1, 1, 4, 4, True),          # a CTA range may be empty
    ((16, 68, 120), ((2, 2), (4, 8), (4, 12)), 1, 2, 2, 2, True),       # 4k-class tiling, 2 channels
    ((16, 68, 120), ((2, 2), (4, 8), (4, 12)), 1, 128, 2, 2, False),    # 4k-class workload, 3 CTAs
]


def _dt(esz):
    import torch
    return torch.float32 if esz == 4 else torch.bfloat16


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[2]}x{c[3]}-{c[4]}{c[5]}" for c in CASES])
def test_extract_stream_model(T, case):
    dims, tiling, B, C, esz, _, full = case
    p, rp = _plan_pair(T, dims, tiling)
    g, starts, buf, offs = T.launch_geometry(p, B, C, False, _dt(esz), _dt(esz), SMS, tables=True)
    assert g["streaming"] == 1
    check_split(starts, g["units"], g["grid"])
    check_tables(p, g, buf, offs, B * C, esz, False)
    lat_bytes, Xv = _latent(B, C, dims, esz)
    ctas = range(g["grid"]) if full else sorted({0, g["grid"] // 2, g["grid"] - 1})
    out, count = model_extract(p, g, starts, B, C, esz, lat_bytes, ctas)
    ref = O.pack(O.extract(rp, Xv.astype(np.float64))).astype(np.float32)
    ref_bytes = (ref.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8) if esz == 2 else ref.view(np.uint8)
    if full:
        assert (count == 1).all(), "a tile element is written zero or several times"
        assert np.array_equal(out, ref_bytes)
    else:
        assert count.max() == 1
        done = np.repeat(count == 1, esz)
        assert np.array_equal(out[done], ref_bytes[done])


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[2]}x{c[3]}-{c[4]}{c[5]}" for c in CASES])
def test_blend_stream_model(T, case):
    dims, tiling, B, C, in_esz, out_esz, full = case
    p, rp = _plan_pair(T, dims, tiling)
    g, starts, buf, offs = T.launch_geometry(p, B, C, True, _dt(in_esz), _dt(out_esz), SMS, tables=True)
    if not g["streaming"]:
        pytest.skip("the general blend kernel takes this shape (its tables exceed the launch's table block)")
    check_split(starts, g["units"], g["grid"])
    check_tables(p, g, buf, offs, B * C, in_esz, True)
    n = p.tiles_numel(B, C)
    rng = np.random.default_rng(7)
    vals = rng.standard_normal(n).astype(np.float32)
    if in_esz == 2:
        bits = ((vals.view(np.uint32) + 0x7FFF + ((vals.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
        tiles_bytes = bits.view(np.uint8).copy()
        tv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        tiles_bytes = vals.view(np.uint8).copy()
        tv = vals.astype(np.float64)
    ctas = range(g["grid"]) if full else sorted({0, g["grid"] // 2, g["grid"] - 1})
    out, count = model_blend(p, g, starts, B, C, in_esz, out_esz, tiles_bytes, ctas)
    ref = O.blend(rp, O.unpack(rp, B, C, tv)).ravel()
    if full:
        assert (count == 1).all(), "an output chunk is written zero or several times"
        assert np.allclose(out, ref, rtol=1e-6, atol=1e-6)
    else:
        assert count.max() == 1
        done = ~np.isnan(out)
        assert done.sum() > 0
        assert np.allclose(out[done], ref[done], rtol=1e-6, atol=1e-6)


SLAB_CASES = [
    # (dims, tiling, B, C, esz in, esz out, (row0, row1))
    ((16, 68, 120), ((2, 2), (4, 8), (4, 12)), 1, 2, 2, 2, (0, 34)),      # 4k-class tiling, rank 0 of 2
    ((16, 68, 120), ((2, 2), (4, 8), (4, 12)), 1, 2, 2, 2, (22, 45)),     # rank 1 of 3: both ends inside overlaps
    ((16, 68, 120), ((2, 2), (4, 8), (4, 12)), 1, 1, 2, 2, (67, 68)),     # one row
    ((4, 16, 24), ((1, 0), (2, 4), (2, 6)), 1, 4, 2, 4, (5, 13)),         # bf16 tiles -> fp32 slab
    ((8, 120, 64), ((2, 1), (4, 8), (2, 8)), 1, 1, 4, 4, (13, 101)),      # two bands, the last one short
]


@pytest.mark.parametrize("case", SLAB_CASES, ids=[f"{c[0]}-{c[6]}" for c in SLAB_CASES])
def test_blend_slab_stream_model(T, case):
    """The streaming blend restricted to output rows [row0, row1) (what
    tdp_blend_slab launches): its tables, its split, and its staging and
    addressing replayed in NumPy, every slab chunk written once and equal to
    those rows of the oracle's blend."""
    dims, tiling, B, C, in_esz, out_esz, rows = case
    p, rp = _plan_pair(T, dims, tiling)
    g, starts, buf, offs = T.launch_geometry(p, B, C, True, _dt(in_esz), _dt(out_esz), SMS, tables=True, rows=rows)
    assert g["streaming"]
    check_split(starts, g["units"], g["grid"])
    check_tables(p, g, buf, offs, B * C, in_esz, True, rows=rows)
    n = p.tiles_numel(B, C)
    vals = np.random.default_rng(11).standard_normal(n).astype(np.float32)
    if in_esz == 2:
        bits = ((vals.view(np.uint32) + 0x7FFF + ((vals.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
        tiles_bytes = bits.view(np.uint8).copy()
        tv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        tiles_bytes = vals.view(np.uint8).copy()
        tv = vals.astype(np.float64)
    out, count = model_blend(p, g, starts, B, C, in_esz, out_esz, tiles_bytes, range(g["grid"]), rows=rows)
    ref = O.blend(rp, O.unpack(rp, B, C, tv))[..., rows[0]:rows[1], :].ravel()
    assert (count == 1).all(), "a slab chunk is written zero or several times"
    assert np.allclose(out, ref, rtol=1e-6, atol=1e-6)


def test_slabs_of_the_4k_workload_stream(T):
    """Every rank's slab of the 4K-class workload, R = 2..7, takes the
    streaming blend (tdp_blend_slab's fast path), its bands cover exactly
    the slab's rows, and every chunk class starts on a warp boundary."""
    p = T.plan((16, 68, 120), ((2, 2), (4, 8), (4, 12)))
    for R in range(2, 8):
        for r in range(R):
            sh = T.shard_plan(p, R, r)
            if sh.row0 == sh.row1:
                continue
            g, starts = T.launch_geometry(p, 1, 128, True, _dt(2), _dt(2), SMS,
                                          rows=(sh.row0, sh.row1))
            assert g["streaming"] == 1, (R, r)
            assert g["nbands"] == -(-(sh.row1 - sh.row0) // g["band_rows"])
            assert all(f % 32 == 0 for f in g["class_first"])
            check_split(starts, g["units"], g["grid"])


def _random_plan(T, rng):
    """A random plan within the partition-of-unity guard (overlap * (n + 1) <= dim)."""
    dims = (int(rng.integers(1, 9)), int(rng.integers(8, 97)), 8 * int(rng.integers(2, 25)))
    tiling = []
    for d in dims:
        n = int(rng.integers(1, min(5, d) + 1))
        tiling.append((n, int(rng.integers(0, d // (n + 1) + 1)) if n > 1 else 0))
    return T.plan(dims, tuple(tiling)), dims


def test_random_blend_geometries(T):
    """Seeded random plans, whole-latent and slab windows, bf16 and fp32:
    wherever the streaming blend takes the call, its tables match an
    independent reconstruction, the split is monotone, every chunk class
    starts on a warp boundary, and in every unit of every CTA each (chunk
    entry, band row) is taken by exactly one thread."""
    rng = np.random.default_rng(2024)
    streamed = 0
    for _ in range(60):
        p, dims = _random_plan(T, rng)
        H = dims[1]
        r0 = int(rng.integers(0, H))
        r1 = int(rng.integers(r0 + 1, H + 1))
        for rows in ((0, H), (r0, r1)):
            esz = int(rng.choice([2, 4]))
            B, C = 1, int(rng.integers(1, 5))
            g, starts, buf, offs = T.launch_geometry(p, B, C, True, _dt(esz), _dt(esz), SMS, tables=True, rows=rows)
            if not g["streaming"]:
                continue
            streamed += 1
            check_split(starts, g["units"], g["grid"])
            check_tables(p, g, buf, offs, B * C, esz, True, rows=rows)
            chunks = np.frombuffer(buf, CHUNK, g["chunks_per_row"], 16 * offs["chunk"])
            ncls = [int((chunks["cls"] == c).sum()) for c in range(4)]
            G, step, first = g["row_groups"], g["row_step"], g["class_first"]
            br = g["band_rows"]
            assert all((G[c] > 0) == (ncls[c] > 0) and G[c] <= br for c in range(4))
            assert all(first[c] % 32 == 0 for c in range(4))
            assert max(first[c] + ncls[c] * G[c] for c in range(4)) <= g["threads"]
            for k in range(3):   # a CTA's first units: the rotating starts cover every row once
                for c in range(4):
                    if G[c] == 0:
                        continue
                    taken = np.zeros(br, np.int64)
                    for grp in range(G[c]):
                        taken[(grp + k * step[c]) % G[c]::G[c]] += 1
                    assert (taken == 1).all()
    assert streamed >= 40   # most random plans stream


def test_random_extract_geometries(T):
    """Seeded random plans, bf16 and fp32: wherever the streaming extract
    takes the call, its tables match an independent reconstruction and the
    split is monotone."""
    rng = np.random.default_rng(4096)
    streamed = 0
    for _ in range(60):
        p, dims = _random_plan(T, rng)
        esz = int(rng.choice([2, 4]))
        B, C = 1, int(rng.integers(1, 5))
        g, starts, buf, offs = T.launch_geometry(p, B, C, False, _dt(esz), _dt(esz), SMS, tables=True)
        if not g["streaming"]:
            continue
        streamed += 1
        check_split(starts, g["units"], g["grid"])
        check_tables(p, g, buf, offs, B * C, esz, False)
    assert streamed >= 30


def test_random_blend_replays(T):
    """Small seeded random plans and slab windows, replayed in NumPy through
    the streaming blend's staging and addressing: every output chunk of the
    window written once and equal to the oracle's blend there."""
    rng = np.random.default_rng(77)
    replayed = 0
    while replayed < 16:
        dims = (int(rng.integers(1, 4)), int(rng.integers(8, 33)), 8 * int(rng.integers(2, 7)))
        tiling = []
        for d in dims:
            n = int(rng.integers(1, min(4, d) + 1))
            tiling.append((n, int(rng.integers(0, d // (n + 1) + 1)) if n > 1 else 0))
        p, rp = _plan_pair(T, dims, tuple(tiling))
        H = dims[1]
        r0 = int(rng.integers(0, H))
        rows = (r0, int(rng.integers(r0 + 1, H + 1))) if replayed % 2 else (0, H)
        esz = int(rng.choice([2, 4]))
        g, starts, buf, offs = T.launch_geometry(p, 1, 1, True, _dt(esz), _dt(esz), SMS, tables=True, rows=rows)
        if not g["streaming"]:
            continue
        n = p.tiles_numel(1, 1)
        vals = rng.standard_normal(n).astype(np.float32)
        if esz == 2:
            bits = ((vals.view(np.uint32) + 0x7FFF + ((vals.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
            tiles_bytes = bits.view(np.uint8).copy()
            tv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        else:
            tiles_bytes = vals.view(np.uint8).copy()
            tv = vals.astype(np.float64)
        out, count = model_blend(p, g, starts, 1, 1, esz, esz, tiles_bytes, range(g["grid"]), rows=rows)
        ref = O.blend(rp, O.unpack(rp, 1, 1, tv))[..., rows[0]:rows[1], :].ravel()
        assert (count == 1).all(), (dims, tiling, rows)
        assert np.allclose(out, ref, rtol=1e-6, atol=1e-6), (dims, tiling, rows)
        replayed += 1


def test_random_extract_replays(T):
    """Small seeded random plans replayed in NumPy through the streaming
    extract's staging and span writes: every tile element written once and
    equal to the oracle's packed tiles (a bit copy)."""
    rng = np.random.default_rng(99)
    replayed = 0
    while replayed < 16:
        dims = (int(rng.integers(1, 4)), int(rng.integers(8, 33)), 8 * int(rng.integers(2, 7)))
        tiling = []
        for d in dims:
            n = int(rng.integers(1, min(4, d) + 1))
            tiling.append((n, int(rng.integers(0, d // (n + 1) + 1)) if n > 1 else 0))
        p, rp = _plan_pair(T, dims, tuple(tiling))
        esz = int(rng.choice([2, 4]))
        g, starts, buf, offs = T.launch_geometry(p, 1, 1, False, _dt(esz), _dt(esz), SMS, tables=True)
        if not g["streaming"]:
            continue
        lat_bytes, Xv = _latent(1, 1, dims, esz, seed=replayed)
        out, count = model_extract(p, g, starts, 1, 1, esz, lat_bytes, range(g["grid"]))
        ref = O.pack(O.extract(rp, Xv.astype(np.float64))).astype(np.float32)
        ref_bytes = (ref.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8) if esz == 2 else ref.view(np.uint8)
        assert (count == 1).all(), (dims, tiling)
        assert np.array_equal(out, ref_bytes), (dims, tiling)
        replayed += 1


def test_launch_geometry_rows_checked(T):
    p = T.plan((4, 16, 16), ((1, 0), (2, 4), (2, 4)))
    for rows in ((0, 0), (5, 3), (-1, 4), (0, 17)):
        with pytest.raises(T.TdpError):
            T.launch_geometry(p, 1, 8, True, _dt(4), _dt(4), SMS, rows=rows)
    with pytest.raises(T.TdpError):   # extract covers the whole latent
        T.launch_geometry(p, 1, 8, False, _dt(4), _dt(4), SMS, rows=(0, 8))


def test_split_balances_bytes(T):
    # every CTA's share of the 4k-class extract and blend is within one unit of the mean
    p = T.plan((16, 68, 120), ((2, 2), (4, 8), (4, 12)))
    import torch
    for blend in (False, True):
        g, starts = T.launch_geometry(p, 1, 128, blend, torch.bfloat16, torch.bfloat16, SMS)
        check_split(starts, g["units"], g["grid"])
        F, H, W = p.dims
        br, nb = g["band_rows"], g["nbands"]
        cost = []
        for u in range(g["units"]):
            bc, f, band = unit_decode(u, 128, nb)
            hb0, hb1 = band * br, min(H, band * br + br)
            rows = sum(max(0, min(hb1, p.end[1][i]) - max(hb0, p.start[1][i])) for i in range(p.num_tiles[1]))
            lo, hi = cover(p, 0, f)
            cost.append(((hb1 - hb0) * W + rows * (hi - lo + 1) * p.prefix[2][p.num_tiles[2]]) * 2)
        cum = np.concatenate([[0], np.cumsum(cost)])
        share = cum[starts[1:]] - cum[starts[:-1]]
        assert share.max() - cum[-1] / g["grid"] <= max(cost)


@pytest.mark.parametrize("name", ["tiny", "stage1", "fullres", "4k", "strips", "grid"])
def test_named_workloads_take_the_streaming_kernels(T, name):
    from overlap_add_blending_gb300.workloads import WORKLOADS
    wl = WORKLOADS[name]
    p = T.plan(wl.dims, wl.tiling)
    dt = _dt(4 if wl.dtype == "f32" else 2)
    for blend in (False, True):
        g, starts = T.launch_geometry(p, wl.B, wl.C, blend, dt, dt, SMS)
        assert g["streaming"] == 1, (name, blend)
        assert g["stages"] >= 2
        check_split(starts, g["units"], g["grid"])
