// Host side of libtdp: interval planning, tile bookkeeping, layout
// statistics and status strings.  Touches no GPU.
//
// Interval split (mold issue #673, "A bug found while porting", and the TDP
// docs' DimensionTilingConfig(num_tiles, overlap)): stride
// s = floor((dim - overlap) / n), tile i = [i*s, i*s + s + overlap), the last
// tile stretched to end at dim; the partition-of-unity guard
// overlap * (n + 1) <= dim is enforced unless TDP_PLAN_UPSTREAM_COMPAT.
#include <algorithm>
#include <cstring>
#include <vector>

#include "tdp.h"
#include "tdp_geometry.h"

namespace {

tdp_status plan_axis(int32_t dim, const tdp_dim_cfg& cfg, uint32_t flags, int d, tdp_plan_t* p) {
    const int32_t n = cfg.num_tiles, o = cfg.overlap;
    if (dim < 1 || n < 1 || o < 0) return TDP_ERR_INVALID_ARG;
    if (n > TDP_MAX_PER_AXIS) return TDP_ERR_TOO_MANY_TILES;
    if (n == 1 && o != 0) return TDP_ERR_INVALID_ARG;
    const int64_t stride = (n == 1) ? dim : ((int64_t)dim - o) / n;
    if (stride < 1) return TDP_ERR_INVALID_ARG;
    if (!(flags & TDP_PLAN_UPSTREAM_COMPAT) && (int64_t)o * (n + 1) > dim) return TDP_ERR_GUARD;
    p->dims[d] = dim;
    p->num_tiles[d] = n;
    p->overlap[d] = o;
    p->stride[d] = (int32_t)stride;
    for (int i = 0; i < n; ++i) {
        p->start[d][i] = (int32_t)(i * stride);
        p->end[d][i] = (int32_t)(i * stride + stride + o);
    }
    p->end[d][n - 1] = dim;
    p->prefix[d][0] = 0;
    for (int i = 0; i < n; ++i) p->prefix[d][i + 1] = p->prefix[d][i] + (p->end[d][i] - p->start[d][i]);
    // Most tiles covering one index: coverage only rises at a tile start.
    int best = 0;
    for (int i = 0; i < n; ++i) {
        int c = 0;
        for (int j = 0; j < n; ++j) c += (p->start[d][j] <= p->start[d][i] && p->start[d][i] < p->end[d][j]);
        best = std::max(best, c);
    }
    p->max_cover[d] = best;
    return TDP_OK;
}

// Per-axis window-sum numerators in units of 1 / (overlap + 1)^2.
std::vector<int64_t> axis_sum_numerators(const tdp_plan_t& p, int d) {
    const int n = p.num_tiles[d], dim = p.dims[d];
    const int64_t o1 = p.overlap[d] + 1;
    std::vector<int64_t> s(dim, 0);
    for (int i = 0; i < n; ++i) {
        const int a = p.start[d][i], e = p.end[d][i];
        for (int x = a; x < e; ++x) {
            const int64_t up = (i == 0) ? o1 : std::min<int64_t>(o1, x - a + 1);
            const int64_t dn = (i == n - 1) ? o1 : std::min<int64_t>(o1, e - x);
            s[x] += up * dn;
        }
    }
    return s;
}

// ---------------------------------------------------------------- layout search
// The criteria of DistVAE "Choosing a tile window" (Benchmark plan
// selection): window area, decoded area, rank imbalance, tile columns.
// Imbalance is heaviest rank / total, compared by cross-multiplying.
bool beats(const tdp_layout_candidate& a, const tdp_layout_candidate& b) {
    const __int128 ia = (__int128)a.heaviest_rank_volume * b.decoded_volume;
    const __int128 ib = (__int128)b.heaviest_rank_volume * a.decoded_volume;
    const bool le = a.window_volume <= b.window_volume && a.decoded_volume <= b.decoded_volume && ia <= ib &&
                    a.num_tiles[2] <= b.num_tiles[2];
    const bool lt = a.window_volume < b.window_volume || a.decoded_volume < b.decoded_volume || ia < ib ||
                    a.num_tiles[2] < b.num_tiles[2];
    return le && lt;
}

// Fixed order among candidates equal on the selection key: less decoded
// area, less imbalance, fewer tile columns, fewer tile rows.
bool before_on_ties(const tdp_layout_candidate& a, const tdp_layout_candidate& b) {
    if (a.decoded_volume != b.decoded_volume) return a.decoded_volume < b.decoded_volume;
    const __int128 ia = (__int128)a.heaviest_rank_volume * b.decoded_volume;
    const __int128 ib = (__int128)b.heaviest_rank_volume * a.decoded_volume;
    if (ia != ib) return ia < ib;
    if (a.num_tiles[2] != b.num_tiles[2]) return a.num_tiles[2] < b.num_tiles[2];
    return a.num_tiles[1] < b.num_tiles[1];
}

double imbalance_of(const tdp_layout_candidate& c, int ranks) {
    return (double)(c.heaviest_rank_volume * ranks) / (double)c.decoded_volume - 1.0;
}

}  // namespace

namespace tdp {
// Full consistency check of a caller-supplied plan: it must be exactly what
// tdp_plan produces for its own dims / counts / overlaps / flags.
bool plan_is_valid(const tdp_plan_t* p) {
    if (!p) return false;
    tdp_plan_t q;
    int32_t dims[3] = {p->dims[0], p->dims[1], p->dims[2]};
    tdp_tile_count_cfg cfg = {{p->num_tiles[0], p->overlap[0]},
                              {p->num_tiles[1], p->overlap[1]},
                              {p->num_tiles[2], p->overlap[2]}};
    if (tdp_plan(dims, &cfg, p->flags, &q) != TDP_OK) return false;
    return std::memcmp(&q, p, sizeof(q)) == 0;
}
}  // namespace tdp

extern "C" {

tdp_status tdp_plan(const int32_t dims_fhw[3], const tdp_tile_count_cfg* cfg, uint32_t flags,
                    tdp_plan_t* out) {
    if (!dims_fhw || !cfg || !out) return TDP_ERR_INVALID_ARG;
    if (flags & ~TDP_PLAN_UPSTREAM_COMPAT) return TDP_ERR_INVALID_ARG;
    tdp_plan_t p;
    std::memset(&p, 0, sizeof(p));
    const tdp_dim_cfg* axes[3] = {&cfg->frames, &cfg->height, &cfg->width};
    for (int d = 0; d < 3; ++d) {
        tdp_status st = plan_axis(dims_fhw[d], *axes[d], flags, d, &p);
        if (st != TDP_OK) return st;
    }
    p.total_tiles = p.num_tiles[0] * p.num_tiles[1] * p.num_tiles[2];
    p.flags = flags;
    *out = p;
    return TDP_OK;
}

int64_t tdp_tile_offset(const tdp_plan_t* plan, int32_t t, int32_t B, int32_t C) {
    if (!plan || t < 0 || t >= plan->total_tiles || B < 0 || C < 0) return -1;
    int i_f, i_h, i_w;
    tdp::tile_coords(*plan, t, i_f, i_h, i_w);
    return (int64_t)B * C * tdp::tile_prefix_volume(*plan, i_f, i_h, i_w);
}

int64_t tdp_tiles_numel(const tdp_plan_t* plan, int32_t B, int32_t C) {
    if (!plan || B < 0 || C < 0) return -1;
    return (int64_t)B * C * tdp::total_volume(*plan);
}

tdp_status tdp_tile_box(const tdp_plan_t* plan, int32_t t, int32_t start[3], int32_t size[3]) {
    if (!plan || !start || !size || t < 0 || t >= plan->total_tiles) return TDP_ERR_INVALID_ARG;
    int i[3];
    tdp::tile_coords(*plan, t, i[0], i[1], i[2]);
    for (int d = 0; d < 3; ++d) {
        start[d] = plan->start[d][i[d]];
        size[d] = tdp::tile_size(*plan, d, i[d]);
    }
    return TDP_OK;
}

// Slab r of R: rows [floor(r H / R), floor((r + 1) H / R)); tiles owned
// round robin; a tile is needed where its rows meet the slab.
tdp_status tdp_shard_plan(const tdp_plan_t* plan, int32_t ranks, int32_t rank, int32_t* row0,
                          int32_t* row1, uint8_t* owned, uint8_t* needed) {
    if (!tdp::plan_is_valid(plan) || ranks < 1 || rank < 0 || rank >= ranks) return TDP_ERR_INVALID_ARG;
    const tdp_plan_t& p = *plan;
    const int64_t H = p.dims[1];
    const int r0 = static_cast<int>(H * rank / ranks), r1 = static_cast<int>(H * (rank + 1) / ranks);
    if (row0) *row0 = r0;
    if (row1) *row1 = r1;
    for (int t = 0; t < p.total_tiles; ++t) {
        int i_f, i_h, i_w;
        tdp::tile_coords(p, t, i_f, i_h, i_w);
        if (owned) owned[t] = (t % ranks == rank) ? 1 : 0;
        if (needed) needed[t] = (r0 < r1 && p.start[1][i_h] < r1 && p.end[1][i_h] > r0) ? 1 : 0;
    }
    return TDP_OK;
}

tdp_status tdp_plan_stats(const tdp_plan_t* plan, int32_t ranks, double* decoded_area,
                          int32_t* seams, double* tile_fraction, double* imbalance,
                          double* max_window_sum) {
    if (!tdp::plan_is_valid(plan) || ranks < 1) return TDP_ERR_INVALID_ARG;
    const tdp_plan_t& p = *plan;
    double latent = 1.0, area = 1.0;
    for (int d = 0; d < 3; ++d) {
        latent *= p.dims[d];
        area *= (double)p.prefix[d][p.num_tiles[d]] / p.dims[d];
    }
    if (decoded_area) *decoded_area = area;
    if (seams) {
        int64_t s = 0;
        for (int a = 0; a < 3; ++a) {
            int64_t others = 1;
            for (int b = 0; b < 3; ++b)
                if (b != a) others *= p.num_tiles[b];
            s += (int64_t)(p.num_tiles[a] - 1) * others;
        }
        *seams = (int32_t)s;
    }
    int64_t largest = 0, total = 0;
    std::vector<int64_t> per_rank(ranks, 0);
    for (int t = 0; t < p.total_tiles; ++t) {
        int i_f, i_h, i_w;
        tdp::tile_coords(p, t, i_f, i_h, i_w);
        const int64_t v = (int64_t)tdp::tile_size(p, 0, i_f) * tdp::tile_size(p, 1, i_h) * tdp::tile_size(p, 2, i_w);
        largest = std::max(largest, v);
        total += v;
        per_rank[t % ranks] += v;
    }
    if (tile_fraction) *tile_fraction = (double)largest / latent;
    if (imbalance) {
        const int64_t heavy = *std::max_element(per_rank.begin(), per_rank.end());
        *imbalance = (double)heavy * ranks / (double)total - 1.0;
    }
    if (max_window_sum) {
        // The 3-D sum is the product of the per-axis sums (all non-negative),
        // so its maximum is the product of the per-axis maxima.
        double m = 1.0;
        for (int d = 0; d < 3; ++d) {
            const std::vector<int64_t> s = axis_sum_numerators(p, d);
            const double o1 = p.overlap[d] + 1.0;
            m *= (double)*std::max_element(s.begin(), s.end()) / (o1 * o1);
        }
        *max_window_sum = m;
    }
    return TDP_OK;
}

tdp_status tdp_balanced_tile_split(int32_t ranks, int32_t* h_tiles, int32_t* w_tiles) {
    if (ranks < 1 || !h_tiles || !w_tiles) return TDP_ERR_INVALID_ARG;
    int32_t h = 1;
    for (int64_t d = 1; d * d <= ranks; ++d)
        if (ranks % d == 0) h = (int32_t)d;
    *h_tiles = h;
    *w_tiles = ranks / h;
    return TDP_OK;
}

tdp_status tdp_search_layouts(const int32_t dims_fhw[3], int32_t ranks, const tdp_dim_cfg* frames,
                              int32_t overlap_h, int32_t overlap_w, uint32_t flags, tdp_layout_candidate* out,
                              int32_t capacity, int32_t* count) {
    if (!dims_fhw || !frames || !count || ranks < 1 || capacity < 0 || (capacity > 0 && !out)) return TDP_ERR_INVALID_ARG;
    if (flags & ~(TDP_PLAN_UPSTREAM_COMPAT | TDP_SEARCH_NO_LIMITS)) return TDP_ERR_INVALID_ARG;
    const bool limits = !(flags & TDP_SEARCH_NO_LIMITS);
    const uint32_t plan_flags = flags & TDP_PLAN_UPSTREAM_COMPAT;
    const int32_t H = dims_fhw[1], W = dims_fhw[2];
    *count = 0;
    std::vector<tdp_layout_candidate> cands;
    if (!(limits && std::min(H, W) < std::max(16, ranks))) {
        const int64_t lo = std::max(2, ranks), hi = 4LL * ranks;
        const int64_t nf = std::max(1, frames->num_tiles);
        for (int32_t n_h = 1; n_h <= std::min(H, TDP_MAX_PER_AXIS) && nf * n_h <= hi; ++n_h) {
            for (int32_t n_w = 1; n_w <= std::min(W, TDP_MAX_PER_AXIS) && nf * n_h * n_w <= hi; ++n_w) {
                if (nf * n_h * n_w < lo) continue;
                const tdp_tile_count_cfg cfg = {*frames, {n_h, n_h > 1 ? overlap_h : 0}, {n_w, n_w > 1 ? overlap_w : 0}};
                tdp_plan_t p;
                if (tdp_plan(dims_fhw, &cfg, plan_flags, &p) != TDP_OK) continue;   // unsupported window
                if (limits) {
                    // overlap >= a quarter of the window (stride + overlap) on every tiled spatial axis
                    bool ok = true;
                    for (int d = 1; d < 3; ++d)
                        if (p.num_tiles[d] > 1 && 4LL * p.overlap[d] < (int64_t)p.end[d][0] - p.start[d][0]) ok = false;
                    if (!ok) continue;
                }
                tdp_layout_candidate c;
                std::memset(&c, 0, sizeof(c));
                std::vector<int64_t> per_rank(ranks, 0);
                for (int t = 0; t < p.total_tiles; ++t) {
                    int i_f, i_h, i_w;
                    tdp::tile_coords(p, t, i_f, i_h, i_w);
                    const int64_t v =
                        (int64_t)tdp::tile_size(p, 0, i_f) * tdp::tile_size(p, 1, i_h) * tdp::tile_size(p, 2, i_w);
                    c.window_volume = std::max(c.window_volume, v);
                    c.decoded_volume += v;
                    per_rank[t % ranks] += v;
                }
                c.heaviest_rank_volume = *std::max_element(per_rank.begin(), per_rank.end());
                for (int d = 0; d < 3; ++d) {
                    c.num_tiles[d] = p.num_tiles[d];
                    c.overlap[d] = p.overlap[d];
                }
                c.seams = (p.num_tiles[0] - 1) * p.num_tiles[1] * p.num_tiles[2] +
                          (p.num_tiles[1] - 1) * p.num_tiles[0] * p.num_tiles[2] +
                          (p.num_tiles[2] - 1) * p.num_tiles[0] * p.num_tiles[1];
                cands.push_back(c);
            }
        }
    }
    std::vector<int> front;
    for (size_t i = 0; i < cands.size(); ++i) {
        bool beaten = false;
        for (size_t j = 0; j < cands.size() && !beaten; ++j) beaten = beats(cands[j], cands[i]);
        cands[i].role = beaten ? TDP_ROLE_DOMINATED : TDP_ROLE_FRONTIER;
        if (!beaten) front.push_back((int)i);
    }
    if (!front.empty()) {
        auto pick = [&](auto better) {   // first frontier member still marked FRONTIER under `better`
            int best = -1;
            for (int i : front)
                if (cands[i].role == TDP_ROLE_FRONTIER && (best < 0 || better(cands[i], cands[best]))) best = i;
            return best;
        };
        const int coarse = pick([](const tdp_layout_candidate& a, const tdp_layout_candidate& b) {
            return a.window_volume != b.window_volume ? a.window_volume > b.window_volume : before_on_ties(a, b);
        });
        cands[coarse].role = TDP_ROLE_COARSE;
        const int fine = pick([](const tdp_layout_candidate& a, const tdp_layout_candidate& b) {
            return a.window_volume != b.window_volume ? a.window_volume < b.window_volume : before_on_ties(a, b);
        });
        if (fine >= 0) {
            cands[fine].role = TDP_ROLE_FINE;
            // worst of the three scores, each divided by its largest value on the frontier
            int64_t top_w = 0, top_d = 0;
            double top_i = 0.0;
            for (int i : front) {
                top_w = std::max(top_w, cands[i].window_volume);
                top_d = std::max(top_d, cands[i].decoded_volume);
                top_i = std::max(top_i, imbalance_of(cands[i], ranks));
            }
            auto score = [&](const tdp_layout_candidate& c) {
                const double s_i = top_i > 0.0 ? imbalance_of(c, ranks) / top_i : 0.0;
                return std::max(std::max((double)c.window_volume / (double)top_w,
                                         (double)c.decoded_volume / (double)top_d), s_i);
            };
            const int balanced = pick([&](const tdp_layout_candidate& a, const tdp_layout_candidate& b) {
                const double sa = score(a), sb = score(b);
                return sa != sb ? sa < sb : before_on_ties(a, b);
            });
            if (balanced >= 0) cands[balanced].role = TDP_ROLE_BALANCED;
        }
    }
    *count = (int32_t)cands.size();
    for (int32_t i = 0; i < std::min<int32_t>(capacity, *count); ++i) out[i] = cands[i];
    return TDP_OK;
}

size_t tdp_plan_struct_size(void) { return sizeof(tdp_plan_t); }

const char* tdp_status_str(tdp_status status) {
    switch (status) {
        case TDP_OK: return "ok";
        case TDP_ERR_INVALID_ARG: return "invalid argument";
        case TDP_ERR_GUARD: return "overlap * (num_tiles + 1) > dim: tile windows would not sum to 1";
        case TDP_ERR_TOO_MANY_TILES: return "more than TDP_MAX_PER_AXIS tiles on an axis";
        case TDP_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
        case TDP_ERR_CUDA: return "CUDA error";
        case TDP_ERR_UNSUPPORTED: return "shape not supported by the kernels (see the call)";
    }
    return "unknown status";
}

}  // extern "C"
