// Layout planning for one FSDP unit.
//
// FLAT  -- the FSDP1 FlatParameter: parameters flattened row-major and
//          concatenated in order ("PyTorch FSDP: Experiences on Scaling Fully
//          Sharded Data Parallel", section 3.2.1, Figure 3); rank k owns
//          [floor(kP/N), floor((k+1)P/N)) ("FSDP Architecture", the GPU-k
//          boundary formula).  One segment per non-empty rank.
// DIM0  -- FSDP2 Shard(0): every parameter chunked along dim 0 with
//          torch.chunk semantics, ceil(m/N) rows per chunk ("FSDP (Fully
//          Sharded Data Parallel)", FSDP1 vs FSDP2; "FSDP Under The Hood",
//          section 2).  One segment per (rank, parameter) with a non-empty
//          chunk, in parameter order within a rank.
// FLAT_PADDED -- the FlatParameter right-padded to a multiple of N and cut
//          into N chunks of ceil(P/N) ("PyTorch FSDP ...", section 3.2.1,
//          Figure 3); rank k's real elements are [min(kc,P), min((k+1)c,P)) and
//          its chunk ends with c - len zero padding elements, stored in its arena.
//
// Device arenas: each rank's arena starts at a multiple of kAlign in a slab
// shared by all ranks, and every segment is placed so that its arena slot is
// congruent to its global index modulo kAlign; the gaps are zero pads.
#include "plan.hpp"

#include <algorithm>

namespace fsdp {

namespace {

int64_t floor_div_mul(int64_t k, int64_t P, int64_t N) {
    // floor(k*P/N) without overflow for k <= N <= 1024 and P < 2^62
    __int128 x = static_cast<__int128>(k) * static_cast<__int128>(P);
    return static_cast<int64_t>(x / N);
}

int64_t pos_mod(int64_t a, int64_t m) {
    int64_t r = a % m;
    return r < 0 ? r + m : r;
}

int64_t round_up(int64_t a, int64_t m) { return (a + m - 1) / m * m; }

}  // namespace

int build_plan(int nparams, const int* ndims, const int64_t* dims, int layout, int N,
               Plan* out, std::string* err) {
    if (nparams < 1 || ndims == nullptr || out == nullptr) {
        *err = "nparams must be >= 1 and ndims/out non-null";
        return FSDP_E_INVALID_ARG;
    }
    if (layout != FSDP_LAYOUT_FLAT && layout != FSDP_LAYOUT_DIM0 && layout != FSDP_LAYOUT_FLAT_PADDED) {
        *err = "layout must be FSDP_LAYOUT_FLAT, FSDP_LAYOUT_DIM0 or FSDP_LAYOUT_FLAT_PADDED";
        return FSDP_E_INVALID_ARG;
    }
    if (N < 1 || N > kMaxRanks) {
        *err = "num_ranks must be in [1, 1024]";
        return FSDP_E_INVALID_ARG;
    }
    Plan plan;
    plan.layout = layout;
    plan.N = N;
    plan.params.resize(nparams);
    int64_t total_dims = 0;
    for (int p = 0; p < nparams; ++p) {
        if (ndims[p] < 0 || ndims[p] > kMaxDims) {
            *err = "ndims[p] must be in [0, 8]";
            return FSDP_E_INVALID_ARG;
        }
        total_dims += ndims[p];
    }
    if (total_dims > 0 && dims == nullptr) {
        *err = "dims is null";
        return FSDP_E_INVALID_ARG;
    }
    const int64_t kMaxNumel = int64_t(1) << 50;
    int64_t di = 0, off = 0;
    for (int p = 0; p < nparams; ++p) {
        ParamInfo& pi = plan.params[p];
        int64_t n = 1, rows = 1, row_len = 1;
        for (int d = 0; d < ndims[p]; ++d) {
            int64_t v = dims[di + d];
            if (v < 0 || v > kMaxNumel) {
                *err = "dimension out of range";
                return FSDP_E_INVALID_ARG;
            }
            if (v != 0 && n > kMaxNumel / v) {
                *err = "parameter too large";
                return FSDP_E_INVALID_ARG;
            }
            n *= v;
            if (d == 0) rows = v; else row_len *= v;
        }
        di += ndims[p];
        if (ndims[p] == 0) { rows = 1; row_len = 1; }
        pi.numel = n;
        pi.rows = rows;
        pi.row_len = row_len;
        pi.offset = off;
        off += n;
        if (off > kMaxNumel) {
            *err = "unit too large";
            return FSDP_E_INVALID_ARG;
        }
    }
    plan.P = off;
    if (plan.P < 1) {
        *err = "the unit has no elements";
        return FSDP_E_INVALID_ARG;
    }

    plan.shard_len.assign(N, 0);
    plan.layout_pad.assign(N, 0);
    plan.arena_len.assign(N, 0);
    plan.arena_base.assign(N, 0);
    plan.rank_first_seg.assign(N + 1, 0);
    for (int k = 0; k < N; ++k) {
        plan.rank_first_seg[k] = static_cast<int64_t>(plan.segs.size());
        int64_t cursor = 0, packed = 0;
        auto place = [&](int32_t param, int64_t g, int64_t len) {
            fsdp_segment s;
            s.rank = k;
            s.param = param;
            s.global_off = g;
            s.shard_off = packed;
            s.arena_off = cursor + pos_mod(g - cursor, kAlign);
            s.len = len;
            cursor = s.arena_off + len;
            packed += len;
            plan.segs.push_back(s);
        };
        if (layout == FSDP_LAYOUT_FLAT) {
            int64_t a = floor_div_mul(k, plan.P, N);
            int64_t b = floor_div_mul(k + 1, plan.P, N);
            if (b > a) place(-1, a, b - a);
        } else if (layout == FSDP_LAYOUT_FLAT_PADDED) {
            const int64_t c = (plan.P + N - 1) / N;
            const int64_t a = std::min<int64_t>(c * k, plan.P);
            const int64_t b = std::min<int64_t>(c * (k + 1), plan.P);
            if (b > a) place(-1, a, b - a);
            plan.layout_pad[k] = c - (b - a);
            cursor += plan.layout_pad[k];   // the chunk's zero padding
        } else {
            for (int p = 0; p < nparams; ++p) {
                const ParamInfo& pi = plan.params[p];
                if (pi.numel == 0) continue;
                int64_t c = (pi.rows + N - 1) / N;   // torch.chunk: ceil(m/N) rows
                int64_t r0 = std::min<int64_t>(c * k, pi.rows);
                int64_t r1 = std::min<int64_t>(c * (k + 1), pi.rows);
                if (r1 > r0) place(p, pi.offset + r0 * pi.row_len, (r1 - r0) * pi.row_len);
            }
        }
        plan.shard_len[k] = packed;
        plan.arena_len[k] = round_up(cursor, kAlign);
    }
    plan.rank_first_seg[N] = static_cast<int64_t>(plan.segs.size());
    int64_t base = 0;
    for (int k = 0; k < N; ++k) {
        plan.arena_base[k] = base;
        base += plan.arena_len[k];
    }
    plan.slab_len = base;
    *out = std::move(plan);
    return FSDP_OK;
}

void build_tiles(const Plan& plan, std::vector<Tile>* tiles) {
    tiles->clear();
    for (const fsdp_segment& s : plan.segs) {
        int64_t g = s.global_off;
        int64_t a = plan.arena_base[s.rank] + s.arena_off;
        int64_t left = s.len;
        while (left > 0) {
            int64_t next = (g / kTile + 1) * kTile;
            int64_t n = std::min(left, next - g);
            tiles->push_back(Tile{g, a, static_cast<int32_t>(n), 0});
            g += n;
            a += n;
            left -= n;
        }
    }
}

void build_load_tiles(const Plan& plan, std::vector<Tile>* tiles) {
    std::vector<Tile> base;
    build_tiles(plan, &base);
    tiles->clear();
    // parameter containing global index g: last p with offset <= g and numel > 0
    auto param_of = [&](int64_t g) {
        int lo = 0, hi = static_cast<int>(plan.params.size()) - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (plan.params[mid].offset <= g) lo = mid; else hi = mid - 1;
        }
        while (plan.params[lo].numel == 0) --lo;   // zero-size params share the next offset
        return lo;
    };
    for (const Tile& t : base) {
        int64_t g = t.g, s = t.s, left = t.len;
        while (left > 0) {
            int p = param_of(g);
            int64_t end = plan.params[p].offset + plan.params[p].numel;
            int64_t n = std::min(left, end - g);
            tiles->push_back(Tile{g, s, static_cast<int32_t>(n), p});
            g += n;
            s += n;
            left -= n;
        }
    }
}

}  // namespace fsdp
