// Chunk planner of libattn (host only, integer-exact).
//
// FLOPs-balanced boundaries (SPPO §3.2 "Imbalanced GPU computation across
// subsequences": later tokens carry more attention work, so chunks start long
// and get shorter; InfiniPipe Eq. (1): chunk cost alpha1((C+s)^2 - C^2)).
// Equal quadratic cost gives b_k = L*sqrt(k/N); the plan rounds it to the
// nearest multiple of 128 (ties up). With m = b_k/128, "nearest, ties up" is
// the largest m >= 0 with m - 1/2 <= L*sqrt(k/N)/128, which for m >= 1 is
//     (2m - 1)^2 * 128^2 * N  <=  4 * L^2 * k,
// evaluated in 128-bit integers, so no floating point decides a boundary.
#include <algorithm>
#include <cmath>
#include <vector>

#include "attn_internal.h"

namespace {

using u128 = unsigned __int128;

bool flops_ok(int64_t m, int64_t L, int64_t k, int64_t N) {
    if (m <= 0) return true;
    u128 lhs = (u128)(2 * m - 1) * (u128)(2 * m - 1) * (u128)(128 * 128) * (u128)N;
    u128 rhs = (u128)4 * (u128)L * (u128)L * (u128)k;
    return lhs <= rhs;
}

int64_t flops_boundary(int64_t L, int64_t k, int64_t N) {
    // start near the answer, then settle on the largest m satisfying flops_ok
    double est = (double)L * std::sqrt((double)k / (double)N) / 128.0 + 0.5;
    int64_t m = std::max<int64_t>(0, (int64_t)est - 2);
    while (!flops_ok(m, L, k, N)) --m;
    while (flops_ok(m + 1, L, k, N)) ++m;
    return 128 * m;
}

// b_0..b_N for one sequence; false if not strictly increasing.
bool boundaries(int64_t L, int32_t N, int32_t mode, std::vector<int64_t>& b) {
    b.assign(N + 1, 0);
    for (int32_t k = 1; k < N; ++k) {
        if (mode == ATTN_PLAN_UNIFORM)
            b[k] = 128 * (((int64_t)k * L) / (128 * (int64_t)N));
        else
            b[k] = flops_boundary(L, k, N);
    }
    b[N] = L;
    for (int32_t i = 0; i < N; ++i)
        if (!(b[i] < b[i + 1])) return false;
    return true;
}

int32_t resplit_point(int32_t qb, int32_t qe) {
    int64_t n = (int64_t)qe - qb;
    int64_t m = qb + 128 * ((n + 128) / 256);  // floor(n/256 + 1/2)
    return (m > qb && m < qe) ? (int32_t)m : 0;
}

bool valid_mode(int32_t mode) {
    return mode == ATTN_PLAN_UNIFORM || mode == ATTN_PLAN_FLOPS || mode == ATTN_PLAN_FLOPS_RESPLIT_EDGES;
}

void apply_resplit(std::vector<attn_chunk>& c) {
    if (c.empty()) return;
    c.front().kv_split = resplit_point(c.front().q_begin, c.front().q_end);
    c.back().kv_split = resplit_point(c.back().q_begin, c.back().q_end);
}

int emit(const std::vector<attn_chunk>& c, attn_chunk* out, int32_t cap, int32_t* n_out) {
    if ((int64_t)c.size() > cap) {
        if (n_out) *n_out = (int32_t)c.size();
        return ATTN_E_CAPACITY;
    }
    std::copy(c.begin(), c.end(), out);
    *n_out = (int32_t)c.size();
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_plan(int64_t L, int32_t N, int32_t mode, attn_chunk* out, int32_t cap,
                         int32_t* n_out) {
    if (!n_out || (!out && cap > 0) || cap < 0) return ATTN_E_INVAL;
    if (L <= 0 || L > INT32_MAX || N <= 0 || !valid_mode(mode)) return ATTN_E_INVAL;
    std::vector<int64_t> b;
    if (!boundaries(L, N, mode, b)) return ATTN_E_INVAL;
    std::vector<attn_chunk> c(N);
    for (int32_t i = 0; i < N; ++i) c[i] = attn_chunk{(int32_t)b[i], (int32_t)b[i + 1], 0, 0};
    if (mode == ATTN_PLAN_FLOPS_RESPLIT_EDGES) apply_resplit(c);
    return emit(c, out, cap, n_out);
}

extern "C" int attn_plan_varlen(const int64_t* cu, int32_t ndocs, int32_t max_chunk_tokens,
                                int32_t mode, attn_chunk* out, int32_t cap, int32_t* n_out) {
    if (!n_out || !cu || (!out && cap > 0) || cap < 0) return ATTN_E_INVAL;
    if (ndocs <= 0 || max_chunk_tokens <= 0 || !valid_mode(mode)) return ATTN_E_INVAL;
    if (cu[0] != 0 || cu[ndocs] > INT32_MAX) return ATTN_E_INVAL;
    std::vector<attn_chunk> c;
    std::vector<int64_t> b;
    int32_t rule = mode == ATTN_PLAN_UNIFORM ? ATTN_PLAN_UNIFORM : ATTN_PLAN_FLOPS;
    for (int32_t d = 0; d < ndocs; ++d) {
        int64_t s = cu[d], e = cu[d + 1];
        if (e < s) return ATTN_E_INVAL;
        int64_t Ld = e - s;
        if (Ld == 0) continue;
        int64_t Nd = (Ld + max_chunk_tokens - 1) / max_chunk_tokens;
        if (!boundaries(Ld, (int32_t)Nd, rule, b)) return ATTN_E_INVAL;
        for (int64_t i = 0; i < Nd; ++i)
            c.push_back(attn_chunk{(int32_t)(s + b[i]), (int32_t)(s + b[i + 1]), (int32_t)s, 0});
    }
    if (mode == ATTN_PLAN_FLOPS_RESPLIT_EDGES) apply_resplit(c);
    return emit(c, out, cap, n_out);
}

// ---------------------------------------------------------------------------
// InfiniPipe Algorithm 1, "Workload-Balanced Sequence Chunking" (§III-B), on
// one GPU. Chunk cost by Eq. (1) with N = d_p = 1 and no all-to-all term:
// beta1 plus, per slice of s tokens after C context tokens,
// alpha1((C+s)^2 - C^2) + alpha2 s. Steps:
//   1. mesh: the longest sequence cut into K slices of equal cost, each
//      boundary the multiple of 128 nearest to the equal-cost point (ties up);
//   2. every sequence longer than the next mesh slice takes it (split chunks);
//      the rest is its tail slice; sequences no longer than the first mesh
//      slice are short;
//   3. one bucket per tail slice; short sequences from the most expensive
//      down, each into the first bucket (by increasing time per token) within
//      the time threshold T_t and token threshold T_m; a new bucket when even
//      the emptiest bucket has no room; T_t loosened to the least time among
//      buckets with room (plus the sequence's time) when no bucket fits.
// T_t starts at the costliest mesh slice; T_m is the caller's token capacity.
// Costs are float64 with the integer parts formed first, in a fixed order.
namespace {

struct IpCost {
    double a1, a2, b1;
    double slice_time(int64_t C, int64_t s) const {
        const int64_t quad = (C + s) * (C + s) - C * C;
        return a1 * (double)quad + a2 * (double)s;
    }
    double prefix(int64_t b) const { return a1 * (double)(b * b) + a2 * (double)b; }
};

struct IpMember {
    int32_t seq;
    int64_t ctx, len;
};

struct IpBucket {
    int32_t order;
    std::vector<IpMember> members;
    double tot_time;
    int64_t tot_tokens;
};

// Boundaries b_0..b_K of the mesh; false if they are not strictly increasing.
bool ip_mesh(int64_t Lmax, int32_t K, const IpCost& c, std::vector<int64_t>& b) {
    const double total = c.prefix(Lmax);
    b.assign(K + 1, 0);
    for (int32_t k = 1; k < K; ++k) {
        const double target = (double)k * total;
        // largest m with K * cost(128 m - 64) <= k * cost(Lmax); the test is
        // monotone in m, so a bisection finds what a scan from m = 0 would
        int64_t lo = 0, hi = Lmax / 128 + 2;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) / 2;
            if ((double)K * c.prefix(128 * mid - 64) <= target)
                lo = mid;
            else
                hi = mid - 1;
        }
        b[k] = 128 * lo;
    }
    b[K] = Lmax;
    for (int32_t i = 0; i < K; ++i)
        if (!(b[i] < b[i + 1])) return false;
    return true;
}

}  // namespace

extern "C" int attn_plan_infinipipe(const int64_t* seq_lens, int32_t nseq, int32_t K, int64_t token_cap,
                                    double alpha1, double alpha2, double beta1, attn_chunk* out, int32_t cap,
                                    int32_t* n_out, int32_t* call_off, int32_t call_cap, int32_t* n_calls) {
    if (!seq_lens || !n_out || !n_calls || nseq <= 0 || K <= 0 || token_cap <= 0) return ATTN_E_INVAL;
    if ((!out && cap > 0) || cap < 0 || (!call_off && call_cap > 0) || call_cap < 0) return ATTN_E_INVAL;
    if (!std::isfinite(alpha1) || !std::isfinite(alpha2) || !std::isfinite(beta1) || alpha1 < 0 || alpha2 < 0 ||
        beta1 < 0 || (alpha1 == 0 && alpha2 == 0))
        return ATTN_E_INVAL;
    std::vector<int64_t> start(nseq + 1, 0);
    int64_t Lmax = 0;
    for (int32_t i = 0; i < nseq; ++i) {
        if (seq_lens[i] < 0) return ATTN_E_INVAL;
        start[i + 1] = start[i] + seq_lens[i];
        if (start[i + 1] > INT32_MAX) return ATTN_E_INVAL;
        Lmax = std::max(Lmax, seq_lens[i]);
    }
    std::vector<std::vector<attn_chunk>> calls;
    if (Lmax > 0) {
        const IpCost c{alpha1, alpha2, beta1};
        std::vector<int64_t> b;
        if (!ip_mesh(Lmax, K, c, b)) return ATTN_E_INVAL;
        std::vector<int64_t> mesh(K);
        for (int32_t i = 0; i < K; ++i) mesh[i] = b[i + 1] - b[i];
        if (token_cap < mesh[0]) return ATTN_E_INVAL;
        double T_t = 0;
        for (int32_t i = 0; i < K; ++i) T_t = std::max(T_t, beta1 + c.slice_time(b[i], mesh[i]));
        const int64_t T_m = token_cap;

        // sharding by the mesh
        std::vector<std::vector<std::pair<int64_t, int64_t>>> slices(nseq);   // (ctx, len)
        std::vector<IpBucket> B;
        std::vector<int32_t> shorts;
        for (int32_t i = 0; i < nseq; ++i) {
            const int64_t L = seq_lens[i];
            if (L == 0) continue;
            int64_t rem = L, ctx = 0;
            for (int32_t j = 0; j < K && rem > mesh[j]; ++j) {
                slices[i].push_back({ctx, mesh[j]});
                ctx += mesh[j];
                rem -= mesh[j];
            }
            if (slices[i].empty()) {
                shorts.push_back(i);
            } else {
                IpBucket bk{(int32_t)B.size(), {IpMember{i, ctx, rem}}, beta1 + c.slice_time(ctx, rem), rem};
                B.push_back(bk);
            }
        }
        // short sequences from the most expensive down (ties: input order)
        std::stable_sort(shorts.begin(), shorts.end(), [&](int32_t x, int32_t y) {
            return c.slice_time(0, seq_lens[x]) > c.slice_time(0, seq_lens[y]);
        });
        std::vector<int32_t> byMetric;
        for (int32_t i : shorts) {
            const int64_t s = seq_lens[i];
            const double t = c.slice_time(0, s);
            for (;;) {
                int64_t min_tok = INT64_MAX;
                for (const IpBucket& bk : B) min_tok = std::min(min_tok, bk.tot_tokens);
                if (B.empty() || min_tok + s > T_m) {
                    B.push_back(IpBucket{(int32_t)B.size(), {IpMember{i, 0, s}}, beta1 + t, s});
                    break;
                }
                byMetric.resize(B.size());
                for (size_t x = 0; x < B.size(); ++x) byMetric[x] = (int32_t)x;
                std::sort(byMetric.begin(), byMetric.end(), [&](int32_t x, int32_t y) {
                    const double mx = B[x].tot_time / (double)B[x].tot_tokens;
                    const double my = B[y].tot_time / (double)B[y].tot_tokens;
                    return mx < my || (mx == my && B[x].order < B[y].order);
                });
                bool placed = false;
                for (int32_t x : byMetric) {
                    IpBucket& bk = B[x];
                    if (bk.tot_time + t <= T_t && bk.tot_tokens + s <= T_m) {
                        bk.members.push_back(IpMember{i, 0, s});
                        bk.tot_time = bk.tot_time + t;
                        bk.tot_tokens = bk.tot_tokens + s;
                        placed = true;
                        break;
                    }
                }
                if (placed) break;
                double least = 0;
                bool any = false;
                for (const IpBucket& bk : B)
                    if (bk.tot_tokens + s <= T_m && (!any || bk.tot_time < least)) {
                        least = bk.tot_time;
                        any = true;
                    }
                T_t = least + t;
            }
        }
        // split chunks by slice index, then the buckets in creation order
        size_t depth = 0;
        for (int32_t i = 0; i < nseq; ++i) depth = std::max(depth, slices[i].size());
        for (size_t j = 0; j < depth; ++j)
            for (int32_t i = 0; i < nseq; ++i)
                if (j < slices[i].size()) {
                    const int64_t s0 = start[i] + slices[i][j].first;
                    calls.push_back({attn_chunk{(int32_t)s0, (int32_t)(s0 + slices[i][j].second), (int32_t)start[i], 0}});
                }
        for (const IpBucket& bk : B) {
            std::vector<attn_chunk> v;
            for (const IpMember& m : bk.members) {
                const int64_t s0 = start[m.seq] + m.ctx;
                v.push_back(attn_chunk{(int32_t)s0, (int32_t)(s0 + m.len), (int32_t)start[m.seq], 0});
            }
            std::sort(v.begin(), v.end(), [](const attn_chunk& x, const attn_chunk& y) { return x.q_begin < y.q_begin; });
            calls.push_back(v);
        }
    }
    int64_t total = 0;
    for (const auto& v : calls) total += (int64_t)v.size();
    if (total > cap || (int64_t)calls.size() + 1 > call_cap) {
        *n_out = (int32_t)total;
        *n_calls = (int32_t)calls.size();
        return ATTN_E_CAPACITY;
    }
    int32_t pos = 0;
    call_off[0] = 0;
    for (size_t x = 0; x < calls.size(); ++x) {
        for (const attn_chunk& ch : calls[x]) out[pos++] = ch;
        call_off[x + 1] = pos;
    }
    *n_out = pos;
    *n_calls = (int32_t)calls.size();
    return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Re-split of a chunk's key range [cb, qe) into P parts with equal numbers of
// visible (query, key) pairs of its queries [qb, qe) (SPPO §4 multiplexing,
// read as a key/value split; Table 3 for the number of parts). The keys before
// K carry pairs(K) = A*n + B*n - B(B-1)/2 with n = qe - qb, A = min(K, qb) - cb
// context keys (seen by every query) and B = max(0, K - qb) of the chunk's own
// keys (key j seen by the queries t >= j). Boundary k_p is cb + 128 m with m
// the number of half-steps cb + 128 j - 64 (j >= 1, not past qe) where
// P * pairs <= p * pairs(qe): the multiple of 128 nearest to the equal-pair
// point, ties up. 128-bit integers throughout.
namespace {

using i128 = __int128;

i128 key_pairs_before(int64_t qb, int64_t qe, int64_t cb, int64_t K) {
    const i128 n = qe - qb;
    const i128 A = std::min(K, qb) - cb;
    const i128 B = std::max<int64_t>(0, K - qb);
    return A * n + B * n - B * (B - 1) / 2;
}

}  // namespace

namespace attn {

bool resplit_bounds(int32_t qb, int32_t qe, int32_t cb, int32_t P, std::vector<int32_t>& k) {
    if (P < 2 || P > 64 || !(cb <= qb && qb < qe)) return false;
    const i128 W = key_pairs_before(qb, qe, cb, qe);
    k.assign(P + 1, cb);
    for (int32_t p = 1; p < P; ++p) {
        // the test is monotone in m: bisection finds what a scan from m = 0 finds
        int64_t lo = 0, hi = ((int64_t)qe - cb + 64) / 128 + 1;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) / 2;
            const int64_t half = (int64_t)cb + 128 * mid - 64;
            if (half <= qe && (i128)P * key_pairs_before(qb, qe, cb, half) <= (i128)p * W)
                lo = mid;
            else
                hi = mid - 1;
        }
        k[p] = (int32_t)(cb + 128 * lo);
    }
    k[P] = qe;
    for (int32_t i = 0; i < P; ++i)
        if (!(k[i] < k[i + 1])) return false;
    return true;
}

}  // namespace attn

extern "C" int attn_plan_multiplex(int64_t L, int32_t N, int32_t PP, attn_chunk* out, int32_t cap,
                                   int32_t* n_out) {
    if (!n_out || (!out && cap > 0) || cap < 0) return ATTN_E_INVAL;
    if (L <= 0 || L > INT32_MAX || N <= 0 || PP <= 0) return ATTN_E_INVAL;
    std::vector<int64_t> b;
    if (!boundaries(L, N, ATTN_PLAN_FLOPS, b)) return ATTN_E_INVAL;
    std::vector<attn_chunk> c(N);
    std::vector<int32_t> k;
    for (int32_t i = 0; i < N; ++i) {
        c[i] = attn_chunk{(int32_t)b[i], (int32_t)b[i + 1], 0, 0};
        const int32_t want = PP - std::min(i, N - 1 - i);
        for (int32_t P = std::min(want, 64); P >= 2; --P)
            if (attn::resplit_bounds(c[i].q_begin, c[i].q_end, 0, P, k)) {
                c[i].kv_split = -P;
                break;
            }
    }
    return emit(c, out, cap, n_out);
}
