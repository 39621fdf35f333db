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

#include "attn.h"

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
