"""Pins of the planner oracle (no GPU).

The FLOPS rule is checked against a brute-force nearest-multiple search done
with exact integer squares (a different route from the oracle's decimal square
roots), against the FLOP-balance bound that rounding to 128 allows, and against
the stored expected plans in tests/golden/plans.json.
"""
import json
from decimal import Decimal, ROUND_FLOOR, localcontext
import math
import os
import random

import pytest

from oracle import plan as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plans.json")


def brute_nearest_multiple(L, k, N, step=128):
    """Nearest multiple of `step` to L*sqrt(k/N), ties up, by linear scan with
    exact comparisons: a*step <= L*sqrt(k/N)  <=>  (a*step)^2 * N <= L^2 * k."""
    a = 0
    while ((a + 1) * step) ** 2 * N <= L * L * k:
        a += 1
    # x in [a*step, (a+1)*step); pick a+1 when x >= a*step + step/2
    half2 = (2 * a * step + step) ** 2 * N          # (2*(a*step + step/2))^2 * N
    return (a + 1) * step if half2 <= 4 * L * L * k else a * step


@pytest.mark.parametrize("L", [1024, 32768, 131072, 1 << 20, 1000, 4097, 65537])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8, 16, 33, 64])
def test_flops_rule_matches_brute_force(L, N):
    try:
        b = P.boundaries(L, N, P.FLOPS)
    except P.PlanError:
        # the rule must really collapse: some brute-force boundary repeats
        bb = [0] + [brute_nearest_multiple(L, k, N) for k in range(1, N)] + [L]
        assert any(not bb[i] < bb[i + 1] for i in range(N))
        return
    assert b[0] == 0 and b[-1] == L and len(b) == N + 1
    for k in range(1, N):
        assert b[k] == brute_nearest_multiple(L, k, N), (L, N, k)


def test_flops_rule_random_lengths():
    rng = random.Random(7)
    for _ in range(300):
        L = rng.randint(128, 1 << 21)
        N = rng.randint(1, 64)
        try:
            b = P.boundaries(L, N, P.FLOPS)
        except P.PlanError:
            continue
        for k in range(1, N):
            assert b[k] == brute_nearest_multiple(L, k, N)


def test_tie_rounds_up():
    # L*sqrt(1/4) = 1344 = 10.5 * 128 exactly -> rounds up to 11 * 128
    assert P.boundaries(2688, 4, P.FLOPS)[1] == 1408
    assert brute_nearest_multiple(2688, 1, 4) == 1408


def test_flop_balance_bound():
    """Each boundary moves <= 64 tokens from L*sqrt(k/N); hence a chunk's pair
    count is within 64(b_i+b_{i+1}) + 4096 + L/2 of L(L+1)/(2N)."""
    for L, N in [(32768, 8), (131072, 16), (1 << 20, 64), (100000, 10)]:
        b = P.boundaries(L, N, P.FLOPS)
        target = L * (L + 1) / (2 * N)
        for i in range(N):
            pairs = P.causal_pairs(b[i], b[i + 1], 0)
            bound = 64 * (b[i] + b[i + 1]) + 4096 + L / 2
            assert abs(pairs - target) <= bound
        total = sum(P.causal_pairs(b[i], b[i + 1], 0) for i in range(N))
        assert total == L * (L + 1) // 2


def test_lengths_non_increasing_up_to_rounding():
    """Longer subsequences first, shorter later (SPPO §3.2); rounding each
    boundary to 128 can swap neighbours by at most 128 tokens."""
    for L, N in [(32768, 8), (131072, 16), (1 << 20, 64)]:
        b = P.boundaries(L, N, P.FLOPS)
        s = [b[i + 1] - b[i] for i in range(N)]
        for i in range(N - 1):
            assert s[i] >= s[i + 1] - 128
        assert s[0] > s[-1]


def test_known_plans():
    b = P.boundaries(32768, 8, P.FLOPS)
    assert b[:5] == [0, 11648, 16384, 20096, 23168]
    assert b[-3:] == [28416, 30592, 32768]
    b = P.boundaries(131072, 16, P.FLOPS)
    assert b[1] == 32768 and b[2] == 46336 and b[15] == 126848
    assert P.boundaries(1024, 4, P.UNIFORM) == [0, 256, 512, 768, 1024]


def test_uniform_rule():
    assert P.boundaries(1000, 3, P.UNIFORM) == [0, 256, 640, 1000]
    with pytest.raises(P.PlanError):
        P.boundaries(200, 3, P.UNIFORM)


def test_too_many_chunks_is_error():
    with pytest.raises(P.PlanError):
        P.boundaries(1024, 16, P.FLOPS)
    with pytest.raises(P.PlanError):
        P.boundaries(0, 1, P.FLOPS)


def test_resplit_point():
    assert P.resplit_point(0, 32768) == 16384
    assert P.resplit_point(126848, 131072) == 126848 + 128 * 17     # 4224/256 = 16.5 -> 17
    assert P.resplit_point(0, 128) == 0          # would land on q_end: no split
    assert P.resplit_point(0, 300) == 128        # floor(300/256 + 0.5) = 1
    c = P.plan(131072, 16, P.FLOPS_RESPLIT_EDGES)
    assert c[0] == (0, 32768, 0, 16384)
    assert c[-1][3] == 129024
    assert all(x[3] == 0 for x in c[1:-1])


def test_varlen_plan_structure():
    cu = [0, 5, 5, 40000, 40130, 100000]
    chunks = P.plan_varlen(cu, 16384, P.FLOPS)
    # contiguous partition of [0, T); every chunk lies inside one document
    assert chunks[0][0] == 0 and chunks[-1][1] == cu[-1]
    for a, b in zip(chunks, chunks[1:]):
        assert a[1] == b[0]
    for qb, qe, cb, m in chunks:
        d = max(i for i in range(len(cu) - 1) if cu[i] <= qb and cu[i + 1] > qb)
        assert cb == cu[d] and qe <= cu[d + 1]
    # doc of 39995 tokens -> ceil(39995/16384) = 3 chunks, FLOPS rule from its start
    doc = [c for c in chunks if c[2] == 5]
    assert len(doc) == 3
    assert [c[0] - 5 for c in doc] + [doc[-1][1] - 5] == P.boundaries(39995, 3, P.FLOPS)
    r = P.plan_varlen(cu, 16384, P.FLOPS_RESPLIT_EDGES)
    assert r[0][3] == 0            # first doc has 5 tokens: no split possible
    assert r[-1][3] != 0


def test_golden_plans():
    with open(GOLDEN) as f:
        gold = json.load(f)
    for name, g in gold.items():
        if "cu_seqlens" in g:
            got = P.plan_varlen(g["cu_seqlens"], g["max_chunk_tokens"], g["mode"])
        else:
            got = P.plan(g["L"], g["N"], g["mode"])
        assert [list(c) for c in got] == g["chunks"], name


# ---------------------------------------------------- re-split into P parts

def test_key_pairs_closed_form_matches_counting():
    rng = random.Random(3)
    for _ in range(300):
        cb = rng.randint(0, 300)
        qb = cb + rng.randint(0, 300)
        qe = qb + rng.randint(1, 300)
        K = rng.randint(cb, qe)
        brute = sum(1 for j in range(cb, K) for t in range(qb, qe) if j <= t)
        assert P.key_pairs_before(qb, qe, cb, K) == brute


def test_resplit_context_dominated_chunk_by_hand():
    """Chunk (4096, 4224) with context from 0: every context key is seen by all
    128 queries, the chunk's own keys by 128..1 of them. W = 4096*128 + 8256 =
    532544; the quarter points fall at keys 1040.1, 2080.3, 3120.4 (inside the
    uniform context), nearest multiples of 128: 1024, 2048, 3072."""
    assert P.key_pairs_before(4096, 4224, 0, 4224) == 532544
    assert P.resplit_boundaries(4096, 4224, 0, 4) == [0, 1024, 2048, 3072, 4224]


@pytest.mark.parametrize("L,Pn", [(32768, 2), (32768, 4), (131072, 3), (4096, 5), (20000, 2)])
def test_resplit_causal_chunk_closed_form(L, Pn):
    """A chunk with no context: key j is seen by L - j queries, so the keys
    before K carry K*L - K(K-1)/2 pairs and the equal-pair points are close to
    L*(1 - sqrt(1 - p/P)) (50-digit decimals); the rule lands on the multiple
    of 128 nearest to that, within one step when the point is near a half."""
    k = P.resplit_boundaries(0, L, 0, Pn)
    assert k[0] == 0 and k[-1] == L and len(k) == Pn + 1
    with localcontext() as ctx:
        ctx.prec = 50
        for p in range(1, Pn):
            x = Decimal(L) * (1 - (1 - Decimal(p) / Decimal(Pn)).sqrt())
            near = 128 * int((x / 128 + Decimal("0.5")).to_integral_value(rounding=ROUND_FLOOR))
            assert abs(k[p] - near) <= 128 and (k[p] == near or abs(x / 128 - int(x / 128) - Decimal("0.5")) < Decimal("0.01"))


def test_resplit_parts_balanced():
    rng = random.Random(9)
    for _ in range(200):
        cb = rng.randint(0, 5000)
        qb = cb + rng.randint(0, 20000)
        qe = qb + rng.randint(128, 20000)
        Pn = rng.randint(2, 6)
        try:
            k = P.resplit_boundaries(qb, qe, cb, Pn)
        except P.PlanError:
            continue
        W = P.key_pairs_before(qb, qe, cb, qe)
        n = qe - qb
        for p in range(Pn):
            part = P.key_pairs_before(qb, qe, cb, k[p + 1]) - P.key_pairs_before(qb, qe, cb, k[p])
            assert abs(part - W / Pn) <= 2 * 64 * n + n, (qb, qe, cb, Pn, p)


def test_resplit_errors_and_key_ranges():
    with pytest.raises(P.PlanError):
        P.resplit_boundaries(0, 200, 0, 4)          # too few 128-token steps
    with pytest.raises(P.PlanError):
        P.resplit_boundaries(0, 4096, 0, 1)
    assert P.key_ranges((0, 1000, 0, 0)) == [(0, 1000)]
    assert P.key_ranges((0, 1000, 0, 300)) == [(0, 300), (300, 1000)]
    k = P.resplit_boundaries(1000, 3000, 0, 3)
    assert P.key_ranges((1000, 3000, 0, -3)) == [(k[0], k[1]), (k[1], k[2]), (k[2], k[3])]


def test_plan_multiplex():
    """SPPO Table 3 with PP = 4 and N = 8: chunks 0 and 7 in four parts, 1 and 6
    in three, 2 and 5 in two, the middle ones whole."""
    c = P.plan_multiplex(131072, 8, 4)
    assert [x[3] for x in c] == [-4, -3, -2, 0, 0, -2, -3, -4]
    assert [x[:2] for x in c] == [(b0, b1) for b0, b1 in zip(P.boundaries(131072, 8, P.FLOPS),
                                                                P.boundaries(131072, 8, P.FLOPS)[1:])]
    assert [x[3] for x in P.plan_multiplex(131072, 8, 1)] == [0] * 8
    assert [x[3] for x in P.plan_multiplex(131072, 3, 3)] == [-3, -2, -3]
    # L = 1024, N = 4, PP = 4, worked by hand. Chunk 0 = (0, 512) has no context:
    # its equal-pair points for 4 parts, 512(1 - sqrt(1 - p/4)) = 68.6, 150, 256,
    # round to 128, 128, 256 and collapse; for 3 parts, 94 and 216 round to 128
    # and 256, so chunk 0 gets -3. Chunk 3 = (896, 1024) sees 896 context keys
    # (128 queries each) and its own 128 keys (128..1 queries): W = 122944, the
    # quarter points fall at keys 240.1, 480.3, 720.4 -> 256, 512, 768: -4.
    small = P.plan_multiplex(1024, 4, 4)
    assert small[0][3] == -3 and P.resplit_boundaries(0, 512, 0, 3) == [0, 128, 256, 512]
    assert small[3][3] == -4 and P.resplit_boundaries(896, 1024, 0, 4) == [0, 256, 512, 768, 1024]
