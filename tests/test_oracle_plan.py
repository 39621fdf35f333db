"""Pins of the planner oracle (no GPU).

The FLOPS rule is checked against a brute-force nearest-multiple search done
with exact integer squares (a different route from the oracle's decimal square
roots), against the FLOP-balance bound that rounding to 128 allows, and against
the stored expected plans in tests/golden/plans.json.
"""
import json
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
