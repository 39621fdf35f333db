"""Pins of the Algorithm 1 oracle (InfiniPipe §III-B), no GPU.

* The page's own example of sharding by a mesh {8K, 4K, 2K}.
* The mesh against the SPPO FLOPS rule (alpha2 = beta1 = 0) and against the
  equal-cost point solved with 50-digit decimal square roots.
* A packing worked out by hand from the algorithm's steps.
* The loosening reading: a bucket that is full of tokens never blocks.
* The bucket order: increasing tot_time/tot_tokens, ties to the older bucket.
* The starting threshold T_t: the costliest mesh slice, worked by hand.
* Invariants on random inputs: every token in exactly one chunk, one call
  never holds two slices of a sequence, at most one tail per bucket, token
  and time thresholds respected, split slices equal to the mesh.
"""
import random
from decimal import Decimal, ROUND_FLOOR, localcontext

import pytest

from oracle import infinipipe as IP
from oracle import plan as P


def test_page_example_sharding_by_mesh():
    """InfiniPipe §III-B: with a mesh {8K, 4K, 2K}, sequences of more than 12K
    tokens become an 8K and a 4K slice and a variable-length remainder."""
    K8, K4, K2 = 8192, 4096, 2048
    mesh = [K8, K4, K2]
    lengths = [14336, 13000, 12289, 12288, 10000, 8193, 8192, 100]
    parts = IP.split_by_mesh(lengths, mesh)
    assert parts[0] == ([(0, K8), (K8, K4)], (K8 + K4, 2048))      # the longest: its last slice is the tail
    assert parts[1] == ([(0, K8), (K8, K4)], (K8 + K4, 13000 - 12288))
    assert parts[2] == ([(0, K8), (K8, K4)], (K8 + K4, 1))
    assert parts[3] == ([(0, K8)], (K8, 4096))                     # exactly 12K: 8K + a 4K remainder
    assert parts[4] == ([(0, K8)], (K8, 10000 - K8))
    assert parts[5] == ([(0, K8)], (K8, 1))
    assert parts[6] == ([], None) and parts[7] == ([], None)       # short sequences


@pytest.mark.parametrize("L", [1024, 32768, 131072, 1000, 65537])
@pytest.mark.parametrize("K", [1, 2, 3, 7, 8])
def test_mesh_is_flops_rule_when_only_quadratic(L, K):
    cost = IP.Cost(alpha1=1.0, alpha2=0.0, beta1=0.0)
    try:
        want = P.boundaries(L, K, P.FLOPS)
    except P.PlanError:
        with pytest.raises(IP.PlanError):
            IP.split_longest(L, K, cost)
        return
    assert IP.split_longest(L, K, cost) == want


def decimal_boundary(L, k, K, a1, a2):
    """Nearest multiple of 128 (ties up) to the root of a1 b^2 + a2 b = (k/K)(a1 L^2 + a2 L),
    by the quadratic formula in 50-digit decimals."""
    with localcontext() as ctx:
        ctx.prec = 50
        A1, A2 = Decimal(a1), Decimal(a2)
        tgt = Decimal(k) / Decimal(K) * (A1 * L * L + A2 * L)
        if A1 == 0:
            x = tgt / A2
        else:
            x = (-A2 + (A2 * A2 + 4 * A1 * tgt).sqrt()) / (2 * A1)
        return 128 * int((x / 128 + Decimal("0.5")).to_integral_value(rounding=ROUND_FLOOR))


@pytest.mark.parametrize("a1,a2", [(1e-9, 3e-4), (2.5e-10, 1e-3), (1.0, 50000.0), (0.0, 1.0), (3.0, 1.0)])
def test_mesh_equal_cost_point(a1, a2):
    cost = IP.Cost(alpha1=a1, alpha2=a2, beta1=7.0)
    for L, K in [(131072, 8), (20000, 5), (4096, 3), (1 << 20, 16)]:
        b = IP.split_longest(L, K, cost)
        assert b[0] == 0 and b[-1] == L
        for k in range(1, K):
            assert b[k] == decimal_boundary(L, k, K, a1, a2), (L, K, k)
        if a2 > 0 and a1 > 0:
            # a linear term pulls the boundaries from the quadratic rule towards equal lengths
            flops = P.boundaries(L, K, P.FLOPS)
            assert all(128 * ((k * L // K) // 128) <= x <= y for k, (x, y) in enumerate(zip(b, flops)) if 0 < k < K)


def test_hand_worked_packing():
    """alpha1 = 1, alpha2 = beta1 = 0, lengths [1024, 300, 256, 200, 128, 100],
    K = 2, token capacity 1024, worked by hand:
      mesh: 1024*sqrt(1/2) = 724.1 -> 768; slices [768, 256], costs 589824 and
            458752, so T_t = 589824.
      seq 0 splits into (0, 768) and a tail (768, 256): bucket 0, time 458752.
      shorts by time: 300, 256, 200, 128, 100.
      300: 458752 + 90000 <= T_t -> bucket 0 (548752, 556 tokens).
      256: 548752 + 65536 > T_t; loosen T_t to 614288 -> bucket 0 (812 tokens).
      200: 614288 + 40000 > T_t; loosen to 654288 -> bucket 0 (1012 tokens).
      128: 1012 + 128 > 1024 even for the emptiest bucket -> new bucket 1.
      100: bucket 1 (metric 128) before bucket 0 (metric 646.5) -> bucket 1."""
    cost = IP.Cost(1.0, 0.0, 0.0)
    calls, info = IP.plan([1024, 300, 256, 200, 128, 100], 2, 1024, cost)
    assert info["mesh"] == [768, 256]
    assert info["T_t"] == 654288.0
    starts = [0, 1024, 1324, 1580, 1780, 1908, 2008]
    assert calls == [
        [(0, 768, 0, 0)],
        [(768, 1024, 0, 0), (1024, 1324, 1024, 0), (1324, 1580, 1324, 0), (1580, 1780, 1580, 0)],
        [(1780, 1908, 1780, 0), (1908, 2008, 1908, 0)],
    ]
    assert starts[-1] == 2008
    assert info["times"] == [589824.0, 654288.0, 16384.0 + 10000.0]


def test_loosening_skips_buckets_full_of_tokens():
    """The bucket with the least time has no room for the sequence's tokens:
    T_t is loosened to the least time among buckets that do have room."""
    cost = IP.Cost(1.0, 0.0, 0.0)
    a = IP.Bucket(order=0, tail=False, members=[(0, 0, 90)], tot_time=100.0, tot_tokens=90)
    b = IP.Bucket(order=1, tail=False, members=[(1, 0, 10)], tot_time=500.0, tot_tokens=10)
    T_t = IP.bfd([a, b], [(2, 20)], T_t=150.0, T_m=100, cost=cost)
    assert T_t == 500.0 + 400.0
    assert b.members[-1] == (2, 0, 20) and a.members == [(0, 0, 90)]


def test_bucket_order_is_increasing_time_per_token():
    """Algorithm 1 visits the buckets in increasing order of tot_time/tot_tokens
    and takes the first that fits: with two buckets that can both take the
    sequence, the one with less time per token receives it; equal ratios go
    to the older bucket."""
    cost = IP.Cost(1.0, 0.0, 0.0)                          # a 10-token sequence costs 100
    a = IP.Bucket(order=0, tail=False, members=[(0, 0, 50)], tot_time=500.0, tot_tokens=50)    # 10 per token
    b = IP.Bucket(order=1, tail=False, members=[(1, 0, 100)], tot_time=300.0, tot_tokens=100)  # 3 per token
    T_t = IP.bfd([a, b], [(2, 10)], T_t=1000.0, T_m=1000, cost=cost)
    assert T_t == 1000.0
    assert b.members[-1] == (2, 0, 10) and a.members == [(0, 0, 50)]
    assert (b.tot_time, b.tot_tokens) == (400.0, 110)
    c = IP.Bucket(order=0, tail=False, members=[(0, 0, 40)], tot_time=200.0, tot_tokens=40)    # 5 per token
    d = IP.Bucket(order=1, tail=False, members=[(1, 0, 20)], tot_time=100.0, tot_tokens=20)    # 5 per token
    IP.bfd([c, d], [(2, 10)], T_t=1000.0, T_m=1000, cost=cost)
    assert c.members[-1] == (2, 0, 10) and d.members == [(1, 0, 20)]


def test_threshold_starts_at_the_costliest_mesh_slice():
    """T_t starts at the largest modeled time of a mesh slice. Worked by hand
    with alpha1 = 1, alpha2 = beta1 = 0, lengths [1024, 800, 700, 100], K = 2,
    token capacity 2048:
      mesh [768, 256]; slice times 768^2 = 589824 and 1024^2 - 768^2 = 458752,
      so T_t = 589824.
      seq 0 -> (0, 768) and the tail (768, 256): bucket 0, time 458752, 256
      tokens (1792 per token). seq 1 -> (0, 768) and the tail (768, 32):
      bucket 1, time 800^2 - 768^2 = 50176, 32 tokens (1568 per token).
      700 (time 490000): bucket 1 first; 540176 <= T_t -> bucket 1.
      100 (time 10000): bucket 1 first (737.9 per token); 550176 <= T_t ->
      bucket 1.
    Starting at the cheapest slice (458752) would loosen T_t to 540176 for the
    700 and send the 100 to bucket 0."""
    cost = IP.Cost(1.0, 0.0, 0.0)
    calls, info = IP.plan([1024, 800, 700, 100], 2, 2048, cost)
    assert info["mesh"] == [768, 256] and info["T_t"] == 589824.0
    assert calls == [
        [(0, 768, 0, 0)],
        [(1024, 1792, 1024, 0)],
        [(768, 1024, 0, 0)],
        [(1792, 1824, 1024, 0), (1824, 2524, 1824, 0), (2524, 2624, 2524, 0)],
    ]
    assert info["times"] == [589824.0, 589824.0, 458752.0, 550176.0]


def random_case(rng):
    n = rng.randint(1, 30)
    lengths = [rng.choice([0, rng.randint(1, 300), rng.randint(1, 5000), rng.randint(1, 40000)]) for _ in range(n)]
    if max(lengths) == 0:
        lengths[0] = rng.randint(1, 40000)
    K = rng.randint(1, 6)
    cost = IP.Cost(rng.choice([1e-9, 2e-10, 1.0]), rng.choice([0.0, 1e-4, 3.0, 5e3]), rng.choice([0.0, 1e-3, 10.0]))
    cap = rng.choice([None, 40000, 60000, 100000])
    return lengths, K, cost, cap


def test_invariants_on_random_inputs():
    rng = random.Random(5)
    seen = 0
    for _ in range(400):
        lengths, K, cost, cap = random_case(rng)
        try:
            b = IP.split_longest(max(lengths), K, cost)
        except IP.PlanError:
            continue
        mesh = [b[i + 1] - b[i] for i in range(K)]
        cap = cap or mesh[0]
        if cap < mesh[0]:
            with pytest.raises(IP.PlanError):
                IP.plan(lengths, K, cap, cost)
            continue
        calls, info = IP.plan(lengths, K, cap, cost)
        seen += 1
        starts = [0]
        for L in lengths:
            starts.append(starts[-1] + L)
        doc_of = {}
        for d in range(len(lengths)):
            for t in range(starts[d], starts[d + 1]):
                doc_of[t] = d
        covered = [0] * starts[-1]
        seq_done = {}
        for ci, call in enumerate(calls):
            docs = [doc_of[c[0]] for c in call]
            assert len(docs) == len(set(docs)), "two slices of one sequence in a call"
            assert call == sorted(call)
            for j in range(1, len(call)):
                assert call[j][2] >= call[j - 1][1]            # disjoint key ranges
            tails = 0
            for qb, qe, cb, m in call:
                d = doc_of[qb]
                assert m == 0 and cb == starts[d] and starts[d] <= qb < qe <= starts[d + 1]
                assert qb == seq_done.get(d, starts[d]), "slices of a sequence out of order"
                seq_done[d] = qe
                for t in range(qb, qe):
                    covered[t] += 1
                if qb > cb:
                    tails += 1
            assert tails <= 1
            if len(call) > 1 or call[0][0] == call[0][2]:
                assert sum(qe - qb for qb, qe, _, _ in call) <= info["T_m"]
            assert info["times"][ci] <= info["T_t"]                # every chunk within the final time threshold
        assert all(c == 1 for c in covered)
        # split slices follow the mesh
        for d, L in enumerate(lengths):
            mine = [c for call in calls for c in call if doc_of.get(c[0]) == d and L > 0]
            for j, c in enumerate(mine[:-1]):
                assert c[1] - c[0] == mesh[j]
    assert seen > 150


def test_errors():
    cost = IP.Cost(1.0, 0.0, 0.0)
    with pytest.raises(IP.PlanError):
        IP.plan([1000], 16, 10 ** 6, cost)           # 16 slices of a 1000-token sequence
    with pytest.raises(IP.PlanError):
        IP.plan([4096, 10], 2, 1000, cost)           # capacity below the first mesh slice
    with pytest.raises(IP.PlanError):
        IP.plan([4096], 2, 4096, IP.Cost(0.0, 0.0, 1.0))
    assert IP.plan([0, 0], 2, 100, cost)[0] == []
