"""Oracle of InfiniPipe's workload-balanced sequence chunking (Algorithm 1).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: InfiniPipe, "Elastic Pipeline Parallelism for Efficient Variable-Length
Long-Context LLM Training":
  * §III-A1 "Definition of Chunk": a chunk is {C, S}, a context length C and a
    set S of slice lengths; split chunks (a slice of a long sequence after the
    slices before it), batched chunks (short sequences, C = 0) and hybrid
    chunks (a tail slice s0 with its context, packed with short sequences); two
    tail slices are never packed together.
  * §III-A2, Eq. (1): the time of chunk {C_k, S_k} is
        (1/N) (alpha1((C+s0)^2 - C^2) + alpha2 s0 + sum_{s in S - s0}(alpha1 s^2 + alpha2 s)) + beta1/d_p.
  * §III-B and Algorithm 1: split the longest sequence into K workload-balanced
    slices (the mesh); shard long sequences by the mesh into split chunks and a
    tail slice; seed one bucket per tail slice; visit short sequences from the
    most to the least expensive and put each into the first bucket, in order of
    increasing tot_time/tot_tokens, that stays within the time threshold T_t
    and the token threshold T_m; open a new bucket when even the bucket with
    the fewest tokens cannot take it; loosen T_t when no bucket fits.

Readings where the pages leave a step open:
  * One GPU: N = 1 and d_p = 1 in Eq. (1); there is no all-to-all term (Eq. 3),
    so a chunk's modeled time is beta1 plus the sum of its slices' terms.
  * Mesh boundaries: b_k is the multiple of 128 nearest to the equal-cost
    point (cost(b) = alpha1 b^2 + alpha2 b reaching k/K of cost(L_max)), ties
    up; evaluated as b_k = 128 * #{j >= 1 : K cost(128 j - 64) <= k cost(L_max)}.
    With alpha2 = 0 this is the FLOPS rule of ``oracle.plan``. Boundaries that
    are not strictly increasing are an error.
  * Sharding by the mesh: mesh slices are taken in order while the remaining
    length is larger than the next slice; what remains is the tail slice. A
    sequence no longer than the first mesh slice is a short sequence.
  * T_t starts at the largest modeled time of a mesh slice (beta1 included).
    T_m is the caller's token capacity per chunk and must hold the first mesh
    slice.
  * Loosening (Alg. 1, the "goto" after no bucket fitted): T_t becomes the
    smallest tot_time among the buckets that can take the sequence by tokens,
    plus the sequence's time. Taken over all buckets, as printed, the loop
    would not end when the bucket with the least time is full of tokens.
  * Output order, for running the chunks one call at a time: the split chunks
    by slice index then sequence, then the buckets in creation order. Every
    sequence's slices come before its tail. Tokens are packed in the given
    sequence order.

Costs are evaluated in float64 with the integer terms formed exactly first, so
that a C implementation that keeps the same operation order takes the same
decisions.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple

TILE = 128

Chunk = Tuple[int, int, int, int]  # (q_begin, q_end, ctx_begin, kv_split) in the packed token layout


class PlanError(ValueError):
    """No plan exists for these inputs."""


@dataclass
class Cost:
    """Eq. (1) on one GPU: alpha1 per squared token, alpha2 per token, beta1 per chunk."""
    alpha1: float
    alpha2: float
    beta1: float

    def slice_time(self, C: int, s: int) -> float:
        """alpha1((C+s)^2 - C^2) + alpha2 s for a slice of s tokens after C context tokens."""
        quad = (C + s) * (C + s) - C * C
        return self.alpha1 * float(quad) + self.alpha2 * float(s)

    def prefix_cost(self, b: int) -> float:
        """Cost of the first b tokens of a sequence: alpha1 b^2 + alpha2 b."""
        return self.alpha1 * float(b * b) + self.alpha2 * float(b)


def split_longest(Lmax: int, K: int, cost: Cost) -> List[int]:
    """M.split(max(S), K): boundaries b_0 = 0 < b_1 < ... < b_K = Lmax of K
    slices of equal modeled cost, rounded to multiples of 128 (nearest, ties up)."""
    if K < 1 or Lmax < 1:
        raise PlanError("need K >= 1 and a non-empty longest sequence")
    total = cost.prefix_cost(Lmax)
    b = [0]
    for k in range(1, K):
        target = float(k) * total
        m = 0
        while float(K) * cost.prefix_cost(TILE * (m + 1) - TILE // 2) <= target:
            m += 1
        b.append(TILE * m)
    b.append(Lmax)
    if any(not b[i] < b[i + 1] for i in range(K)):
        raise PlanError(f"the longest sequence ({Lmax} tokens) cannot be cut into {K} slices of 128-token steps")
    return b


def split_by_mesh(lengths: Sequence[int], mesh: Sequence[int]):
    """split(S, mesh): for each sequence, the mesh slices taken (with their
    contexts) and the tail slice, or None when the sequence is short.
    Returns a list of (slices [(ctx, len)], tail (ctx, len) or None)."""
    out = []
    for L in lengths:
        rem, ctx, slices = L, 0, []
        for m in mesh:
            if rem > m:
                slices.append((ctx, m))
                ctx += m
                rem -= m
            else:
                break
        out.append((slices, (ctx, rem) if slices else None))
    return out


@dataclass
class Bucket:
    order: int                                       # creation index
    tail: bool
    members: List[Tuple[int, int, int]] = field(default_factory=list)   # (sequence, ctx, len)
    tot_time: float = 0.0
    tot_tokens: int = 0

    def metric(self) -> float:
        return self.tot_time / self.tot_tokens


def bfd(buckets: List[Bucket], shorts: Sequence[Tuple[int, int]], T_t: float, T_m: int, cost: Cost) -> float:
    """Lines 3-28 of Algorithm 1 on the given buckets: place every short
    sequence (index, length) in that order. Returns the final T_t."""
    for idx, s in shorts:
        t = cost.slice_time(0, s)
        while True:
            if not buckets or min(b.tot_tokens for b in buckets) + s > T_m:
                nb = Bucket(order=len(buckets), tail=False)
                nb.members.append((idx, 0, s))
                nb.tot_time = cost.beta1 + t
                nb.tot_tokens = s
                buckets.append(nb)
                break
            placed = False
            for b in sorted(buckets, key=lambda x: (x.metric(), x.order)):
                if b.tot_time + t <= T_t and b.tot_tokens + s <= T_m:
                    b.members.append((idx, 0, s))
                    b.tot_time = b.tot_time + t
                    b.tot_tokens = b.tot_tokens + s
                    placed = True
                    break
            if placed:
                break
            T_t = min(b.tot_time for b in buckets if b.tot_tokens + s <= T_m) + t
    return T_t


def plan(lengths: Sequence[int], K: int, token_cap: int, cost: Cost):
    """Algorithm 1. Returns (calls, info): calls is a list of chunk lists in
    the packed layout (sequences back to back in the given order), one list
    per chunk {C, S}, in an order that can be run forward one call at a time;
    info holds the mesh, T_t, T_m and each call's modeled time."""
    if cost.alpha1 < 0 or cost.alpha2 < 0 or cost.beta1 < 0 or (cost.alpha1 == 0 and cost.alpha2 == 0):
        raise PlanError("costs must be non-negative with alpha1 or alpha2 positive")
    if any(L < 0 for L in lengths):
        raise PlanError("negative sequence length")
    starts = [0]
    for L in lengths:
        starts.append(starts[-1] + L)
    live = [i for i, L in enumerate(lengths) if L > 0]
    if not live:
        return [], {"mesh": [], "T_t": 0.0, "T_m": token_cap, "times": []}
    Lmax = max(lengths)
    b = split_longest(Lmax, K, cost)
    mesh = [b[i + 1] - b[i] for i in range(K)]
    if token_cap < mesh[0]:
        raise PlanError(f"token capacity {token_cap} below the first mesh slice {mesh[0]}")
    T_t = max(cost.beta1 + cost.slice_time(b[i], mesh[i]) for i in range(K))
    T_m = token_cap
    parts = split_by_mesh(lengths, mesh)
    buckets: List[Bucket] = []
    for i in live:
        slices, tail = parts[i]
        if tail is not None:
            bk = Bucket(order=len(buckets), tail=True)
            bk.members.append((i, tail[0], tail[1]))
            bk.tot_time = cost.beta1 + cost.slice_time(tail[0], tail[1])
            bk.tot_tokens = tail[1]
            buckets.append(bk)
    shorts = [(i, lengths[i]) for i in live if parts[i][1] is None]
    shorts.sort(key=lambda x: (-cost.slice_time(0, x[1]), x[0]))
    T_t = bfd(buckets, shorts, T_t, T_m, cost)

    calls, times = [], []
    depth = max(len(parts[i][0]) for i in live)
    for j in range(depth):
        for i in live:
            slices = parts[i][0]
            if j < len(slices):
                ctx, m = slices[j]
                calls.append([(starts[i] + ctx, starts[i] + ctx + m, starts[i], 0)])
                times.append(cost.beta1 + cost.slice_time(ctx, m))
    for bk in buckets:
        chunks = sorted((starts[i] + ctx, starts[i] + ctx + s, starts[i], 0) for i, ctx, s in bk.members)
        calls.append(chunks)
        times.append(bk.tot_time)
    return calls, {"mesh": mesh, "T_t": T_t, "T_m": T_m, "times": times}
