"""Oracle for the chunk planner (integer boundaries), written from the pages.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources
-------
* SPPO, "Efficient Long-sequence LLM Training via Adaptive Sequence Pipeline
  Parallel Offloading", §3.2 "Imbalanced GPU computation across subsequences":
  attention work grows with token position, so a FLOPs-based partition starts
  with long subsequences and moves to shorter ones; a length-based partition
  keeps one length for all subsequences.
* InfiniPipe, "Elastic Pipeline Parallelism for Efficient Variable-Length
  Long-Context LLM Training", §III-A2, Eq. (1): chunk cost is quadratic in
  context, alpha1((C+s)^2 - C^2). Equal quadratic cost for chunks [b_{k-1}, b_k)
  of one sequence means b_k^2 - b_{k-1}^2 = L^2/N, i.e. b_k = L*sqrt(k/N).
* SPPO §4 "Multiplexing Sequence Partition" and §6.2: the subsequences next to
  the pipeline bubbles (first and last) are re-split into two sub-subsequences
  whose partial results are combined afterwards.
* InfiniPipe §III-A1 "Definition of Chunk": a split chunk is a slice of a long
  sequence with a context C (the preceding slices); short sequences form
  batched chunks with C = 0.

Readings taken where the pages leave a step open:
* FLOPS rule: b_k = nearest multiple of 128 to L*sqrt(k/N), ties rounded up,
  b_0 = 0, b_N = L; a plan whose boundaries are not strictly increasing is an
  error (too many chunks for L), never clamped.
* UNIFORM rule: b_k = 128*floor(k*L/(128*N)), b_N = L.
* Re-split point m = q_begin + 128*floor((q_end - q_begin)/256 + 1/2); the
  split is along the key/value range (parts [ctx_begin, m) and [m, q_end));
  no split when m does not fall strictly inside (q_begin, q_end).
* Re-split into P parts (kv_split = -P): the chunk's key range [ctx_begin,
  q_end) is cut into P parts carrying equal numbers of visible (query, key)
  pairs of the chunk's queries; boundary k_p is the multiple of 128 (counted
  from ctx_begin) nearest to the point where the pairs of keys before it reach
  p/P of the total (ties up); boundaries that collapse are an error. SPPO
  Table 3 (multiplexed partition): the SP range of the edge subsequences
  shrinks by one device per subsequence away from each pipeline end, read as
  chunk i and chunk N-1-i of N getting PP - i parts (the largest valid count
  up to that), for PP pipeline stages.
* Varlen: a document of length L_d is cut into ceil(L_d / max_chunk_tokens)
  chunks with the same rule measured from the document start; every chunk of a
  document has ctx_begin = document start. Empty documents give no chunk. In
  re-split mode the first and last chunk of the whole plan are re-split.

This module computes the FLOPS rule with 60-digit decimal square roots and
round-half-up, which is a different route from the integer search the
library uses; ``tests/test_oracle_plan.py`` pins both against a brute-force
nearest-multiple search done with exact integer squares.
"""
from __future__ import annotations

from decimal import ROUND_HALF_UP, Decimal, localcontext
from typing import List, Sequence, Tuple

UNIFORM = 0
FLOPS = 1
FLOPS_RESPLIT_EDGES = 2

TILE = 128

Chunk = Tuple[int, int, int, int]  # (q_begin, q_end, ctx_begin, kv_split)


class PlanError(ValueError):
    """The requested plan does not exist (e.g. more chunks than 128-token steps)."""


def _flops_boundary(L: int, k: int, N: int) -> int:
    """Nearest multiple of 128 to L*sqrt(k/N), ties up (SPPO §3.2 FLOPs policy)."""
    with localcontext() as ctx:
        ctx.prec = 60
        x = Decimal(L) * (Decimal(k) / Decimal(N)).sqrt() / Decimal(TILE)
        m = x.quantize(Decimal(1), rounding=ROUND_HALF_UP)
    return TILE * int(m)


def boundaries(L: int, N: int, mode: int) -> List[int]:
    """Chunk boundaries b_0 = 0 < b_1 < ... < b_N = L for one causal sequence."""
    if L <= 0 or N <= 0:
        raise PlanError("L and N must be positive")
    if mode not in (UNIFORM, FLOPS, FLOPS_RESPLIT_EDGES):
        raise PlanError("unknown mode")
    b = [0]
    for k in range(1, N):
        if mode == UNIFORM:
            b.append(TILE * ((k * L) // (TILE * N)))
        else:
            b.append(_flops_boundary(L, k, N))
    b.append(L)
    for i in range(N):
        if not b[i] < b[i + 1]:
            raise PlanError("boundaries not strictly increasing")
    return b


def resplit_point(q_begin: int, q_end: int) -> int:
    """Sub-subsequence boundary of a re-split edge chunk, 0 when no split."""
    n = q_end - q_begin
    # floor(n/256 + 1/2) == floor((n + 128) / 256) for integer n
    m = q_begin + TILE * ((n + TILE) // (2 * TILE))
    return m if q_begin < m < q_end else 0


def _apply_resplit(chunks: List[List[int]]) -> None:
    if not chunks:
        return
    for idx in {0, len(chunks) - 1}:
        c = chunks[idx]
        c[3] = resplit_point(c[0], c[1])


def plan(L: int, N: int, mode: int) -> List[Chunk]:
    """Chunks (q_begin, q_end, ctx_begin=0, kv_split) of one causal sequence."""
    b = boundaries(L, N, mode)
    chunks = [[b[i], b[i + 1], 0, 0] for i in range(N)]
    if mode == FLOPS_RESPLIT_EDGES:
        _apply_resplit(chunks)
    return [tuple(c) for c in chunks]


def plan_varlen(cu_seqlens: Sequence[int], max_chunk_tokens: int, mode: int) -> List[Chunk]:
    """Chunks of a packed batch of documents (InfiniPipe split/batched chunks)."""
    if max_chunk_tokens <= 0:
        raise PlanError("max_chunk_tokens must be positive")
    if len(cu_seqlens) < 2 or cu_seqlens[0] != 0:
        raise PlanError("cu_seqlens must start at 0 and hold at least one document")
    chunks: List[List[int]] = []
    for d in range(len(cu_seqlens) - 1):
        s, e = int(cu_seqlens[d]), int(cu_seqlens[d + 1])
        if e < s:
            raise PlanError("cu_seqlens must be non-decreasing")
        Ld = e - s
        if Ld == 0:
            continue
        Nd = -(-Ld // max_chunk_tokens)
        rule = UNIFORM if mode == UNIFORM else FLOPS
        b = boundaries(Ld, Nd, rule)
        for i in range(Nd):
            chunks.append([s + b[i], s + b[i + 1], s, 0])
    if mode == FLOPS_RESPLIT_EDGES:
        _apply_resplit(chunks)
    return [tuple(c) for c in chunks]


def key_pairs_before(q_begin: int, q_end: int, ctx_begin: int, K: int) -> int:
    """Visible (query, key) pairs of a chunk's queries [q_begin, q_end) with the
    keys in [ctx_begin, K): a context key is seen by every query, key j inside
    the chunk by the queries t >= j."""
    n = q_end - q_begin
    A = min(K, q_begin) - ctx_begin
    B = max(0, K - q_begin)
    return A * n + B * n - B * (B - 1) // 2


def resplit_boundaries(q_begin: int, q_end: int, ctx_begin: int, P: int) -> List[int]:
    """Key-range boundaries ctx_begin = k_0 < k_1 < ... < k_P = q_end of a chunk
    re-split into P parts of equal visible-pair count (nearest multiple of 128
    from ctx_begin, ties up)."""
    if P < 2:
        raise PlanError("a re-split needs at least two parts")
    W = key_pairs_before(q_begin, q_end, ctx_begin, q_end)
    k = [ctx_begin]
    for p in range(1, P):
        m = 0
        while True:
            half = ctx_begin + TILE * (m + 1) - TILE // 2
            if half > q_end or P * key_pairs_before(q_begin, q_end, ctx_begin, half) > p * W:
                break
            m += 1
        k.append(ctx_begin + TILE * m)
    k.append(q_end)
    if any(not k[i] < k[i + 1] for i in range(P)):
        raise PlanError(f"chunk ({q_begin}, {q_end}, {ctx_begin}) cannot be re-split into {P} parts")
    return k


def key_ranges(chunk: Chunk) -> List[Tuple[int, int]]:
    """The key ranges whose partials a chunk merges: one range, two (split at
    kv_split > 0) or P FLOPs-balanced parts (kv_split = -P)."""
    qb, qe, cb, m = chunk
    if m == 0:
        return [(cb, qe)]
    if m > 0:
        return [(cb, m), (m, qe)]
    k = resplit_boundaries(qb, qe, cb, -m)
    return [(k[i], k[i + 1]) for i in range(len(k) - 1)]


def plan_multiplex(L: int, N: int, PP: int) -> List[Chunk]:
    """FLOPS chunks of one sequence with the edge chunks re-split as in SPPO
    Table 3: chunk i and chunk N-1-i get PP - i parts (the largest count from
    2 up to that which the chunk can hold; none below 2)."""
    if PP < 1:
        raise PlanError("PP must be positive")
    b = boundaries(L, N, FLOPS)
    chunks = [[b[i], b[i + 1], 0, 0] for i in range(N)]
    for i in range(N):
        want = PP - min(i, N - 1 - i)
        for P in range(want, 1, -1):
            try:
                resplit_boundaries(b[i], b[i + 1], 0, P)
            except PlanError:
                continue
            chunks[i][3] = -P
            break
    return [tuple(c) for c in chunks]


def causal_pairs(q_begin: int, q_end: int, ctx_begin: int) -> int:
    """Number of visible (query, key) pairs of a chunk: sum over t of t-ctx_begin+1."""
    a = q_begin - ctx_begin + 1
    b = q_end - ctx_begin
    return (a + b) * (b - a + 1) // 2
