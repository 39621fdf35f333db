"""Float64 oracle of causal softmax attention, forward and backward.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

All functions act on ONE (batch, head) slice: ``q, k, v, do`` are ``[T, D]``
arrays (any float dtype; they are upcast to float64, so bf16 inputs are used
at their exact values). Documents are given by ``cu_seqlens`` (document start
offsets, first 0, last T); ``None`` means one causal sequence.

Definition (the result every schedule must reach)
-------------------------------------------------
Key j is visible to query t iff j and t lie in the same document and j <= t
(InfiniPipe §II-A "Pipeline Parallelism": a token's query reads only the keys
and values of preceding tokens; §II-B "Sequence Packing" for the per-document
[sum(S), D] layout). With S_tj = scale * q_t . k_j:

    LSE_t = ln sum_{j visible} exp(S_tj)          (natural log)
    P_tj  = exp(S_tj - LSE_t)
    O_t   = sum_j P_tj v_j

Backward for a given upstream gradient dO (the standard analytic gradient of
the definition above):

    D_t   = dO_t . O_t
    dP_tj = dO_t . v_j
    dS_tj = P_tj (dP_tj - D_t)
    dQ_t  = scale sum_j dS_tj k_j
    dK_j  = scale sum_t dS_tj q_t
    dV_j  = sum_t P_tj dO_t

The chunked method (SPPO §5.1 "Two-Level Activation Management": the
attention of subsequence i reads its own Q against all K/V produced so far;
the RSA blog's "Deep Dive", where a chunk's output is assembled from one
partial per key/value block, O^n = sum_i S_i^n V_i) reaches this same result;
the blog says sequence parallelism computes exactly the forward pass of a
single device. ``chunked_forward`` evaluates it that way, block by block with a
log-sum-exp merge of per-block partials, so that tests can check it against
the plain definition.

Evaluation uses explicit score rows in row blocks (the full L x L matrix of a
32K sequence would be 8.6 GB per head), with the usual max-subtraction before
``exp``; no other reordering of the definition.
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _docs(T: int, cu_seqlens: Optional[Sequence[int]]) -> List[Tuple[int, int]]:
    if cu_seqlens is None:
        return [(0, T)]
    cu = [int(c) for c in cu_seqlens]
    assert cu[0] == 0 and cu[-1] == T, "cu_seqlens must run from 0 to T"
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1) if cu[i + 1] > cu[i]]


def doc_start_of_rows(T: int, cu_seqlens: Optional[Sequence[int]]) -> np.ndarray:
    """Document start of every token (the first key a token may see)."""
    start = np.zeros(T, dtype=np.int64)
    for s, e in _docs(T, cu_seqlens):
        start[s:e] = s
    return start


def _score_rows(q, k, scale, r0, r1, s):
    """Masked scaled scores of rows [r0, r1) against keys [s, r1): j <= t."""
    S = scale * (q[r0:r1] @ k[s:r1].T)
    t = np.arange(r0, r1)[:, None]
    j = np.arange(s, r1)[None, :]
    return np.where(j <= t, S, NEG_INF)


def _softmax_rows(S):
    mx = S.max(axis=1, keepdims=True)
    E = np.exp(S - mx)
    l = E.sum(axis=1, keepdims=True)
    return E / l, (mx + np.log(l))[:, 0]


def forward(q, k, v, scale: float, cu_seqlens=None, row_block: int = 512):
    """O [T, D] and LSE [T] of causal (per-document) softmax attention."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T = q.shape[0]
    O = np.zeros((T, v.shape[1]))
    LSE = np.full(T, NEG_INF)
    for s, e in _docs(T, cu_seqlens):
        for r0 in range(s, e, row_block):
            r1 = min(r0 + row_block, e)
            P, lse = _softmax_rows(_score_rows(q, k, scale, r0, r1, s))
            O[r0:r1] = P @ v[s:r1]
            LSE[r0:r1] = lse
    return O, LSE


def backward(q, k, v, do, scale: float, cu_seqlens=None, row_block: int = 512):
    """(dQ, dK, dV, O, LSE) for upstream gradient dO; O and LSE are the oracle's own."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    T = q.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    O = np.zeros((T, v.shape[1]))
    LSE = np.full(T, NEG_INF)
    for s, e in _docs(T, cu_seqlens):
        for r0 in range(s, e, row_block):
            r1 = min(r0 + row_block, e)
            P, lse = _softmax_rows(_score_rows(q, k, scale, r0, r1, s))
            o = P @ v[s:r1]
            O[r0:r1] = o
            LSE[r0:r1] = lse
            D = np.sum(do[r0:r1] * o, axis=1, keepdims=True)
            dP = do[r0:r1] @ v[s:r1].T
            dS = P * (dP - D)
            dq[r0:r1] = scale * (dS @ k[s:r1])
            dk[s:r1] += scale * (dS.T @ q[r0:r1])
            dv[s:r1] += P.T @ do[r0:r1]
    return dq, dk, dv, O, LSE


# --------------------------------------------------------------------------
# Sampled forms for sequences too long for the full oracle.
# --------------------------------------------------------------------------

def _row_groups(rows, start, max_elems=1 << 27):
    """Sampled rows sorted and grouped by document, each group small enough
    that its score matrix (rows x keys) stays under ``max_elems`` entries."""
    order = np.argsort(rows, kind="stable")
    groups, cur = [], []
    for idx in order:
        t = int(rows[idx])
        if cur:
            t0 = int(rows[cur[0]])
            same_doc = start[t] == start[t0]
            keys = t - start[t0] + 1
            if not same_doc or (len(cur) + 1) * keys > max_elems:
                groups.append(cur)
                cur = []
        cur.append(idx)
    if cur:
        groups.append(cur)
    return groups


def _rows_probs(q, k, rows_g, s, scale):
    """Softmax rows P (rows x keys [s, t_max]) of a group of rows of one
    document; each row is the definition applied to that row alone."""
    tmax = int(rows_g.max())
    S = scale * (q[rows_g] @ k[s:tmax + 1].T)
    j = np.arange(s, tmax + 1)[None, :]
    S = np.where(j <= rows_g[:, None], S, NEG_INF)
    return _softmax_rows(S), tmax


def forward_rows(q, k, v, rows: Iterable[int], scale: float, cu_seqlens=None):
    """O and LSE of the given query rows only (each row is independent)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T = q.shape[0]
    start = doc_start_of_rows(T, cu_seqlens)
    rows = np.asarray(list(rows), dtype=np.int64)
    O = np.zeros((len(rows), v.shape[1]))
    LSE = np.zeros(len(rows))
    for grp in _row_groups(rows, start):
        rg = rows[grp]
        s = int(start[rg[0]])
        (P, lse), tmax = _rows_probs(q, k, rg, s, scale)
        O[grp] = P @ v[s:tmax + 1]
        LSE[grp] = lse
    return O, LSE


def dq_rows(q, k, v, do, rows: Iterable[int], scale: float, cu_seqlens=None):
    """dQ of the given query rows; D_t uses the oracle's own O_t."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    T = q.shape[0]
    start = doc_start_of_rows(T, cu_seqlens)
    rows = np.asarray(list(rows), dtype=np.int64)
    dq = np.zeros((len(rows), q.shape[1]))
    for grp in _row_groups(rows, start):
        rg = rows[grp]
        s = int(start[rg[0]])
        (P, _), tmax = _rows_probs(q, k, rg, s, scale)
        o = P @ v[s:tmax + 1]
        D = np.sum(do[rg] * o, axis=1, keepdims=True)
        dP = do[rg] @ v[s:tmax + 1].T
        dS = P * (dP - D)
        dq[grp] = scale * (dS @ k[s:tmax + 1])
    return dq


def dkdv_keys(q, k, v, do, keys: Iterable[int], scale: float, cu_seqlens=None,
              row_block: int = 256):
    """dK and dV of the given keys. Needs O_t, LSE_t for every row t >= key in
    its document, so keep the sampled keys near a document end."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    T = q.shape[0]
    start = doc_start_of_rows(T, cu_seqlens)
    docs = _docs(T, cu_seqlens)
    end_of = np.zeros(T, dtype=np.int64)
    for s, e in docs:
        end_of[s:e] = e
    keys = np.asarray(list(keys), dtype=np.int64)
    dk = np.zeros((len(keys), k.shape[1]))
    dv = np.zeros((len(keys), v.shape[1]))
    # rows needed: union of [j, end(j)) over sampled keys, evaluated once per doc
    by_doc = {}
    for i, j in enumerate(keys):
        by_doc.setdefault(int(start[j]), []).append(i)
    for s, idxs in by_doc.items():
        e = int(end_of[keys[idxs[0]]])
        jmin = int(min(keys[i] for i in idxs))
        for r0 in range(jmin, e, row_block):
            r1 = min(r0 + row_block, e)
            P, _ = _softmax_rows(_score_rows(q, k, scale, r0, r1, s))
            o = P @ v[s:r1]
            D = np.sum(do[r0:r1] * o, axis=1)
            for i in idxs:
                j = int(keys[i])
                if j >= r1:
                    continue
                pj = P[:, j - s]                      # P_tj for t in [r0, r1)
                dpj = do[r0:r1] @ v[j]
                dsj = pj * (dpj - D)
                dk[i] += scale * (dsj @ q[r0:r1])
                dv[i] += pj @ do[r0:r1]
    return dk, dv


# --------------------------------------------------------------------------
# The chunked method: per-chunk partials over key/value ranges, LSE merge.
# --------------------------------------------------------------------------

def partial(q, k, v, r0: int, r1: int, kv_lo: int, kv_hi: int, scale: float):
    """Partial (O_p, LSE_p) of query rows [r0, r1) over keys [kv_lo, kv_hi)
    with the causal rule j <= t. A row with no visible key in the range gets
    LSE_p = -inf and O_p = 0 (an empty block contributes nothing)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = r1 - r0
    O = np.zeros((n, v.shape[1]))
    LSE = np.full(n, NEG_INF)
    if kv_hi <= kv_lo:
        return O, LSE
    S = scale * (q[r0:r1] @ k[kv_lo:kv_hi].T)
    t = np.arange(r0, r1)[:, None]
    j = np.arange(kv_lo, kv_hi)[None, :]
    S = np.where(j <= t, S, NEG_INF)
    has = np.isfinite(S).any(axis=1)
    if has.any():
        Sh = S[has]
        mx = Sh.max(axis=1, keepdims=True)
        E = np.exp(Sh - mx)
        l = E.sum(axis=1, keepdims=True)
        O[has] = (E / l) @ v[kv_lo:kv_hi]
        LSE[has] = (mx + np.log(l))[:, 0]
    return O, LSE


def lse_merge(parts: Sequence[Tuple[np.ndarray, np.ndarray]]):
    """Merge partials of disjoint key blocks: LSE = ln sum_p exp(LSE_p),
    O = sum_p exp(LSE_p - LSE) O_p; a part with LSE_p = -inf has weight 0."""
    lses = np.stack([_f64(p[1]) for p in parts])          # [P, n]
    mx = lses.max(axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    tot = np.sum(np.exp(lses - safe), axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(tot > 0, safe + np.log(tot), NEG_INF)
    O = np.zeros_like(_f64(parts[0][0]))
    for o_p, l_p in parts:
        w = np.where(np.isfinite(l_p), np.exp(_f64(l_p) - np.where(np.isfinite(lse), lse, 0.0)), 0.0)
        O += w[:, None] * _f64(o_p)
    return O, lse


def chunked_forward(q, k, v, chunks: Sequence[Tuple[int, int, int, int]], scale: float,
                    kv_block: Optional[int] = None):
    """The chunked method: for each chunk (q_begin, q_end, ctx_begin, kv_split)
    the chunk's queries attend to the resident keys [ctx_begin, q_end); with a
    re-split point m > 0 the key range is split into [ctx_begin, m) and
    [m, q_end), with kv_split = -P into P parts of equal visible-pair count
    (``oracle.plan.key_ranges``), and the partials are merged by LSE. ``kv_block`` further cuts every
    key range into blocks of that many keys, each contributing one partial
    (the ring's one-block-per-hop accumulation)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T = q.shape[0]
    O = np.zeros((T, v.shape[1]))
    LSE = np.full(T, NEG_INF)
    from oracle.plan import key_ranges
    for qb, qe, cb, m in chunks:
        ranges = key_ranges((qb, qe, cb, m))
        if kv_block:
            ranges = [(a, min(a + kv_block, b)) for lo, b in ranges for a in range(lo, b, kv_block)]
        parts = [partial(q, k, v, qb, qe, lo, hi, scale) for lo, hi in ranges]
        o, l = lse_merge(parts)
        O[qb:qe] = o
        LSE[qb:qe] = l
    return O, LSE


def grouped_backward(qs, k, v, dos, scale: float, cu_seqlens=None, row_block: int = 512):
    """Grouped key/value heads (GQA/MQA): the query heads in ``qs`` (each
    [T, D], upstream gradients in ``dos``) all read the one key/value head
    (k, v). Each query head is plain attention against (k, v); the gradient of
    the shared k and v is the sum of the per-head gradients (the chain rule
    for a tensor used by several heads). Returns (dQ per head, dK, dV, O per
    head, LSE per head)."""
    dqs, Os, Ls = [], [], []
    dk = np.zeros_like(_f64(k))
    dv = np.zeros_like(_f64(v))
    for q, do in zip(qs, dos):
        dq, dk_h, dv_h, O, L = backward(q, k, v, do, scale, cu_seqlens, row_block)
        dqs.append(dq)
        Os.append(O)
        Ls.append(L)
        dk += dk_h
        dv += dv_h
    return dqs, dk, dv, Os, Ls


def chunk_backward(q, k, v, do, qb: int, qe: int, cb: int, scale: float, row_block: int = 512):
    """Contributions of the query rows of ONE chunk, [qb, qe) with context
    starting at cb (the document start), to the gradients: the definition's
    sums restricted to t in [qb, qe). Returns (dQ rows [qb, qe), dK and dV
    contributions for keys [cb, qe)).

    This is how the chunked method runs the backward (InfiniPipe §II-A: the
    K/V gradients of a token gather contributions from all later tokens; SPPO
    §5.1 keeps each subsequence's K/V resident for the later subsequences):
    chunks are processed in reverse order and each chunk adds its queries'
    share to the keys of its context. dQ of the chunk's rows is complete,
    because every key a row can see lies in [cb, qe)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq = np.zeros((qe - qb, q.shape[1]))
    dk = np.zeros((qe - cb, k.shape[1]))
    dv = np.zeros((qe - cb, v.shape[1]))
    for r0 in range(qb, qe, row_block):
        r1 = min(r0 + row_block, qe)
        P, _ = _softmax_rows(_score_rows(q, k, scale, r0, r1, cb))   # keys [cb, r1)
        o = P @ v[cb:r1]
        D = np.sum(do[r0:r1] * o, axis=1, keepdims=True)
        dP = do[r0:r1] @ v[cb:r1].T
        dS = P * (dP - D)
        dq[r0 - qb:r1 - qb] = scale * (dS @ k[cb:r1])
        dk[:r1 - cb] += scale * (dS.T @ q[r0:r1])
        dv[:r1 - cb] += P.T @ do[r0:r1]
    return dq, dk, dv


# --------------------------------------------------------------------------
# Closed form for periodic keys: a full-size check of every row and key.
# --------------------------------------------------------------------------

def periodic_keys(q, kc, v, do, scale: float):
    """O, LSE, dQ and dV of one causal sequence whose keys repeat with period
    p: k_j = kc[j mod p]. Then the scores of row t take only p values
    s_tc = scale q_t . kc[c], so with n_c(t) = #{j <= t : j mod p = c}:

        Z_t = sum_c n_c(t) e^{s_tc},   LSE_t = ln Z_t,   W_tc = e^{s_tc} / Z_t = P_tj (j in class c)
        O_t  = sum_c W_tc CV_c(t),     CV_c(t) = sum_{j <= t, j = c mod p} v_j
        dQ_t = scale sum_c W_tc (dO_t . CV_c(t) - n_c(t) D_t) kc[c],   D_t = dO_t . O_t
        dV_j = sum_{t >= j} W_{t, j mod p} dO_t

    i.e. the definition regrouped by key class, evaluated with cumulative
    sums in O(T p D). dK is not produced (it needs D x D running sums)."""
    q, kc, v, do = _f64(q), _f64(kc), _f64(v), _f64(do)
    T, D = q.shape
    p = kc.shape[0]
    t = np.arange(T)
    n = np.stack([np.where(t >= c, (t - c) // p + 1, 0) for c in range(p)], axis=1).astype(np.float64)
    s = scale * (q @ kc.T)
    s = np.where(n > 0, s, NEG_INF)
    M = s.max(axis=1)
    E = np.where(n > 0, np.exp(s - M[:, None]), 0.0)
    Z = (n * E).sum(axis=1)
    LSE = M + np.log(Z)
    W = E / Z[:, None]
    O = np.zeros((T, D))
    g = np.zeros((T, p))
    cls = t % p
    CVs = []
    for c in range(p):
        CV = np.cumsum(np.where((cls == c)[:, None], v, 0.0), axis=0)
        O += W[:, c:c + 1] * CV
        CVs.append(CV)
    Dt = np.sum(do * O, axis=1)
    for c in range(p):
        g[:, c] = np.sum(do * CVs[c], axis=1) - n[:, c] * Dt
    dQ = scale * ((W * g) @ kc)
    dV = np.zeros((T, D))
    for c in range(p):
        R = np.cumsum((W[:, c:c + 1] * do)[::-1], axis=0)[::-1]
        dV[cls == c] = R[cls == c]
    return O, LSE, dQ, dV


# --------------------------------------------------------------------------
# Closed form for periodic queries: a full-size check of every key's dK.
# --------------------------------------------------------------------------

def _suffix_sums(x):
    """Inclusive suffix sums along axis 0: out[j] = sum_{t >= j} x[t]."""
    return np.cumsum(x[::-1], axis=0)[::-1]


def periodic_queries(qc, k, v, do, scale: float):
    """O, LSE, dK and dV of one causal sequence whose queries repeat with
    period p: q_t = qc[t mod p]; keys, values and dO are arbitrary. The score
    of row t against key j then depends on t only through its class
    c = t mod p: s_cj = scale qc[c] . k_j. With E_cj = e^{s_cj - M_c}, where
    M_c = max_j s_cj (a shift that cancels in P):

        Z_t   = sum_{j <= t} E_cj,       LSE_t = M_c + ln Z_t,       P_tj = E_cj / Z_t
        O_t   = sum_{j <= t} E_cj v_j / Z_t,                         D_t  = dO_t . O_t
        R_c(j) = sum_{t >= j, t = c mod p} dO_t / Z_t,   r_c(j) = sum_{t >= j, t = c mod p} D_t / Z_t
        dV_j  = sum_t P_tj dO_t                      = sum_c E_cj R_c(j)
        dK_j  = scale sum_t P_tj (dO_t . v_j - D_t) q_t = scale sum_c E_cj (v_j . R_c(j) - r_c(j)) qc[c]

    i.e. the definition's sums regrouped by query class, evaluated with
    prefix sums over keys (forward) and suffix sums over queries (backward)
    in O(T p D), so that every key's dK and dV can be checked at full size,
    including the first keys, whose sums run over the whole sequence. dQ is
    not produced (its sum needs D x D running sums); the periodic-keys form
    covers it."""
    qc, k, v, do = _f64(qc), _f64(k), _f64(v), _f64(do)
    T, D = k.shape
    p = qc.shape[0]
    t = np.arange(T)
    cls = t % p
    s = scale * (k @ qc.T)                          # [T keys, p classes]
    M = s.max(axis=0)
    E = np.exp(s - M[None, :])
    O = np.zeros((T, D))
    LSE = np.zeros(T)
    Z = np.zeros(T)
    for c in range(p):
        rows = cls == c
        Zc = np.cumsum(E[:, c])                     # Z_t for a row t of class c
        num = np.cumsum(E[:, c:c + 1] * v, axis=0)  # sum_{j <= t} E_cj v_j
        Z[rows] = Zc[rows]
        O[rows] = num[rows] / Zc[rows, None]
        LSE[rows] = M[c] + np.log(Zc[rows])
        del num
    Dt = np.sum(do * O, axis=1)
    dK = np.zeros((T, D))
    dV = np.zeros((T, D))
    for c in range(p):
        w = np.where(cls == c, 1.0 / Z, 0.0)        # 1/Z_t on the rows of class c
        R = _suffix_sums(w[:, None] * do)           # R_c(j)
        r = _suffix_sums(w * Dt)                    # r_c(j)
        dV += E[:, c:c + 1] * R
        dK += (scale * E[:, c] * (np.sum(v * R, axis=1) - r))[:, None] * qc[c][None, :]
        del R
    return O, LSE, dK, dV
