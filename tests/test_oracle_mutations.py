"""Strength of the oracle's pins (no GPU): plausible mistakes are planted in
the oracle on the CPU, by replacing its internals for the duration of one
test, and each must make at least one of the independent pins in
test_oracle_attention.py / test_oracle_plan.py fail. A planted mistake that
every pin still passed would mean that part of the oracle is not pinned.

Forward: the causal mask, the scale, the log-sum-exp, the normalisation.
Backward: the row term D_t, the sign of dS, the scale of dK, dV's upstream
operand, dQ's operand. Merge: the partial weights. Planner: the rounding of
the FLOPs rule, the re-split point."""
import numpy as np
import pytest

import test_oracle_attention as TA
import test_oracle_plan as TP
from oracle import attention as A
from oracle import plan as P


def fails(fn, *args) -> bool:
    """True when the pin rejects the (mutated) oracle."""
    try:
        with np.errstate(all="ignore"):
            fn(*args)
    except (AssertionError, ValueError, IndexError, FloatingPointError):
        return True
    return False


FORWARD_PINS = [
    (TA.test_forward_matches_brute_force, (40, 8, [0, 7, 8, 31, 40])),
    (TA.test_against_torch_sdpa_and_autograd, (257, 32, 5)),
    (TA.test_q_zero_closed_form, ()),
    (TA.test_rows_sum_to_one_and_first_row, ()),
    (TA.test_shift_invariances, ()),
]
BACKWARD_PINS = [
    (TA.test_against_torch_sdpa_and_autograd, (200, 16, 12)),
    (TA.test_finite_differences, ()),
    (TA.test_backward_invariants_and_last_key, ()),
    (TA.test_q_zero_closed_form, ()),
]


def test_pins_pass_on_the_oracle_itself():
    for fn, args in FORWARD_PINS + BACKWARD_PINS:
        assert not fails(fn, *args), fn.__name__


# ------------------------------------------------------------------ forward

def _scores_strict_mask(q, k, scale, r0, r1, s):
    S = scale * (q[r0:r1] @ k[s:r1].T)
    t = np.arange(r0, r1)[:, None]
    j = np.arange(s, r1)[None, :]
    return np.where(j < t, S, A.NEG_INF)                    # the key t itself dropped


def _scores_scale_twice(q, k, scale, r0, r1, s):
    S = scale * scale * (q[r0:r1] @ k[s:r1].T)
    t = np.arange(r0, r1)[:, None]
    j = np.arange(s, r1)[None, :]
    return np.where(j <= t, S, A.NEG_INF)


def _softmax_lse_without_max(S):
    mx = S.max(axis=1, keepdims=True)
    E = np.exp(S - mx)
    l = E.sum(axis=1, keepdims=True)
    return E / l, np.log(l)[:, 0]                           # the max term dropped


def _softmax_unnormalised(S):
    mx = S.max(axis=1, keepdims=True)
    E = np.exp(S - mx)
    l = E.sum(axis=1, keepdims=True)
    return E, (mx + np.log(l))[:, 0]                        # P not divided by l


@pytest.mark.parametrize("name,attr,fn", [
    ("mask j < t", "_score_rows", _scores_strict_mask),
    ("scale applied twice", "_score_rows", _scores_scale_twice),
    ("LSE without the max", "_softmax_rows", _softmax_lse_without_max),
    ("P not normalised", "_softmax_rows", _softmax_unnormalised),
])
def test_forward_mistake_is_caught(monkeypatch, name, attr, fn):
    monkeypatch.setattr(A, attr, fn)
    caught = [pin.__name__ for pin, args in FORWARD_PINS if fails(pin, *args)]
    assert caught, f"no forward pin catches: {name}"


# ------------------------------------------------------------------ backward

def _mutated_backward(kind):
    """The oracle's backward with one planted mistake of the given kind."""
    def backward(q, k, v, do, scale, cu_seqlens=None, row_block=512):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        T = q.shape[0]
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        O = np.zeros((T, v.shape[1]))
        LSE = np.full(T, A.NEG_INF)
        for s, e in A._docs(T, cu_seqlens):
            for r0 in range(s, e, row_block):
                r1 = min(r0 + row_block, e)
                Pm, lse = A._softmax_rows(A._score_rows(q, k, scale, r0, r1, s))
                o = Pm @ v[s:r1]
                O[r0:r1] = o
                LSE[r0:r1] = lse
                dP = do[r0:r1] @ v[s:r1].T
                D = dP.sum(axis=1, keepdims=True) if kind == "D from dP" else \
                    np.sum(do[r0:r1] * o, axis=1, keepdims=True)
                dS = Pm * (D - dP) if kind == "dS sign" else Pm * (dP - D)
                dq[r0:r1] = scale * ((Pm if kind == "dQ from P" else dS) @ k[s:r1])
                dk[s:r1] += (1.0 if kind == "dK unscaled" else scale) * (dS.T @ q[r0:r1])
                dv[s:r1] += Pm.T @ (o if kind == "dV from O" else do[r0:r1])
        return dq, dk, dv, O, LSE
    return backward


@pytest.mark.parametrize("kind", ["D from dP", "dS sign", "dK unscaled", "dV from O", "dQ from P"])
def test_backward_mistake_is_caught(monkeypatch, kind):
    monkeypatch.setattr(A, "backward", _mutated_backward(kind))
    caught = [pin.__name__ for pin, args in BACKWARD_PINS if fails(pin, *args)]
    assert caught, f"no backward pin catches: {kind}"


def test_mutated_backward_without_mistake_passes(monkeypatch):
    """The copy used above is the oracle's backward when no mistake is planted."""
    monkeypatch.setattr(A, "backward", _mutated_backward("none"))
    for pin, args in BACKWARD_PINS:
        assert not fails(pin, *args), pin.__name__


# ------------------------------------------------------------------ merge

def _merge_linear_weights(parts):
    lses = np.stack([np.asarray(p[1], dtype=np.float64) for p in parts])
    mx = lses.max(axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    tot = np.sum(np.exp(lses - safe), axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(tot > 0, safe + np.log(tot), A.NEG_INF)
    O = np.zeros_like(np.asarray(parts[0][0], dtype=np.float64))
    for o_p, l_p in parts:
        w = np.where(np.isfinite(l_p), 1.0 / len(parts), 0.0)     # weights not e^{LSE_p - LSE}
        O += w[:, None] * np.asarray(o_p, dtype=np.float64)
    return O, lse


def test_merge_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(A, "lse_merge", _merge_linear_weights)
    assert fails(TA.test_chunked_equals_unchunked, P.FLOPS_RESPLIT_EDGES) or fails(TA.test_merge_with_empty_part)


# ------------------------------------------------------------------ planner

def _flops_boundary_floor(L, k, N):
    step = P.TILE
    a = 0
    while ((a + 1) * step) ** 2 * N <= L * L * k:
        a += 1
    return a * step                                          # rounds down instead of to the nearest


def test_planner_rounding_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(P, "_flops_boundary", _flops_boundary_floor)
    assert fails(TP.test_flops_rule_matches_brute_force, 131072, 16) or fails(TP.test_known_plans)


def test_resplit_point_mistake_is_caught(monkeypatch):
    def resplit_off_by_one_tile(q_begin, q_end):
        n = q_end - q_begin
        m = q_begin + P.TILE * ((n + P.TILE) // (2 * P.TILE)) + P.TILE
        return m if q_begin < m < q_end else 0
    monkeypatch.setattr(P, "resplit_point", resplit_off_by_one_tile)
    assert fails(TP.test_resplit_point) or fails(TP.test_golden_plans)


# ------------------------------------------------------------------ InfiniPipe Algorithm 1

def test_infinipipe_mesh_rounding_mistake_is_caught(monkeypatch):
    import test_oracle_infinipipe as TI
    from oracle import infinipipe as IP

    def split_longest_floor(Lmax, K, cost):
        total = cost.prefix_cost(Lmax)
        b = [0]
        for k in range(1, K):
            m = 0
            while float(K) * cost.prefix_cost(IP.TILE * (m + 1)) <= float(k) * total:
                m += 1
            b.append(IP.TILE * m)                            # rounds down instead of to the nearest
        b.append(Lmax)
        if any(not b[i] < b[i + 1] for i in range(K)):
            raise IP.PlanError("collapsed")
        return b
    monkeypatch.setattr(IP, "split_longest", split_longest_floor)
    assert fails(TI.test_mesh_equal_cost_point, 1e-9, 3e-4) or fails(TI.test_hand_worked_packing)


def test_infinipipe_bucket_order_mistake_is_caught(monkeypatch):
    import test_oracle_infinipipe as TI
    from oracle import infinipipe as IP

    def bfd_most_loaded_first(buckets, shorts, T_t, T_m, cost):
        for idx, s in shorts:
            t = cost.slice_time(0, s)
            while True:
                if not buckets or min(b.tot_tokens for b in buckets) + s > T_m:
                    nb = IP.Bucket(order=len(buckets), tail=False)
                    nb.members.append((idx, 0, s))
                    nb.tot_time = cost.beta1 + t
                    nb.tot_tokens = s
                    buckets.append(nb)
                    break
                placed = False
                # buckets by decreasing tot_time/tot_tokens instead of increasing
                for b in sorted(buckets, key=lambda x: (-x.metric(), x.order)):
                    if b.tot_time + t <= T_t and b.tot_tokens + s <= T_m:
                        b.members.append((idx, 0, s))
                        b.tot_time += t
                        b.tot_tokens += s
                        placed = True
                        break
                if placed:
                    break
                T_t = min(b.tot_time for b in buckets if b.tot_tokens + s <= T_m) + t
        return T_t
    monkeypatch.setattr(IP, "bfd", bfd_most_loaded_first)
    assert fails(TI.test_bucket_order_is_increasing_time_per_token)


# ------------------------------------------------------------------ more of the planner

def test_key_pairs_mistake_is_caught(monkeypatch):
    def key_pairs_off_by_one(q_begin, q_end, ctx_begin, K):
        n = q_end - q_begin
        A_ = min(K, q_begin) - ctx_begin
        B = max(0, K - q_begin)
        return A_ * n + B * n - B * (B + 1) // 2                 # one diagonal too few
    monkeypatch.setattr(P, "key_pairs_before", key_pairs_off_by_one)
    assert fails(TP.test_key_pairs_closed_form_matches_counting)


def test_resplit_rounding_mistake_is_caught(monkeypatch):
    def resplit_floor(q_begin, q_end, ctx_begin, Pn):
        W = P.key_pairs_before(q_begin, q_end, ctx_begin, q_end)
        k = [ctx_begin]
        for p in range(1, Pn):
            m = 0
            while True:
                nxt = ctx_begin + P.TILE * (m + 1)               # rounds down instead of to the nearest
                if nxt > q_end or Pn * P.key_pairs_before(q_begin, q_end, ctx_begin, nxt) > p * W:
                    break
                m += 1
            k.append(ctx_begin + P.TILE * m)
        k.append(q_end)
        if any(not k[i] < k[i + 1] for i in range(Pn)):
            raise P.PlanError("collapsed")
        return k
    monkeypatch.setattr(P, "resplit_boundaries", resplit_floor)
    assert (fails(TP.test_resplit_causal_chunk_closed_form, 131072, 3)
            or fails(TP.test_resplit_context_dominated_chunk_by_hand) or fails(TP.test_plan_multiplex))


def test_varlen_chunk_count_mistake_is_caught(monkeypatch):
    real = P.boundaries

    def boundaries_one_chunk_short(L, N, mode):                  # floor(L_d / cap) chunks, at least one
        return real(L, max(1, N - 1) if N > 1 else N, mode)
    monkeypatch.setattr(P, "boundaries", boundaries_one_chunk_short)
    assert fails(TP.test_varlen_plan_structure) or fails(TP.test_golden_plans)


# ------------------------------------------------------------------ more of the attention oracle

def test_chunk_backward_mistake_is_caught(monkeypatch):
    def chunk_backward_without_context(q, k, v, do, qb, qe, cb, scale, row_block=512):
        # keys before the chunk dropped: context treated as absent
        dq, dk, dv = A_chunk_backward_ref(q, k, v, do, qb, qe, qb, scale, row_block)
        pad = np.zeros((qb - cb, dk.shape[1]))
        return dq, np.vstack([pad, dk]), np.vstack([pad, dv])
    A_chunk_backward_ref = A.chunk_backward
    monkeypatch.setattr(A, "chunk_backward", chunk_backward_without_context)
    assert fails(TA.test_chunk_backward_matches_autograd, 170, 300, 100)


def test_grouped_backward_mistake_is_caught(monkeypatch):
    def grouped_last_head_only(qs, k, v, dos, scale, cu_seqlens=None, row_block=512):
        dqs, Os, Ls = [], [], []
        for q, do in zip(qs, dos):
            dq, dk, dv, O, L = A.backward(q, k, v, do, scale, cu_seqlens, row_block)
            dqs.append(dq)
            Os.append(O)
            Ls.append(L)
        return dqs, dk, dv, Os, Ls                               # the group's sum dropped
    monkeypatch.setattr(A, "grouped_backward", grouped_last_head_only)
    assert fails(TA.test_grouped_backward_matches_autograd, 4, None)


def test_sampled_rows_mistake_is_caught(monkeypatch):
    real = A.doc_start_of_rows

    def starts_ignore_documents(T, cu_seqlens):
        return real(T, None)                                     # every row sees from token 0
    monkeypatch.setattr(A, "doc_start_of_rows", starts_ignore_documents)
    assert fails(TA.test_sampled_forms_match_full)


def test_partial_mask_mistake_is_caught(monkeypatch):
    real = A.partial

    def partial_strict(q, k, v, r0, r1, kv_lo, kv_hi, scale):
        # a key range ending one key early: the diagonal key of the last part lost
        return real(q, k, v, r0, r1, kv_lo, max(kv_lo, kv_hi - 1) if kv_hi == r1 else kv_hi, scale)
    monkeypatch.setattr(A, "partial", partial_strict)
    assert fails(TA.test_chunked_equals_unchunked, P.FLOPS)


# ------------------------------------------------------------------ more of Algorithm 1

def test_infinipipe_sharding_mistake_is_caught(monkeypatch):
    import test_oracle_infinipipe as TI
    from oracle import infinipipe as IP

    def split_by_mesh_ge(lengths, mesh):
        out = []
        for L in lengths:
            rem, ctx, slices = L, 0, []
            for m in mesh:
                if rem >= m:                                     # a slice equal to the remainder taken
                    slices.append((ctx, m))
                    ctx += m
                    rem -= m
                else:
                    break
            out.append((slices, (ctx, rem) if slices else None))
        return out
    monkeypatch.setattr(IP, "split_by_mesh", split_by_mesh_ge)
    assert fails(TI.test_page_example_sharding_by_mesh)


def test_infinipipe_cost_mistake_is_caught(monkeypatch):
    import test_oracle_infinipipe as TI
    from oracle import infinipipe as IP

    def slice_time_without_context(self, C, s):
        return self.alpha1 * float(s * s) + self.alpha2 * float(s)   # the context's cross term dropped
    monkeypatch.setattr(IP.Cost, "slice_time", slice_time_without_context)
    assert fails(TI.test_hand_worked_packing)


def test_infinipipe_threshold_mistake_is_caught(monkeypatch):
    import test_oracle_infinipipe as TI
    from oracle import infinipipe as IP

    def plan_threshold(lengths, K, token_cap, cost, pick):
        # Algorithm 1 with T_t started at pick() over the mesh slices' times
        # (the oracle takes the maximum); every other step as in the oracle
        starts = [0]
        for L in lengths:
            starts.append(starts[-1] + L)
        live = [i for i, L in enumerate(lengths) if L > 0]
        b = IP.split_longest(max(lengths), K, cost)
        mesh = [b[i + 1] - b[i] for i in range(K)]
        T_t = pick(cost.beta1 + cost.slice_time(b[i], mesh[i]) for i in range(K))
        parts = IP.split_by_mesh(lengths, mesh)
        buckets = []
        for i in live:
            slices, tail = parts[i]
            if tail is not None:
                bk = IP.Bucket(order=len(buckets), tail=True)
                bk.members.append((i, tail[0], tail[1]))
                bk.tot_time = cost.beta1 + cost.slice_time(tail[0], tail[1])
                bk.tot_tokens = tail[1]
                buckets.append(bk)
        shorts = sorted(((i, lengths[i]) for i in live if parts[i][1] is None),
                        key=lambda x: (-cost.slice_time(0, x[1]), x[0]))
        T_t = IP.bfd(buckets, shorts, T_t, token_cap, cost)
        calls, times = [], []
        depth = max(len(parts[i][0]) for i in live)
        for j in range(depth):
            for i in live:
                if j < len(parts[i][0]):
                    ctx, m = parts[i][0][j]
                    calls.append([(starts[i] + ctx, starts[i] + ctx + m, starts[i], 0)])
                    times.append(cost.beta1 + cost.slice_time(ctx, m))
        for bk in buckets:
            calls.append(sorted((starts[i] + ctx, starts[i] + ctx + s_, starts[i], 0) for i, ctx, s_ in bk.members))
            times.append(bk.tot_time)
        return calls, {"mesh": mesh, "T_t": T_t, "T_m": token_cap, "times": times}

    cost = IP.Cost(1.0, 0.0, 0.0)
    for lengths in ([1024, 300, 256, 200, 128, 100], [1024, 800, 700, 100]):   # the copy is the oracle
        assert plan_threshold(lengths, 2, 2048, cost, max) == IP.plan(lengths, 2, 2048, cost)
    monkeypatch.setattr(IP, "plan", lambda lengths, K, cap, cost: plan_threshold(lengths, K, cap, cost, min))
    assert fails(TI.test_threshold_starts_at_the_costliest_mesh_slice)


# ------------------------------------------------------------------ closed forms at full size

def test_periodic_queries_suffix_mistake_is_caught(monkeypatch):
    def suffix_exclusive(x):
        # sums over t > j: the diagonal query of every key dropped
        out = np.cumsum(x[::-1], axis=0)[::-1]
        return out - x
    monkeypatch.setattr(A, "_suffix_sums", suffix_exclusive)
    assert fails(TA.test_periodic_queries_closed_form_matches_definition, 130, 7, 32)


def test_periodic_queries_class_mistake_is_caught(monkeypatch):
    real = A.periodic_queries

    def classes_shifted(qc, k, v, do, scale):
        # row t read as class (t + 1) mod p: the query period misaligned
        return real(np.roll(np.asarray(qc), -1, axis=0), k, v, do, scale)
    monkeypatch.setattr(A, "periodic_queries", classes_shifted)
    assert fails(TA.test_periodic_queries_closed_form_matches_definition, 700, 3, 16)
