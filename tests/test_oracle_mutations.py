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
