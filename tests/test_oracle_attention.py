"""Pins of the float64 attention oracle (no GPU).

Each check is independent of the oracle's own formula: pure-Python brute force,
torch float64 library routines (scaled_dot_product_attention, logsumexp,
autograd), closed forms that Q = 0 gives, per-row invariants, central finite
differences, and the chunked method's equality with the plain definition.
"""
import math
import random

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import plan as P


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def docs_cu(T, seed, n_docs):
    rng = random.Random(seed)
    cuts = sorted(rng.sample(range(1, T), n_docs - 1))
    return [0] + cuts + [T]


# ----------------------------------------------------------------- brute force

def brute_forward(q, k, v, scale, cu):
    T, D = len(q), len(q[0])
    start = [0] * T
    for d in range(len(cu) - 1):
        for t in range(cu[d], cu[d + 1]):
            start[t] = cu[d]
    O = [[0.0] * len(v[0]) for _ in range(T)]
    LSE = [0.0] * T
    for t in range(T):
        s = [scale * sum(q[t][x] * k[j][x] for x in range(D)) for j in range(start[t], t + 1)]
        z = sum(math.exp(x) for x in s)
        LSE[t] = math.log(z)
        for i, j in enumerate(range(start[t], t + 1)):
            p = math.exp(s[i]) / z
            for x in range(len(v[0])):
                O[t][x] += p * v[j][x]
    return np.array(O), np.array(LSE)


@pytest.mark.parametrize("T,D,cu", [(17, 5, None), (40, 8, [0, 7, 8, 31, 40]), (64, 4, [0, 64])])
def test_forward_matches_brute_force(T, D, cu):
    q, k, v = rand((T, D), 1), rand((T, D), 2), rand((T, D), 3)
    scale = 1 / math.sqrt(D)
    O, L = A.forward(q, k, v, scale, cu, row_block=7)
    Ob, Lb = brute_forward(q.tolist(), k.tolist(), v.tolist(), scale, cu or [0, T])
    np.testing.assert_allclose(O, Ob, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L, Lb, atol=1e-12, rtol=0)


# ---------------------------------------------------- torch float64 routines

def torch_ref(q, k, v, do, scale, cu):
    T = q.shape[0]
    mask = torch.zeros(T, T, dtype=torch.bool)
    for s, e in zip(cu[:-1], cu[1:]):
        mask[s:e, s:e] = torch.tril(torch.ones(e - s, e - s, dtype=torch.bool))
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=mask[None, None], scale=scale)[0, 0]
    o.backward(torch.tensor(do, dtype=torch.float64))
    scores = (tq @ tk.T * scale).masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(scores, dim=1)
    return (o.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy())


@pytest.mark.parametrize("T,D,ndocs", [(300, 64, 1), (512, 128, 1), (257, 32, 5), (200, 16, 12)])
def test_against_torch_sdpa_and_autograd(T, D, ndocs):
    q, k, v, do = (rand((T, D), s) for s in (10, 11, 12, 13))
    cu = [0, T] if ndocs == 1 else docs_cu(T, 3, ndocs)
    scale = 1 / math.sqrt(D)
    O, L = A.forward(q, k, v, scale, cu, row_block=64)
    dq, dk, dv, O2, L2 = A.backward(q, k, v, do, scale, cu, row_block=48)
    to, tl, tdq, tdk, tdv = torch_ref(q, k, v, do, scale, cu)
    for a, b in ((O, to), (L, tl), (O2, to), (L2, tl), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, atol=1e-10, rtol=1e-10)


# ------------------------------------------------------ closed forms, invariants

def test_q_zero_closed_form():
    T, D = 300, 16
    cu = [0, 1, 120, 300]
    k, v, do = rand((T, D), 4), rand((T, D), 5), rand((T, D), 6)
    q = np.zeros((T, D))
    O, L = A.forward(q, k, v, 0.25, cu, row_block=50)
    dq, dk, dv, _, _ = A.backward(q, k, v, do, 0.25, cu, row_block=50)
    for s, e in zip(cu[:-1], cu[1:]):
        for t in range(s, e):
            np.testing.assert_allclose(O[t], v[s:t + 1].mean(axis=0), atol=1e-12)
            assert abs(L[t] - math.log(t - s + 1)) < 1e-12
        for j in range(s, e):
            expect = sum(do[t] / (t - s + 1) for t in range(j, e))
            np.testing.assert_allclose(dv[j], expect, atol=1e-12)
    np.testing.assert_allclose(dk, 0.0, atol=1e-12)


def test_rows_sum_to_one_and_first_row():
    T, D = 200, 32
    cu = [0, 50, 51, 200]
    q, k = rand((T, D), 7), rand((T, D), 8)
    O, L = A.forward(q, k, np.ones((T, 3)), 0.3, cu)
    np.testing.assert_allclose(O, 1.0, atol=1e-12)           # softmax rows sum to 1
    v = rand((T, D), 9)
    O, L = A.forward(q, k, v, 0.3, cu)
    for s in cu[:-1]:
        np.testing.assert_allclose(O[s], v[s], atol=1e-12)
        assert abs(L[s] - 0.3 * q[s] @ k[s]) < 1e-12


def test_shift_invariances():
    T, D, sc = 150, 8, 0.4
    q, k, v = rand((T, D), 1), rand((T, D), 2), rand((T, D), 3)
    c = rand((D,), 4)
    O, L = A.forward(q, k, v, sc)
    O2, L2 = A.forward(q, k + c, v, sc)
    np.testing.assert_allclose(O2, O, atol=1e-12)
    np.testing.assert_allclose(L2, L + sc * (q @ c), atol=1e-12)
    O3, L3 = A.forward(q, k, v + c, sc)
    np.testing.assert_allclose(O3, O + c, atol=1e-12)
    np.testing.assert_allclose(L3, L, atol=1e-12)


def test_backward_invariants_and_last_key():
    T, D, sc = 240, 16, 0.25
    cu = [0, 100, 101, 240]
    q, k, v, do = (rand((T, D), s) for s in (21, 22, 23, 24))
    dq, dk, dv, O, L = A.backward(q, k, v, do, sc, cu, row_block=33)
    for s, e in zip(cu[:-1], cu[1:]):
        np.testing.assert_allclose(dk[s:e].sum(axis=0), 0.0, atol=1e-11)
        np.testing.assert_allclose(dv[s:e].sum(axis=0), do[s:e].sum(axis=0), atol=1e-11)
        t = e - 1
        p = math.exp(sc * q[t] @ k[t] - L[t])
        ds = p * (do[t] @ v[t] - do[t] @ O[t])
        np.testing.assert_allclose(dv[t], p * do[t], atol=1e-12)
        np.testing.assert_allclose(dk[t], sc * ds * q[t], atol=1e-12)


def test_finite_differences():
    T, D, sc, h = 24, 6, 0.45, 1e-6
    cu = [0, 9, 24]
    q, k, v, do = (rand((T, D), s) for s in (31, 32, 33, 34))
    dq, dk, dv, _, _ = A.backward(q, k, v, do, sc, cu, row_block=5)

    def loss(qq, kk, vv):
        return float(np.sum(do * A.forward(qq, kk, vv, sc, cu)[0]))

    rng = np.random.default_rng(0)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(12):
            t, x = int(rng.integers(T)), int(rng.integers(D))
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][t, x] += h
            args_m[which][t, x] -= h
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[t, x]) < 1e-7, (which, t, x, fd, grad[t, x])


# ---------------------------------------------------- the chunked method

@pytest.mark.parametrize("mode", [P.UNIFORM, P.FLOPS, P.FLOPS_RESPLIT_EDGES])
def test_chunked_equals_unchunked(mode):
    T, D, sc = 1000, 16, 0.25
    q, k, v = rand((T, D), 41), rand((T, D), 42), rand((T, D), 43)
    O, L = A.forward(q, k, v, sc)
    for N in (1, 2, 3, 5):
        chunks = P.plan(T, N, mode)
        for kvb in (None, 128, 100):
            Oc, Lc = A.chunked_forward(q, k, v, chunks, sc, kv_block=kvb)
            np.testing.assert_allclose(Oc, O, atol=1e-12)
            np.testing.assert_allclose(Lc, L, atol=1e-12)


def test_chunked_varlen_equals_unchunked():
    T, D, sc = 900, 8, 0.3
    cu = [0, 3, 3, 410, 411, 900]
    q, k, v = rand((T, D), 51), rand((T, D), 52), rand((T, D), 53)
    O, L = A.forward(q, k, v, sc, cu)
    for mode in (P.UNIFORM, P.FLOPS, P.FLOPS_RESPLIT_EDGES):
        chunks = P.plan_varlen(cu, 200, mode)
        Oc, Lc = A.chunked_forward(q, k, v, chunks, sc)
        np.testing.assert_allclose(Oc, O, atol=1e-12)
        np.testing.assert_allclose(Lc, L, atol=1e-12)


def test_merge_with_empty_part():
    """Rows before the re-split point see no key of part B: LSE_B = -inf must
    get weight 0 and leave part A's result unchanged."""
    T, D, sc = 512, 8, 0.3
    q, k, v = rand((T, D), 61), rand((T, D), 62), rand((T, D), 63)
    oa, la = A.partial(q, k, v, 0, T, 0, 256, sc)
    ob, lb = A.partial(q, k, v, 0, T, 256, T, sc)
    assert np.all(np.isneginf(lb[:256])) and np.all(ob[:256] == 0)
    o, l = A.lse_merge([(oa, la), (ob, lb)])
    np.testing.assert_array_equal(o[:256], oa[:256])
    np.testing.assert_array_equal(l[:256], la[:256])
    O, L = A.forward(q, k, v, sc)
    np.testing.assert_allclose(o, O, atol=1e-12)
    np.testing.assert_allclose(l, L, atol=1e-12)
    # all parts empty -> -inf LSE, zero output
    o0, l0 = A.lse_merge([(np.zeros((2, 3)), np.full(2, -np.inf))] * 2)
    assert np.all(np.isneginf(l0)) and np.all(o0 == 0)


# ---------------------------------------------------- sampled forms

def test_sampled_forms_match_full():
    T, D, sc = 700, 16, 0.25
    cu = [0, 333, 700]
    q, k, v, do = (rand((T, D), s) for s in (71, 72, 73, 74))
    dq, dk, dv, O, L = A.backward(q, k, v, do, sc, cu)
    rows = [0, 1, 332, 333, 334, 699, 500]
    Or, Lr = A.forward_rows(q, k, v, rows, sc, cu)
    np.testing.assert_allclose(Or, O[rows], atol=1e-12)
    np.testing.assert_allclose(Lr, L[rows], atol=1e-12)
    np.testing.assert_allclose(A.dq_rows(q, k, v, do, rows, sc, cu), dq[rows], atol=1e-12)
    keys = [332, 330, 699, 600, 334]
    dkk, dvk = A.dkdv_keys(q, k, v, do, keys, sc, cu, row_block=50)
    np.testing.assert_allclose(dkk, dk[keys], atol=1e-12)
    np.testing.assert_allclose(dvk, dv[keys], atol=1e-12)


def test_pair_count():
    pairs = P.causal_pairs(0, 131072, 0)
    assert pairs == 131072 * 131073 // 2 == 8590000128


@pytest.mark.parametrize("T,p,D", [(700, 3, 16), (257, 1, 8), (130, 7, 32)])
def test_periodic_keys_closed_form_matches_definition(T, p, D):
    q, v, do = rand((T, D), 81), rand((T, D), 82), rand((T, D), 83)
    kc = rand((p, D), 84)
    k = kc[np.arange(T) % p]
    sc = 1 / math.sqrt(D)
    dq, dk, dv, O, L = A.backward(q, k, v, do, sc, None, row_block=64)
    Op, Lp, dqp, dvp = A.periodic_keys(q, kc, v, do, sc)
    for a, b in ((Op, O), (Lp, L), (dqp, dq), (dvp, dv)):
        np.testing.assert_allclose(a, b, atol=1e-10, rtol=1e-10)


@pytest.mark.parametrize("T,p,D", [(700, 3, 16), (257, 1, 8), (130, 7, 32), (5, 9, 4)])
def test_periodic_queries_closed_form_matches_definition(T, p, D):
    """The periodic-queries closed form against the plain definition
    (A.backward, itself pinned to brute force, torch and finite differences),
    including a period longer than the sequence."""
    k, v, do = rand((T, D), 85), rand((T, D), 86), rand((T, D), 87)
    qc = rand((p, D), 88)
    q = qc[np.arange(T) % p]
    sc = 1 / math.sqrt(D)
    dq, dk, dv, O, L = A.backward(q, k, v, do, sc, None, row_block=64)
    Op, Lp, dkp, dvp = A.periodic_queries(qc, k, v, do, sc)
    for a, b in ((Op, O), (Lp, L), (dkp, dk), (dvp, dv)):
        np.testing.assert_allclose(a, b, atol=1e-10, rtol=1e-10)


def test_periodic_queries_against_autograd():
    """Library pin: torch float64 SDPA and autograd on the periodic queries,
    with large scores (scale 1) so that the shift by each class's maximum
    matters."""
    T, p, D = 300, 4, 16
    k, v, do = rand((T, D), 95), rand((T, D), 96), rand((T, D), 97)
    qc = 2.0 * rand((p, D), 98)
    q = qc[np.arange(T) % p]
    o, lse, _, tdk, tdv = torch_ref(q, k, v, do, 1.0, [0, T])
    Op, Lp, dkp, dvp = A.periodic_queries(qc, k, v, do, 1.0)
    for a, b in ((Op, o), (Lp, lse), (dkp, tdk), (dvp, tdv)):
        np.testing.assert_allclose(a, b, atol=1e-9, rtol=1e-9)


# ---------------------------------------------------- chunk-streamed backward

def torch_chunk_grads(q, k, v, do, qb, qe, cb, sc):
    """Library pin: torch float64 autograd of sum(dO . O) over the chunk's rows
    only, O from an explicitly masked softmax of the chunk's queries against
    its context keys [cb, qe)."""
    Q = torch.tensor(q[qb:qe], dtype=torch.float64, requires_grad=True)
    K = torch.tensor(k[cb:qe], dtype=torch.float64, requires_grad=True)
    V = torch.tensor(v[cb:qe], dtype=torch.float64, requires_grad=True)
    t = torch.arange(qb, qe)[:, None]
    j = torch.arange(cb, qe)[None, :]
    S = (Q @ K.T) * sc
    S = S.masked_fill(j > t, float("-inf"))
    O = torch.softmax(S, dim=-1) @ V
    (O * torch.tensor(do[qb:qe], dtype=torch.float64)).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("qb,qe,cb", [(0, 96, 0), (130, 257, 0), (300, 301, 0), (170, 300, 100)])
def test_chunk_backward_matches_autograd(qb, qe, cb):
    T, D, sc = 301, 8, 0.35
    q, k, v, do = (rand((T, D), s) for s in (81, 82, 83, 84))
    dq, dk, dv = A.chunk_backward(q, k, v, do, qb, qe, cb, sc, row_block=40)
    tq, tk, tv = torch_chunk_grads(q, k, v, do, qb, qe, cb, sc)
    np.testing.assert_allclose(dq, tq, atol=1e-11)
    np.testing.assert_allclose(dk, tk, atol=1e-11)
    np.testing.assert_allclose(dv, tv, atol=1e-11)


@pytest.mark.parametrize("mode", [P.UNIFORM, P.FLOPS, P.FLOPS_RESPLIT_EDGES])
def test_chunk_backward_streamed_equals_full(mode):
    """Chunks processed in reverse order: summed contributions equal the
    plain backward, and after chunk c has run, the keys of chunk c hold their
    final gradients (later chunks have all contributed already)."""
    T, D, sc = 1000, 16, 0.25
    for docs, chunks in (([0, T], P.plan(T, 4, mode)),
                         ([0, 3, 3, 410, 411, T], P.plan_varlen([0, 3, 3, 410, 411, T], 200, mode))):
        q, k, v, do = (rand((T, D), s) for s in (91, 92, 93, 94))
        dq, dk, dv, _, _ = A.backward(q, k, v, do, sc, docs)
        adk, adv, gq = np.zeros_like(dk), np.zeros_like(dv), np.zeros_like(dq)
        for qb, qe, cb, _m in reversed(chunks):
            cq, ck, cv = A.chunk_backward(q, k, v, do, qb, qe, cb, sc)
            gq[qb:qe] = cq
            adk[cb:qe] += ck
            adv[cb:qe] += cv
            np.testing.assert_allclose(adk[qb:qe], dk[qb:qe], atol=1e-12)
            np.testing.assert_allclose(adv[qb:qe], dv[qb:qe], atol=1e-12)
        np.testing.assert_allclose(gq, dq, atol=1e-12)
        np.testing.assert_allclose(adk, dk, atol=1e-12)
        np.testing.assert_allclose(adv, dv, atol=1e-12)


# ---------------------------------------------------- grouped key/value heads

@pytest.mark.parametrize("G,cu", [(4, None), (3, [0, 50, 51, 120]), (1, None)])
def test_grouped_backward_matches_autograd(G, cu):
    """GQA/MQA: G query heads share one key/value head. Library pin: torch
    float64 SDPA of each query head against the shared K, V tensors (leaf
    tensors with requires_grad), whose .grad autograd sums over the heads."""
    T, D, sc = 120, 8, 0.3
    qs = [rand((T, D), 200 + g) for g in range(G)]
    dos = [rand((T, D), 300 + g) for g in range(G)]
    k, v = rand((T, D), 401), rand((T, D), 402)
    dqs, dk, dv, Os, Ls = A.grouped_backward(qs, k, v, dos, sc, cu)
    K = torch.tensor(k, requires_grad=True)
    V = torch.tensor(v, requires_grad=True)
    mask = torch.zeros(T, T, dtype=torch.bool)
    docs = cu or [0, T]
    for s_, e_ in zip(docs[:-1], docs[1:]):
        mask[s_:e_, s_:e_] = torch.tril(torch.ones(e_ - s_, e_ - s_, dtype=torch.bool))
    total = 0
    Qs = []
    for g in range(G):
        Q = torch.tensor(qs[g], requires_grad=True)
        Qs.append(Q)
        O = torch.nn.functional.scaled_dot_product_attention(Q[None, None], K[None, None], V[None, None],
                                                             attn_mask=mask, scale=sc)[0, 0]
        np.testing.assert_allclose(O.detach().numpy(), Os[g], atol=1e-12)
        total = total + (O * torch.tensor(dos[g])).sum()
    total.backward()
    for g in range(G):
        np.testing.assert_allclose(Qs[g].grad.numpy(), dqs[g], atol=1e-11)
    np.testing.assert_allclose(K.grad.numpy(), dk, atol=1e-11)
    np.testing.assert_allclose(V.grad.numpy(), dv, atol=1e-11)


def test_chunked_forward_with_p_part_resplits():
    """Chunks re-split into P parts of equal pair count (kv_split = -P) merge
    back to the plain definition."""
    T, D, sc = 1500, 8, 0.3
    q, k, v = rand((T, D), 71), rand((T, D), 72), rand((T, D), 73)
    O, L = A.forward(q, k, v, sc)
    chunks = [(0, 700, 0, -4), (700, 1100, 0, -3), (1100, 1500, 0, -2)]
    Oc, Lc = A.chunked_forward(q, k, v, chunks, sc)
    np.testing.assert_allclose(Oc, O, atol=1e-12)
    np.testing.assert_allclose(Lc, L, atol=1e-12)
    for ch in P.plan_multiplex(T, 3, 3):
        Op, Lp = A.chunked_forward(q, k, v, [ch], sc)
        np.testing.assert_allclose(Op[ch[0]:ch[1]], O[ch[0]:ch[1]], atol=1e-12)
