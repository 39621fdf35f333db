"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: sampled query rows (O, LSE, dQ) that the oracle computes row
by row, sampled keys near the sequence end (dK, dV), whole documents of the
packed batch, and invariants that hold at any size:
    sum_j dK_j = 0  and  sum_j dV_j = sum_t dO_t   per (head, document),
because softmax rows sum to one and dS rows sum to zero."""
import numpy as np
import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300.workloads import WORKLOADS, workload_inputs
from oracle import attention as A
from oracle import plan as P

from parity import GRAD_REL_L2, check_fwd, check_grad, head, lse_head, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(cca._lib.LIB_PATH):
        from chunked_causal_attention_gb300 import build
        build.build()


def plan_of(w):
    if w.packed:
        return cca.attn_plan_varlen(w.cu_seqlens(), w.max_chunk_tokens, w.mode)
    return cca.attn_plan(w.L, w.N, w.mode)


def sampled_rows_check(w, q, k, v, do, o, lse, dq, n_rows, seed, what):
    rng = np.random.default_rng(seed)
    heads = rng.integers(0, w.H, n_rows)
    rows = rng.integers(0, w.L, n_rows)
    cu = w.cu_seqlens()
    go, gl, gq, ro, rl, rq = [], [], [], [], [], []
    for h in np.unique(heads):
        r = rows[heads == h]
        qh, kh, vh, doh = (head(x, 0, int(h), w.packed) for x in (q, k, v, do))
        o_ref, l_ref = A.forward_rows(qh, kh, vh, r, w.scale, cu)
        dq_ref = A.dq_rows(qh, kh, vh, doh, r, w.scale, cu)
        go.append(head(o, 0, int(h), w.packed)[r]); gl.append(lse_head(lse, 0, int(h))[r])
        gq.append(head(dq, 0, int(h), w.packed)[r])
        ro.append(o_ref); rl.append(l_ref); rq.append(dq_ref)
    check_fwd(np.concatenate(go), np.concatenate(gl), np.concatenate(ro), np.concatenate(rl), what)
    check_grad(np.concatenate(gq), np.concatenate(rq), what + " dQ")


def invariants_check(w, q, do, dk, dv, what):
    """sum_j dV_j = sum_t dO_t and sum_j dK_j = 0 per (head, document). The
    tolerance is relative to the size of the summed terms: bf16 rounding of P
    (relative 2^-8) and of the dK/dV outputs leaves a deviation of order
    2^-8 * sqrt(sum of squared terms), far below a missing or doubled tile.
    Measured sum-dV deviations grow with the accumulation length: 8.7e-5 at
    32K, 1.8e-4 at 128K, 1.2e-3 at 1M tokens; a missing 128-key tile gives
    more than 1e-1."""
    cu = w.cu_seqlens() or [0, w.L]
    worst_v = worst_k = 0.0
    for h in range(w.H):
        dkh = head(dk, 0, h, w.packed)
        dvh = head(dv, 0, h, w.packed)
        doh = head(do, 0, h, w.packed)
        qh = head(q, 0, h, w.packed)
        for s, e in zip(cu[:-1], cu[1:]):
            sv = dvh[s:e].sum(axis=0) - doh[s:e].sum(axis=0)
            nv = np.linalg.norm(sv) / np.sqrt((doh[s:e] ** 2).sum())
            sk = dkh[s:e].sum(axis=0)
            nk = np.linalg.norm(sk) / (w.scale * np.sqrt((qh[s:e] ** 2).sum()) + np.sqrt((dkh[s:e] ** 2).sum()))
            worst_v, worst_k = max(worst_v, nv), max(worst_k, nk)
            assert nv <= 5e-3, f"{what} sum dV h{h} doc {s}: {nv}"
            assert nk <= 1e-2, f"{what} sum dK h{h} doc {s}: {nk}"
    print(f"[parity] {what} invariants: sum dV rel {worst_v:.3e}, sum dK rel {worst_k:.3e}")


def tail_keys_check(w, q, k, v, do, dk, dv, heads, n_keys, seed, what):
    rng = np.random.default_rng(seed)
    keys = np.sort(rng.choice(np.arange(w.L - 1024, w.L), n_keys, replace=False))
    keys[-1] = w.L - 1                         # the last key: P_tt * dO_t only
    gk, gv, rk, rv = [], [], [], []
    for h in heads:
        qh, kh, vh, doh = (head(x, 0, h, w.packed) for x in (q, k, v, do))
        dk_ref, dv_ref = A.dkdv_keys(qh, kh, vh, doh, keys, w.scale, w.cu_seqlens())
        gk.append(head(dk, 0, h, w.packed)[keys]); gv.append(head(dv, 0, h, w.packed)[keys])
        rk.append(dk_ref); rv.append(dv_ref)
    check_grad(np.concatenate(gk), np.concatenate(rk), what + " dK")
    check_grad(np.concatenate(gv), np.concatenate(rv), what + " dV")


def test_7b_32k():
    w = WORKLOADS["7b_32k"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = plan_of(w)
    assert chunks == P.plan(w.L, w.N, w.mode)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks)
    # head 0 in full (every row and key), the others on sampled rows
    qh, kh, vh, doh = (head(x, 0, 0, False) for x in (q, k, v, do))
    rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, w.scale, None, row_block=1024)
    check_fwd(head(o, 0, 0, False), lse_head(lse, 0, 0), ro, rl, "32k h0")
    check_grad(head(dq, 0, 0, False), rdq, "32k dQ h0")
    check_grad(head(dk, 0, 0, False), rdk, "32k dK h0")
    check_grad(head(dv, 0, 0, False), rdv, "32k dV h0")
    sampled_rows_check(w, q, k, v, do, o, lse, dq, 1024, 5, "32k")
    invariants_check(w, q, do, dk, dv, "32k")
    assert cca.attn_status(cca.workspace(cca.shape_of(q), chunks, 0)) in (0,)


def test_7b_128k():
    w = WORKLOADS["7b_128k"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = plan_of(w)
    assert chunks == P.plan(w.L, w.N, w.mode) and chunks[0][3] and chunks[-1][3]
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks)
    sampled_rows_check(w, q, k, v, do, o, lse, dq, 4096, 6, "128k")
    # rows on both sides of the two re-split points
    for m in (chunks[0][3], chunks[-1][3]):
        r = np.array([m - 2, m - 1, m, m + 1])
        qh, kh, vh = (head(x, 0, 3, False) for x in (q, k, v))
        ro, rl = A.forward_rows(qh, kh, vh, r, w.scale)
        check_fwd(head(o, 0, 3, False)[r], lse_head(lse, 0, 3)[r], ro, rl, f"128k split {m}")
    tail_keys_check(w, q, k, v, do, dk, dv, [0, 17], 48, 7, "128k")
    invariants_check(w, q, do, dk, dv, "128k")


def test_packed_256k():
    w = WORKLOADS["packed_256k"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = plan_of(w)
    assert chunks == P.plan_varlen(w.cu_seqlens(), w.max_chunk_tokens, w.mode)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks, packed=True)
    cu = w.cu_seqlens()
    # every document up to 16K tokens in full on head 5 (documents are independent)
    h = 5
    qh, kh, vh, doh = (head(x, 0, h, True) for x in (q, k, v, do))
    gl = lse_head(lse, 0, h)
    for s, e in zip(cu[:-1], cu[1:]):
        if e - s > 16384:
            continue
        rdq, rdk, rdv, ro, rl = A.backward(qh[s:e], kh[s:e], vh[s:e], doh[s:e], w.scale, None, row_block=1024)
        check_fwd(head(o, 0, h, True)[s:e], gl[s:e], ro, rl, f"packed doc {s}")
        check_grad(head(dq, 0, h, True)[s:e], rdq, f"packed dQ doc {s}")
        check_grad(head(dk, 0, h, True)[s:e], rdk, f"packed dK doc {s}")
        check_grad(head(dv, 0, h, True)[s:e], rdv, f"packed dV doc {s}")
    sampled_rows_check(w, q, k, v, do, o, lse, dq, 2048, 8, "packed")
    invariants_check(w, q, do, dk, dv, "packed")


@pytest.mark.slow
def test_13b_1m():
    w = WORKLOADS["13b_1m"]
    q, k, v, do = (x for x in workload_inputs(w, device="cuda"))
    chunks = plan_of(w)
    assert chunks == P.plan(w.L, w.N, w.mode)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks)
    sampled_rows_check(w, q, k, v, do, o, lse, dq, 4096, 9, "1m")
    tail_keys_check(w, q, k, v, do, dk, dv, [11], 16, 10, "1m")
    invariants_check(w, q, do, dk, dv, "1m")


@pytest.mark.parametrize("name", ["7b_128k", pytest.param("13b_1m", marks=pytest.mark.slow)])
def test_periodic_keys_every_row_and_key(name):
    """Keys repeating with period 3 (k_j = kc[j mod 3]) make the float64 oracle
    linear in T (oracle.attention.periodic_keys), so O, LSE, dQ are checked on
    every row and dV on every key at full size, including the first keys whose
    dV sums over the whole sequence."""
    from chunked_causal_attention_gb300.workloads import randn_bf16
    w = WORKLOADS[name]
    q, _, v, do = workload_inputs(w, device="cuda")
    p = 3
    kc = randn_bf16((w.B, w.H, p, w.D), w.seed * 4 + 7, device="cuda")
    k = kc[:, :, torch.arange(w.L, device="cuda") % p, :].contiguous()
    chunks = plan_of(w)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks)
    for h in (0, w.H - 1):
        kch = kc[0, h].float().cpu().numpy().astype(np.float64)
        ro, rl, rdq, rdv = A.periodic_keys(head(q, 0, h, False), kch, head(v, 0, h, False), head(do, 0, h, False),
                                           w.scale)
        check_fwd(head(o, 0, h, False), lse_head(lse, 0, h), ro, rl, f"{name} periodic h{h} all rows")
        gdq, gdv = head(dq, 0, h, False), head(dv, 0, h, False)
        check_grad(gdq, rdq, f"{name} periodic dQ h{h} all rows")
        check_grad(gdv, rdv, f"{name} periodic dV h{h} all keys")
        check_grad(gdv[:4096], rdv[:4096], f"{name} periodic dV h{h} first 4096 keys")
        check_grad(gdv[-4096:], rdv[-4096:], f"{name} periodic dV h{h} last 4096 keys")
