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

from parity import (GRAD_REL_L2, check_fwd, check_grad, head, invariants_check, lse_head, plan_of, run_gpu,
                    sampled_rows_check, tail_keys_check)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(cca._lib.LIB_PATH):
        from chunked_causal_attention_gb300 import build
        build.build()


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


def test_d256_32k():
    """256-dim heads at 32K tokens (the split backward's items walk up to 512
    query blocks): head 0 in full, sampled rows of the others, invariants."""
    w = WORKLOADS["d256_32k"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = plan_of(w)
    assert chunks == P.plan(w.L, w.N, w.mode)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks)
    qh, kh, vh, doh = (head(x, 0, 0, False) for x in (q, k, v, do))
    rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, w.scale, None, row_block=1024)
    check_fwd(head(o, 0, 0, False), lse_head(lse, 0, 0), ro, rl, "d256 h0")
    check_grad(head(dq, 0, 0, False), rdq, "d256 dQ h0")
    check_grad(head(dk, 0, 0, False), rdk, "d256 dK h0")
    check_grad(head(dv, 0, 0, False), rdv, "d256 dV h0")
    sampled_rows_check(w, q, k, v, do, o, lse, dq, 512, 7, "d256")
    invariants_check(w, q, do, dk, dv, "d256")


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


def test_7b_128k_multiplex_plan():
    """The 128K workload with SPPO Table 3 edge re-splits for 4 pipeline
    stages (chunks 0 and 15 in four key parts, 1 and 14 in three, 2 and 13 in
    two): sampled rows and rows around every part boundary of the first chunk."""
    w = WORKLOADS["7b_128k"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = cca.attn_plan_multiplex(w.L, w.N, 4)
    assert chunks == P.plan_multiplex(w.L, w.N, 4)
    assert [c[3] for c in chunks[:3]] == [-4, -3, -2] and [c[3] for c in chunks[-3:]] == [-2, -3, -4]
    o, lse = cca.forward(q, k, v, chunks)
    torch.cuda.synchronize()
    sampled_rows_check(w, q, k, v, do, o, lse, None, 2048, 13, "128k multiplex", backward=False)
    kb = P.resplit_boundaries(chunks[0][0], chunks[0][1], 0, 4)
    r = np.array(sorted({x + d for x in kb[1:-1] for d in (-1, 0, 1)}))
    qh, kh, vh = (head(x, 0, 9, False) for x in (q, k, v))
    ro, rl = A.forward_rows(qh, kh, vh, r, w.scale)
    check_fwd(head(o, 0, 9, False)[r], lse_head(lse, 0, 9)[r], ro, rl, "128k multiplex boundaries")


@pytest.mark.parametrize("name", ["7b_128k", pytest.param("13b_1m", marks=pytest.mark.slow)])
def test_periodic_queries_every_key_and_row(name):
    """Queries repeating with period 3 (q_t = qc[t mod 3]) with random keys,
    values and dO make the float64 oracle linear in T
    (oracle.attention.periodic_queries), so dK and dV are checked on every key
    and O and LSE on every row, of two heads at full size: in the benchmark's
    launch configuration and plan. The first keys' dK sums over every later
    query of the sequence (the longest accumulation the backward does)."""
    from chunked_causal_attention_gb300.workloads import randn_bf16
    w = WORKLOADS[name]
    _, k, v, do = workload_inputs(w, device="cuda")
    p = 3
    qc = randn_bf16((w.B, w.H, p, w.D), w.seed * 4 + 9, device="cuda")
    q = qc[:, :, torch.arange(w.L, device="cuda") % p, :].contiguous()
    chunks = plan_of(w)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks)
    for h in (0, w.H - 1):
        qch = qc[0, h].float().cpu().numpy().astype(np.float64)
        ro, rl, rdk, rdv = A.periodic_queries(qch, head(k, 0, h, False), head(v, 0, h, False),
                                              head(do, 0, h, False), w.scale)
        check_fwd(head(o, 0, h, False), lse_head(lse, 0, h), ro, rl, f"{name} periodic-q h{h} all rows")
        gdk, gdv = head(dk, 0, h, False), head(dv, 0, h, False)
        check_grad(gdk, rdk, f"{name} periodic-q dK h{h} all keys")
        check_grad(gdv, rdv, f"{name} periodic-q dV h{h} all keys")
        check_grad(gdk[:4096], rdk[:4096], f"{name} periodic-q dK h{h} first 4096 keys")
        check_grad(gdk[-4096:], rdk[-4096:], f"{name} periodic-q dK h{h} last 4096 keys")
        # every 128-key tile on its own: no tile's dK may hide behind the whole-head norm
        worst = max(float(np.linalg.norm(gdk[t:t + 128] - rdk[t:t + 128]) / np.linalg.norm(rdk[t:t + 128]))
                    for t in range(0, w.L, 128))
        assert worst <= GRAD_REL_L2, f"{name} periodic-q dK h{h} worst 128-key tile rel-L2 {worst}"
        print(f"[parity] {name} periodic-q dK h{h}: worst 128-key tile rel-L2 {worst:.3e}")
