"""GPU parity of the chunk-streamed calls: the forward one chunk at a time in
chunk order (attn_fwd with a single chunk against the resident keys before
it) and the backward one chunk at a time in reverse order (attn_bwd_chunk,
fp32 dK/dV accumulators shared across calls; InfiniPipe §II-A: a token's K/V
gradients gather every later token). Checked element by element against the
float64 oracle on small cases, per call against the oracle's per-chunk
contributions, and on sampled rows and keys at the benchmark's 128K size."""
import numpy as np
import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from oracle import attention as A
from oracle import plan as P

from parity import (check_fwd, check_grad, default_scale, docs_of, head, invariants_check, lse_head,
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


def streamed_check(q, k, v, do, chunks, packed, what):
    B = 1 if packed else q.shape[0]
    H, D = q.shape[1], q.shape[-1]
    sc = default_scale(D)
    o, lse = cca.forward_streamed(q, k, v, chunks, packed=packed)
    dq, dk, dv, dk_acc, dv_acc = cca.backward_streamed(q, k, v, o, lse, do, chunks, packed=packed)
    torch.cuda.synchronize()
    # the whole-call forward computes every row tile the same way
    o1, lse1 = cca.forward(q, k, v, chunks, packed=packed)
    torch.cuda.synchronize()
    assert torch.equal(o, o1) and torch.equal(lse, lse1)
    # every key row was emitted from its accumulator
    assert torch.equal(dk, dk_acc.to(torch.bfloat16)) and torch.equal(dv, dv_acc.to(torch.bfloat16))
    cu = docs_of(chunks)
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = (head(x, b, h, packed) for x in (q, k, v, do))
            rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, sc, cu)
            check_fwd(head(o, b, h, packed), lse_head(lse, b, h), ro, rl, f"{what} b{b}h{h}")
            check_grad(head(dq, b, h, packed), rdq, f"{what} dQ b{b}h{h}")
            check_grad(head(dk, b, h, packed), rdk, f"{what} dK b{b}h{h}")
            check_grad(head(dv, b, h, packed), rdv, f"{what} dV b{b}h{h}")


@pytest.mark.parametrize("L", [129, 1000, 2500])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode,N", [(0, 3), (1, 4), (2, 5)])
def test_streamed_dense(L, D, mode, N):
    try:
        chunks = P.plan(L, N, mode)
    except P.PlanError:
        pytest.skip("plan does not exist for this L")
    q, k, v, do = (x.cuda() for x in make_inputs(2, 2, L, D, seed=300 + L + D + N))
    streamed_check(q, k, v, do, chunks, False, f"streamed L{L} D{D} m{mode} N{N}")


def test_streamed_packed_documents():
    lens = [1, 127, 129, 300, 1, 700, 2, 1000]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    chunks = P.plan_varlen(cu, 256, P.FLOPS_RESPLIT_EDGES)
    q, k, v, do = (x.cuda() for x in make_inputs(1, 3, cu[-1], 128, seed=301, packed=True))
    streamed_check(q, k, v, do, chunks, True, "streamed packed")


def test_chunk_boundaries_off_the_tile_grid():
    """Chunk cuts that are not multiples of 128: a key tile then straddles the
    cut (keys before it are context, keys after it the chunk's own)."""
    L, H, D = 1100, 2, 128
    chunks = [(0, 300, 0, 0), (300, 650, 0, 0), (650, 1001, 0, 800), (1001, 1100, 0, 0)]
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=302))
    streamed_check(q, k, v, do, chunks, False, "streamed off-grid")


def test_one_call_against_oracle_contributions():
    """A single call for the last chunk: dq rows, the fp32 accumulators over
    the context, and the bf16 rows it emits; rows it must not touch keep
    their contents."""
    L, H, D = 1500, 2, 128
    qb, qe, cb = 1000, 1500, 200
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=303))
    docs = [(0, 200, 0, 0), (200, 1000, 200, 0), (1000, 1500, 200, 0)]
    o, lse = cca.forward(q, k, v, docs)
    shape = cca.shape_of(q)
    dq = torch.full_like(q, 3.0)
    dk, dv = torch.full_like(k, 5.0), torch.full_like(v, 6.0)
    dk_acc = torch.full(k.shape, 7.0, dtype=torch.float32, device=k.device)
    dv_acc = torch.full(v.shape, 7.0, dtype=torch.float32, device=v.device)
    dk_acc[:, :, cb:qe] = 0
    dv_acc[:, :, cb:qe] = 0
    ws = cca.workspace(shape, [(qb, qe, cb, 0)], cca.PASS_BWD_CHUNK)
    cca.attn_bwd_chunk(q, k, v, o, lse, do, [(qb, qe, cb, 0)], shape, dq, dk, dv, dk_acc, dv_acc, ws)
    torch.cuda.synchronize()
    assert cca.attn_status(ws) == 0
    sc = default_scale(D)
    for h in range(H):
        qh, kh, vh, doh = (head(x, 0, h, False) for x in (q, k, v, do))
        cq, ck, cv = A.chunk_backward(qh, kh, vh, doh, qb, qe, cb, sc)
        check_grad(head(dq, 0, h, False)[qb:qe], cq, f"one call dQ h{h}")
        check_grad(dk_acc[0, h, cb:qe].double().cpu().numpy(), ck, f"one call dK acc h{h}")
        check_grad(dv_acc[0, h, cb:qe].double().cpu().numpy(), cv, f"one call dV acc h{h}")
    assert torch.equal(dk[:, :, qb:qe], dk_acc[:, :, qb:qe].to(torch.bfloat16))
    assert torch.equal(dv[:, :, qb:qe], dv_acc[:, :, qb:qe].to(torch.bfloat16))
    assert torch.all(dq[:, :, :qb] == 3.0) and torch.all(dk[:, :, :qb] == 5.0) and torch.all(dv[:, :, :qb] == 6.0)
    assert torch.all(dk_acc[:, :, :cb] == 7.0) and torch.all(dv_acc[:, :, :cb] == 7.0)


def test_streamed_7b_128k_sampled():
    """The benchmark's 128K workload streamed chunk by chunk (16 forward and 16
    backward calls), checked on sampled rows, tail keys and the invariants."""
    w = WORKLOADS["7b_128k"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = cca.attn_plan(w.L, w.N, w.mode)
    o, lse = cca.forward_streamed(q, k, v, chunks)
    dq, dk, dv, dk_acc, dv_acc = cca.backward_streamed(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    del dk_acc, dv_acc
    sampled_rows_check(w, q, k, v, do, o, lse, dq, 2048, 11, "streamed 128k")
    tail_keys_check(w, q, k, v, do, dk, dv, [5], 32, 12, "streamed 128k")
    invariants_check(w, q, do, dk, dv, "streamed 128k")


def test_calls_holding_several_documents():
    """Calls that hold slices of several documents (InfiniPipe batched and
    hybrid chunks {C, S}): a long document split into three slices, whose
    tail shares a call with two short documents; another call batches three
    short documents. Forward in call order, backward in reverse."""
    lens = [1500, 200, 77, 300, 129, 1]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    L = cu[-1]
    long0 = [(0, 700, 0, 0), (700, 1150, 0, 0)]                      # split chunks of document 0
    hybrid = [(1150, 1500, 0, 0), (1500, 1700, 1500, 0), (1700, 1777, 1700, 0)]   # tail + two short docs
    batched = [(1777, 2077, 1777, 0), (2077, 2206, 2077, 0), (2206, 2207, 2206, 0)]
    calls = [[long0[0]], batched, [long0[1]], hybrid]
    q, k, v, do = (x.cuda() for x in make_inputs(1, 2, L, 128, seed=304, packed=True))
    o, lse = cca.forward_streamed(q, k, v, calls, packed=True)
    dq, dk, dv, dk_acc, dv_acc = cca.backward_streamed(q, k, v, o, lse, do, calls, packed=True)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk_acc.to(torch.bfloat16)) and torch.equal(dv, dv_acc.to(torch.bfloat16))
    sc = default_scale(128)
    for h in range(2):
        qh, kh, vh, doh = (head(x, 0, h, True) for x in (q, k, v, do))
        rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, sc, cu)
        check_fwd(head(o, 0, h, True), lse_head(lse, 0, h), ro, rl, f"calls h{h}")
        check_grad(head(dq, 0, h, True), rdq, f"calls dQ h{h}")
        check_grad(head(dk, 0, h, True), rdk, f"calls dK h{h}")
        check_grad(head(dv, 0, h, True), rdv, f"calls dV h{h}")


def test_infinipipe_plan_streamed():
    """Calls planned by InfiniPipe Algorithm 1 (split chunks, hybrid chunks
    holding a tail slice with short sequences, batched chunks), run one call
    at a time, against the oracle."""
    from oracle import infinipipe as IP
    lens = [3000, 1, 700, 129, 2500, 40, 900, 64, 300, 1100]
    cost = (1e-9, 2e-5, 0.0)
    calls = cca.attn_plan_infinipipe(lens, 3, 4096, *cost)
    want, _ = IP.plan(lens, 3, 4096, IP.Cost(*cost))
    assert calls == [list(c) for c in want]
    assert any(len(c) > 1 and c[0][0] > c[0][2] for c in calls)          # a hybrid chunk
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    q, k, v, do = (x.cuda() for x in make_inputs(1, 2, cu[-1], 128, seed=305, packed=True))
    o, lse = cca.forward_streamed(q, k, v, calls, packed=True)
    dq, dk, dv, _, _ = cca.backward_streamed(q, k, v, o, lse, do, calls, packed=True)
    torch.cuda.synchronize()
    sc = default_scale(128)
    for h in range(2):
        qh, kh, vh, doh = (head(x, 0, h, True) for x in (q, k, v, do))
        rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, sc, cu)
        check_fwd(head(o, 0, h, True), lse_head(lse, 0, h), ro, rl, f"infinipipe h{h}")
        check_grad(head(dq, 0, h, True), rdq, f"infinipipe dQ h{h}")
        check_grad(head(dk, 0, h, True), rdk, f"infinipipe dK h{h}")
        check_grad(head(dv, 0, h, True), rdv, f"infinipipe dV h{h}")


@pytest.mark.parametrize("D", [40, 96])
def test_streamed_head_dims_between_tile_widths(D):
    """Chunk-streamed calls with fp32 dK/dV accumulators of a head dim that
    is neither 64 nor 128."""
    chunks = P.plan(1000, 4, P.FLOPS_RESPLIT_EDGES)
    q, k, v, do = (x.cuda() for x in make_inputs(2, 2, 1000, D, seed=310 + D))
    streamed_check(q, k, v, do, chunks, False, f"streamed D{D}")


@pytest.mark.parametrize("L,N,PP", [(3000, 6, 4), (2600, 4, 3)])
def test_streamed_p_part_plan(L, N, PP):
    """Chunk-streamed calls of a plan whose edge chunks are re-split into P
    key parts (SPPO Table 3): every forward call merges its own parts."""
    chunks = cca.attn_plan_multiplex(L, N, PP)
    assert chunks == P.plan_multiplex(L, N, PP) and any(c[3] < 0 for c in chunks)
    q, k, v, do = (x.cuda() for x in make_inputs(2, 2, L, 128, seed=320 + L + PP))
    streamed_check(q, k, v, do, chunks, False, f"streamed multiplex L{L} N{N} PP{PP}")
