"""GPU parity, element by element, at sizes the float64 oracle finishes in
seconds: several 128-row tiles, ragged tails, packed documents down to one
token, re-split chunks, strided layouts, and the stage entry points.
Everything runs through the C ABI (libattn.so)."""
import numpy as np
import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from oracle import attention as A
from oracle import plan as P

from parity import check_fwd, check_grad, default_scale, docs_of, head, lse_head, rel_l2, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from chunked_causal_attention_gb300 import build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(cca._lib.LIB_PATH):
        build.build()


def full_check(q, k, v, do, chunks, packed, scale=None, backward=True, what=""):
    B = 1 if packed else q.shape[0]
    H = q.shape[1]
    D = q.shape[-1]
    sc = default_scale(D) if scale is None else scale
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, chunks, packed, scale, backward)
    cu = docs_of(chunks)
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = (head(x, b, h, packed) for x in (q, k, v, do))
            if backward:
                rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, sc, cu)
            else:
                ro, rl = A.forward(qh, kh, vh, sc, cu)
            check_fwd(head(o, b, h, packed), lse_head(lse, b, h), ro, rl, f"{what} b{b}h{h}")
            if backward:
                check_grad(head(dq, b, h, packed), rdq, f"{what} dQ b{b}h{h}")
                check_grad(head(dk, b, h, packed), rdk, f"{what} dK b{b}h{h}")
                check_grad(head(dv, b, h, packed), rdv, f"{what} dV b{b}h{h}")
    return o, lse, dq, dk, dv


def test_tiny_workload_full():
    w = WORKLOADS["tiny"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = cca.attn_plan(w.L, w.N, w.mode)
    assert chunks == P.plan(w.L, w.N, w.mode)
    full_check(q, k, v, do, chunks, False, what="tiny")


@pytest.mark.parametrize("L", [1, 7, 129, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode,N", [(0, 1), (0, 3), (1, 2), (2, 1), (2, 3)])
def test_ragged_dense(L, D, mode, N):
    try:
        chunks = P.plan(L, N, mode)
    except P.PlanError:
        pytest.skip("plan does not exist for this L")
    q, k, v, do = (x.cuda() for x in make_inputs(2, 3, L, D, seed=100 + L + D))
    full_check(q, k, v, do, chunks, False, what=f"L{L} D{D} m{mode} N{N}")


def test_token_major_strides():
    """[B, L, H, D] storage (token stride H*D, head stride D) via the strided ABI."""
    B, L, H, D = 2, 700, 3, 128
    base = [x.cuda() for x in make_inputs(B, H, L, D, seed=7)]
    tm = [x.permute(0, 2, 1, 3).contiguous() for x in base]        # [B, L, H, D]
    views = [x.permute(0, 2, 1, 3) for x in tm]                      # logical [B, H, L, D] view
    chunks = P.plan(L, 3, P.FLOPS_RESPLIT_EDGES)
    o, lse, dq, dk, dv = full_check(*views, chunks, False, what="token-major")
    o2, lse2, dq2, dk2, dv2 = run_gpu(*base, chunks)
    assert torch.equal(o.contiguous(), o2) and torch.equal(lse, lse2)
    assert torch.equal(dk.contiguous(), dk2) and torch.equal(dv.contiguous(), dv2)


@pytest.mark.parametrize("mct,mode", [(128, 1), (256, 2), (1000, 0), (16384, 1)])
def test_packed_documents(mct, mode):
    lens = [1, 1, 127, 129, 300, 1, 700, 2, 1000]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    try:
        chunks = P.plan_varlen(cu, mct, mode)
    except P.PlanError:
        pytest.skip("no plan")
    assert cca.attn_plan_varlen(cu, mct, mode) == chunks
    assert docs_of(chunks) == cu
    q, k, v, do = (x.cuda() for x in make_inputs(1, 4, cu[-1], 128, seed=21, packed=True))
    full_check(q, k, v, do, chunks, True, what=f"packed mct{mct} m{mode}")


def test_forward_partial_coverage_and_arbitrary_splits():
    """Chunks that cover part of the rows, with re-split points that are not
    multiples of 128 and one that lies before q_begin; untouched rows keep
    their contents."""
    L, H, D = 1100, 2, 128
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=33))
    chunks = [(0, 200, 0, 77), (300, 700, 0, 150), (700, 1001, 0, 901), (1001, 1100, 1001, 0)]
    shape = cca.shape_of(q)
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, H, L), 9.0, device=q.device)
    ws = cca.workspace(shape, chunks, 0)
    cca.attn_fwd(q, k, v, chunks, shape, o, lse, ws)
    torch.cuda.synchronize()
    sc = default_scale(D)
    for h in range(H):
        qh, kh, vh = (head(x, 0, h, False) for x in (q, k, v))
        for qb, qe, cb, m in chunks:
            ro, rl = A.chunked_forward(qh, kh, vh, [(qb, qe, cb, m)], sc)
            check_fwd(head(o, 0, h, False)[qb:qe], lse_head(lse, 0, h)[qb:qe], ro[qb:qe], rl[qb:qe], "partial")
        assert torch.all(o[0, h, 200:300] == 7.0) and torch.all(lse[0, h, 200:300] == 9.0)


def test_stage_entry_points_equal_composed_calls():
    L, H, D = 2000, 2, 128
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=44))
    chunks = P.plan(L, 3, P.FLOPS_RESPLIT_EDGES)
    shape = cca.shape_of(q)
    o, lse = cca.forward(q, k, v, chunks)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    ws = cca.workspace(shape, chunks, 0)
    cca.attn_fwd_tiles(q, k, v, chunks, shape, o2, lse2, ws)
    cca.attn_fwd_merge(chunks, shape, o2, lse2, ws)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    wsb = cca.workspace(shape, chunks, 1)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    cca.attn_bwd_prep(o, do, chunks, shape, wsb)
    cca.attn_bwd_tiles(q, k, v, lse, do, chunks, shape, dk2, dv2, wsb)
    cca.attn_bwd_dq(chunks, shape, dq2, wsb)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)       # one CTA owns each key tile
    assert (dq.float() - dq2.float()).abs().max().item() <= 2e-2   # fp32 atomics: order may differ
    assert cca.attn_status(ws) == 0 and cca.attn_status(wsb) == 0


def test_kernel_launch_count_per_call():
    """Each stage call enqueues its kernel plus one copy kernel per 31 KB of work
    list it writes into the workspace, and the library counts exactly those."""
    L, H, D = 2000, 2, 128
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=44))
    chunks = P.plan(L, 3, P.FLOPS_RESPLIT_EDGES)
    assert any(c[3] for c in chunks)
    shape = cca.shape_of(q)
    o, lse = torch.empty_like(q), torch.empty((1, H, L), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws, wsb = cca.workspace(shape, chunks, 0), cca.workspace(shape, chunks, 1)

    def delta(fn):
        n0 = cca.kernel_launches()
        fn()
        return cca.kernel_launches() - n0

    assert delta(lambda: cca.attn_fwd_tiles(q, k, v, chunks, shape, o, lse, ws)) == 2       # items + tiles
    assert delta(lambda: cca.attn_fwd_merge(chunks, shape, o, lse, ws)) == 3                # segs, bounds + merge
    assert delta(lambda: cca.attn_bwd_prep(o, do, chunks, shape, wsb)) == 2                 # rows + prep
    assert delta(lambda: cca.attn_bwd_tiles(q, k, v, lse, do, chunks, shape, dk, dv, wsb)) == 2
    assert delta(lambda: cca.attn_bwd_dq(chunks, shape, dq, wsb)) == 2
    # 1024 forward items of 32 bytes: the work list takes two copy kernels
    T = 131072
    q1, k1, v1, _ = (x.cuda() for x in make_inputs(1, 1, T, 64, seed=45))
    ch = P.plan(T, 1, P.UNIFORM)
    sh = cca.shape_of(q1)
    o1, l1 = torch.empty_like(q1), torch.empty((1, 1, T), dtype=torch.float32, device="cuda")
    assert delta(lambda: cca.attn_fwd_tiles(q1, k1, v1, ch, sh, o1, l1, cca.workspace(sh, ch, 0))) == 3
    torch.cuda.synchronize()
    assert cca.attn_status(ws) == 0 and cca.attn_status(wsb) == 0


def test_backward_independent_of_chunk_cuts():
    L, H, D = 1500, 2, 64
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=55))
    c1 = P.plan(L, 1, P.FLOPS)
    c2 = P.plan(L, 5, P.FLOPS_RESPLIT_EDGES)
    o, lse = cca.forward(q, k, v, c1)
    _, _, dk1, dv1 = (None,) + cca.backward(q, k, v, o, lse, do, c1)
    _, _, dk2, dv2 = (None,) + cca.backward(q, k, v, o, lse, do, c2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)


def test_host_errors_with_device_memory():
    L, H, D = 512, 1, 128
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=66))
    chunks = P.plan(L, 2, P.FLOPS)
    shape = cca.shape_of(q)
    o, lse = torch.empty_like(q), torch.empty(1, H, L, device="cuda")
    ws = cca.workspace(shape, chunks, 0)
    with pytest.raises(cca.AttnError) as e:
        cca.attn_fwd(q, k, v, chunks, shape, o, lse, ws[:16])
    assert e.value.status == 4
    flat = torch.empty(q.numel() + 1, dtype=torch.bfloat16, device="cuda")
    qm = flat[1:].view_as(q)                                   # 2-byte offset: not 16-byte aligned
    with pytest.raises(cca.AttnError) as e:
        cca.attn_fwd(qm, k, v, chunks, shape, o, lse, ws)
    assert e.value.status == 2
    assert cca.attn_status(ws) == 0


def test_repeated_runs_bit_identical():
    """O, LSE, dK and dV have no order-dependent reduction, so repeated runs
    must agree bit for bit; a synchronisation race between the warp roles of a
    tile kernel shows up here as a run-to-run difference."""
    L, H, D = 8192, 8, 128
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=77))
    chunks = P.plan(L, 4, P.FLOPS_RESPLIT_EDGES)
    ref = None
    for _ in range(6):
        o, lse = cca.forward(q, k, v, chunks)
        dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
        torch.cuda.synchronize()
        if ref is None:
            ref = (o.clone(), lse.clone(), dk.clone(), dv.clone())
            continue
        assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])
        assert torch.equal(dk, ref[2]) and torch.equal(dv, ref[3])


@pytest.mark.parametrize("D", [64, 96, 128])
def test_p_part_resplits(D):
    """Key ranges re-split into P parts of equal pair count (kv_split = -P),
    including chunks with a long context and chunks whose parts end off the
    128-row grid of the queries; every row against the oracle."""
    L, H = 2300, 2
    chunks = [(0, 640, 0, -3), (640, 1000, 0, -3), (1000, 1100, 0, -5), (1100, 2300, 0, -2)]
    assert all(P.key_ranges(c) for c in chunks)
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=77 + D))
    full_check(q, k, v, do, chunks, False, what=f"P-part D{D}")


def test_p_part_resplits_packed_and_multiplex_plan():
    lens = [2000, 1, 900, 1500]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    chunks = [(0, 1000, 0, -3), (1000, 2000, 0, -4), (2000, 2001, 2000, 0), (2001, 2901, 2001, -2),
              (2901, 4401, 2901, -6)]
    q, k, v, do = (x.cuda() for x in make_inputs(1, 3, cu[-1], 128, seed=78, packed=True))
    full_check(q, k, v, do, chunks, True, what="P-part packed")
    plan = cca.attn_plan_multiplex(3000, 6, 4)
    assert plan == P.plan_multiplex(3000, 6, 4) and plan[0][3] < 0
    q, k, v, do = (x.cuda() for x in make_inputs(1, 2, 3000, 128, seed=79))
    full_check(q, k, v, do, plan, False, what="multiplex plan")


@pytest.mark.parametrize("D", [8, 40, 80, 96, 120])
def test_head_dims_between_tile_widths(D):
    """Head dims that are not 64 or 128 run on the 64- or 128-wide tiles with
    the dims past D loaded as zeros: dense rows with ragged tiles and an edge
    re-split (the merge path), then packed documents, every row against the
    oracle."""
    q, k, v, do = (x.cuda() for x in make_inputs(2, 3, 1000, D, seed=90 + D))
    full_check(q, k, v, do, P.plan(1000, 3, P.FLOPS_RESPLIT_EDGES), False, what=f"D{D} dense")
    lens = [1, 127, 129, 300, 700]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    q, k, v, do = (x.cuda() for x in make_inputs(1, 2, cu[-1], D, seed=95 + D, packed=True))
    full_check(q, k, v, do, P.plan_varlen(cu, 256, P.FLOPS_RESPLIT_EDGES), True, what=f"D{D} packed")


@pytest.mark.parametrize("D", [136, 192, 256])
def test_wide_head_dims(D):
    """Head dims above 128 run on 256-wide tiles: the forward with 64-key K/V
    tiles, the backward with each 128-key tile split into two work items by
    output dims and 64-query blocks. Dense rows with ragged tiles and an edge
    re-split (the merge path of 256-wide rows), P-part re-splits, packed
    documents with one-token and off-grid documents, grouped key/value heads
    and chunk-streamed calls (fp32 dK/dV accumulators), every row and key
    against the oracle."""
    q, k, v, do = (x.cuda() for x in make_inputs(2, 3, 1000, D, seed=190 + D))
    full_check(q, k, v, do, P.plan(1000, 3, P.FLOPS_RESPLIT_EDGES), False, what=f"D{D} dense")
    q, k, v, do = (x.cuda() for x in make_inputs(1, 2, 1500, D, seed=191 + D))
    full_check(q, k, v, do, [(0, 700, 0, -4), (700, 1100, 0, -3), (1100, 1500, 0, 0)], False, what=f"D{D} P-part")
    lens = [1, 63, 65, 127, 129, 300, 700]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    q, k, v, do = (x.cuda() for x in make_inputs(1, 2, cu[-1], D, seed=195 + D, packed=True))
    full_check(q, k, v, do, P.plan_varlen(cu, 256, P.FLOPS_RESPLIT_EDGES), True, what=f"D{D} packed")
    # grouped key/value heads: 4 query heads on 2 key/value heads; dK/dV of a
    # key/value head sum over its query heads
    L, H, Hkv = 640, 4, 2
    q, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=197 + D)[0:4:3])
    k, v = (x.cuda() for x in make_inputs(1, Hkv, L, D, seed=198 + D)[1:3])
    chunks = P.plan(L, 2, P.FLOPS)
    o, lse = cca.forward(q, k, v, chunks)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    sc = default_scale(D)
    for hk in range(Hkv):
        hs = range(2 * hk, 2 * hk + 2)
        rdqs, rdk, rdv, ros, rls = A.grouped_backward([head(q, 0, h, False) for h in hs], head(k, 0, hk, False),
                                                      head(v, 0, hk, False), [head(do, 0, h, False) for h in hs],
                                                      sc, None)
        for g, h in enumerate(hs):
            check_fwd(head(o, 0, h, False), lse_head(lse, 0, h), ros[g], rls[g], f"D{D} grouped h{h}")
            check_grad(head(dq, 0, h, False), rdqs[g], f"D{D} grouped dQ h{h}")
        check_grad(head(dk, 0, hk, False), rdk, f"D{D} grouped dK hk{hk}")
        check_grad(head(dv, 0, hk, False), rdv, f"D{D} grouped dV hk{hk}")
    # chunk-streamed calls: forward per chunk, backward per chunk in reverse order
    # with the fp32 accumulators; every key row is emitted from its accumulator
    chunks = P.plan(1000, 4, P.FLOPS_RESPLIT_EDGES)
    q, k, v, do = (x.cuda() for x in make_inputs(1, 2, 1000, D, seed=199 + D))
    o, lse = cca.forward_streamed(q, k, v, chunks)
    dq, dk, dv, dk_acc, dv_acc = cca.backward_streamed(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk_acc.to(torch.bfloat16)) and torch.equal(dv, dv_acc.to(torch.bfloat16))
    for h in range(2):
        qh, kh, vh, doh = (head(x, 0, h, False) for x in (q, k, v, do))
        rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, sc, None)
        check_fwd(head(o, 0, h, False), lse_head(lse, 0, h), ro, rl, f"D{D} streamed h{h}")
        check_grad(head(dq, 0, h, False), rdq, f"D{D} streamed dQ h{h}")
        check_grad(head(dk, 0, h, False), rdk, f"D{D} streamed dK h{h}")
        check_grad(head(dv, 0, h, False), rdv, f"D{D} streamed dV h{h}")


def test_head_dim_padding_leaves_neighbours_untouched():
    """With D = 80 on the 128-wide tiles, the dims past D of a row are never
    written: rows of a wider buffer viewed with D = 80 keep their tail."""
    L, H, D, W = 700, 2, 80, 128
    base = [x.cuda() for x in make_inputs(1, H, L, W, seed=97)]
    views = [x[..., :D] for x in base]                               # strides of the W-wide buffer
    chunks = P.plan(L, 2, P.FLOPS_RESPLIT_EDGES)
    shape = cca.shape_of(views[0])
    o_buf = torch.full((1, H, L, W), 5.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, H, L), dtype=torch.float32, device="cuda")
    ws = cca.workspace(shape, chunks, 0)
    cca.attn_fwd(*views[:3], chunks, shape, o_buf[..., :D], lse, ws)
    grads = [torch.full((1, H, L, W), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    wsb = cca.workspace(shape, chunks, 1)
    cca.attn_bwd(*views[:3], o_buf[..., :D], lse, views[3], chunks, shape, *(g[..., :D] for g in grads), wsb)
    torch.cuda.synchronize()
    assert cca.attn_status(ws) == 0 and cca.attn_status(wsb) == 0
    assert torch.all(o_buf[..., D:] == 5.0)
    for g in grads:
        assert torch.all(g[..., D:] == 3.0)
    o, lse2, dq, dk, dv = full_check(*views, chunks, False, what="D80 in a 128-wide buffer")
    assert torch.equal(o_buf[..., :D], o) and torch.equal(lse, lse2)


def test_concurrent_calls_on_two_streams():
    """The calls that take a caller workspace keep no state that changes a
    result between calls (attn_fwd_noalloc shares one library-held scratch
    area among its calls, as its header says): two problems run at the same
    time on two streams, each with its own workspace, give what they give one
    after the other (O, LSE, dK, dV bit for bit; dQ, whose fp32
    reduce-adds run in any order, within the tolerance)."""
    cases = [(1, 4, 3000, 128, P.plan(3000, 3, P.FLOPS_RESPLIT_EDGES), 401),
             (2, 3, 2000, 64, P.plan(2000, 2, P.FLOPS), 402)]
    inputs = [[x.cuda() for x in make_inputs(B, H, L, D, seed=sd)] for B, H, L, D, _, sd in cases]
    serial = []
    for (q, k, v, do), c in zip(inputs, cases):
        o, lse = cca.forward(q, k, v, c[4])
        dq, dk, dv = cca.backward(q, k, v, o, lse, do, c[4])
        serial.append((o, lse, dq, dk, dv))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [None, None]
    for rep in range(3):
        for i, ((q, k, v, do), c) in enumerate(zip(inputs, cases)):
            with torch.cuda.stream(streams[i]):
                o, lse = cca.forward(q, k, v, c[4], stream=streams[i])
                dq, dk, dv = cca.backward(q, k, v, o, lse, do, c[4], stream=streams[i])
                outs[i] = (o, lse, dq, dk, dv)
        torch.cuda.synchronize()
        for i in range(2):
            o, lse, dq, dk, dv = outs[i]
            so, slse, sdq, sdk, sdv = serial[i]
            assert torch.equal(o, so) and torch.equal(lse, slse), (rep, i)
            assert torch.equal(dk, sdk) and torch.equal(dv, sdv), (rep, i)
            assert rel_l2(dq.float().cpu().numpy(), sdq.float().cpu().numpy()) < 1e-3, (rep, i)


def test_empty_chunk_list():
    """No chunks: the forward enqueues nothing and leaves its outputs as they
    were; the backward, which needs a partition of [0, T), refuses it on the
    host (ATTN_E_INVAL) before anything is enqueued."""
    L, H, D = 300, 2, 64
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=41))
    shape = cca.shape_of(q)
    ws = cca.workspace(shape, [], 0)
    o = torch.full_like(q, 2.0)
    lse = torch.full((1, H, L), 3.0, device="cuda")
    cca.attn_fwd(q, k, v, [], shape, o, lse, ws)
    torch.cuda.synchronize()
    assert cca.attn_status(ws) == 0
    assert torch.all(o == 2.0) and torch.all(lse == 3.0)
    with pytest.raises(cca.AttnError) as e:
        cca.attn_workspace_size(shape, [], 1)
    assert e.value.status == 1
