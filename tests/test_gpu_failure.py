"""Failure detection without a GPU fault.

Every mbarrier wait in the tile kernels is bounded. With the test-only
producer stall (ATTN_TEST_STALL_PRODUCER=1) no tile is ever loaded, so every
wait runs out after ATTN_WAIT_LIMIT_MS; the kernels record ATTN_E_TIMEOUT in
the workspace status word, release TMEM and return. The host reads the status,
and the same CUDA context then runs a normal forward and backward that match
the oracle.

Every kernel checks each work descriptor it reads from the workspace before it
forms an address from it. With ATTN_TEST_INCONSISTENT_ITEM=1 the host makes
one descriptor inconsistent in a way that addresses nothing outside the
buffers; the kernels report ATTN_E_BOUNDS."""
import numpy as np
import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300.workloads import make_inputs
from oracle import attention as A
from oracle import plan as P

from parity import check_fwd, check_grad, default_scale, head, lse_head

pytestmark = pytest.mark.gpu

ATTN_E_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(cca._lib.LIB_PATH):
        from chunked_causal_attention_gb300 import build
        build.build()


@pytest.mark.parametrize("D", [128, 256])
def test_stalled_producer_times_out_and_context_survives(monkeypatch, D):
    """D = 256 runs the 256-wide forward and the backward split by output dims."""
    L, H = 2048, 2
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=88))
    chunks = P.plan(L, 2, P.FLOPS)
    shape = cca.shape_of(q)
    o, lse = torch.zeros_like(q), torch.zeros(1, H, L, device="cuda")
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(q), torch.zeros_like(q)
    ws_f = cca.workspace(shape, chunks, 0)
    ws_b = cca.workspace(shape, chunks, 1)

    monkeypatch.setenv("ATTN_WAIT_LIMIT_MS", "200")
    monkeypatch.setenv("ATTN_TEST_STALL_PRODUCER", "1")
    cca.attn_fwd(q, k, v, chunks, shape, o, lse, ws_f)          # enqueues and returns ATTN_OK
    assert cca.attn_status(ws_f) == ATTN_E_TIMEOUT
    assert cca.attn_status(ws_f) == 0                           # read clears the word
    cca.attn_bwd(q, k, v, o, lse, do, chunks, shape, dq, dk, dv, ws_b)
    assert cca.attn_status(ws_b) == ATTN_E_TIMEOUT

    monkeypatch.delenv("ATTN_TEST_STALL_PRODUCER")
    monkeypatch.delenv("ATTN_WAIT_LIMIT_MS")
    o, lse = cca.forward(q, k, v, chunks)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    sc = default_scale(D)
    for h in range(H):
        qh, kh, vh, doh = (head(x, 0, h, False) for x in (q, k, v, do))
        rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, sc)
        check_fwd(head(o, 0, h, False), lse_head(lse, 0, h), ro, rl, f"after timeout h{h}")
        check_grad(head(dq, 0, h, False), rdq, f"after timeout dQ h{h}")
        check_grad(head(dk, 0, h, False), rdk, f"after timeout dK h{h}")
        check_grad(head(dv, 0, h, False), rdv, f"after timeout dV h{h}")


ATTN_E_BOUNDS = 7


@pytest.mark.parametrize("D", [128, 256])
def test_inconsistent_work_item_is_reported_and_not_used(monkeypatch, D):
    """Device-side index checks. With the test-only switch the first work item
    of each tile kernel gets an empty row range (forward: r1 = r0; backward:
    q_end = q_lo), a descriptor that addresses nothing outside the buffers but
    does not fit the shape's rules. Every role of the kernel checks the item
    before forming an address from it, records ATTN_E_BOUNDS and stops. The
    item's output rows keep their sentinel values (nothing was written for
    it), and the same CUDA context then runs a normal forward and backward.
    D = 256 runs the 256-wide forward and the backward split by output dims,
    where both work items of the key tile (its two halves of dims) stop."""
    L, H = 2048, 2
    q, k, v, do = (x.cuda() for x in make_inputs(1, H, L, D, seed=89))
    chunks = P.plan(L, 2, P.FLOPS)
    shape = cca.shape_of(q)
    nan = float("nan")
    o, lse = torch.full_like(q, nan), torch.full((1, H, L), nan, device="cuda")
    dq, dk, dv = torch.full_like(q, nan), torch.full_like(q, nan), torch.full_like(q, nan)
    ws_f = cca.workspace(shape, chunks, 0)
    ws_b = cca.workspace(shape, chunks, 1)
    o_good, lse_good = cca.forward(q, k, v, chunks)

    monkeypatch.setenv("ATTN_TEST_INCONSISTENT_ITEM", "1")
    cca.attn_fwd(q, k, v, chunks, shape, o, lse, ws_f)
    assert cca.attn_status(ws_f) == ATTN_E_BOUNDS
    # the first forward item is the heaviest: the last 128 rows of head 0
    assert torch.isnan(o[0, 0, L - 128:].float()).all() and torch.isnan(lse[0, 0, L - 128:]).all()
    cca.attn_bwd(q, k, v, o_good, lse_good, do, chunks, shape, dq, dk, dv, ws_b)
    assert cca.attn_status(ws_b) == ATTN_E_BOUNDS
    # the first backward item is the heaviest: key tile 0 of head 0 (all its dims)
    assert torch.isnan(dk[0, 0, :128].float()).all() and torch.isnan(dv[0, 0, :128].float()).all()

    monkeypatch.delenv("ATTN_TEST_INCONSISTENT_ITEM")
    o, lse = cca.forward(q, k, v, chunks)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    sc = default_scale(D)
    for h in range(H):
        qh, kh, vh, doh = (head(x, 0, h, False) for x in (q, k, v, do))
        rdq, rdk, rdv, ro, rl = A.backward(qh, kh, vh, doh, sc)
        check_fwd(head(o, 0, h, False), lse_head(lse, 0, h), ro, rl, f"after index check h{h}")
        check_grad(head(dq, 0, h, False), rdq, f"after index check dQ h{h}")
        check_grad(head(dk, 0, h, False), rdk, f"after index check dK h{h}")
        check_grad(head(dv, 0, h, False), rdv, f"after index check dV h{h}")
