"""GPU parity with grouped key/value heads (GQA/MQA): H query heads read
H / Hkv key/value heads; the gradient of a key/value head is the sum over
its query heads (oracle.attention.grouped_backward, pinned to torch
autograd). Dense and packed layouts, MQA, token-major strides, the
chunk-streamed calls, and the 128K grouped workload on sampled rows."""
import numpy as np
import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from oracle import attention as A
from oracle import plan as P

from parity import check_fwd, check_grad, default_scale, docs_of, head, lse_head

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(cca._lib.LIB_PATH):
        from chunked_causal_attention_gb300 import build
        build.build()


def grouped_check(q, k, v, do, o, lse, dq, dk, dv, cu, packed, what):
    B = 1 if packed else q.shape[0]
    H, Hkv, D = q.shape[1], k.shape[1], q.shape[-1]
    G = H // Hkv
    sc = default_scale(D)
    for b in range(B):
        for hk in range(Hkv):
            hs = range(hk * G, hk * G + G)
            qs = [head(q, b, h, packed) for h in hs]
            dos = [head(do, b, h, packed) for h in hs]
            kh, vh = head(k, b, hk, packed), head(v, b, hk, packed)
            rdqs, rdk, rdv, ros, rls = A.grouped_backward(qs, kh, vh, dos, sc, cu)
            for g, h in enumerate(hs):
                check_fwd(head(o, b, h, packed), lse_head(lse, b, h), ros[g], rls[g], f"{what} b{b}h{h}")
                check_grad(head(dq, b, h, packed), rdqs[g], f"{what} dQ b{b}h{h}")
            check_grad(head(dk, b, hk, packed), rdk, f"{what} dK b{b}hk{hk}")
            check_grad(head(dv, b, hk, packed), rdv, f"{what} dV b{b}hk{hk}")


@pytest.mark.parametrize("L", [129, 1000])
@pytest.mark.parametrize("D", [48, 64, 96, 128])
@pytest.mark.parametrize("H,Hkv", [(8, 2), (4, 1), (3, 3)])
def test_grouped_dense(L, D, H, Hkv):
    chunks = P.plan(L, 1 if L < 300 else 3, P.FLOPS_RESPLIT_EDGES)
    q, k, v, do = (x.cuda() for x in make_inputs(2, H, L, D, seed=500 + L + D + H, Hkv=Hkv))
    o, lse = cca.forward(q, k, v, chunks)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    assert dk.shape == k.shape and dq.shape == q.shape
    grouped_check(q, k, v, do, o, lse, dq, dk, dv, None, False, f"gqa L{L} D{D} H{H}/{Hkv}")


def test_grouped_packed_and_streamed():
    lens = [1, 300, 129, 1000, 77, 700]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    chunks = P.plan_varlen(cu, 256, P.FLOPS)
    q, k, v, do = (x.cuda() for x in make_inputs(1, 6, cu[-1], 128, seed=501, packed=True, Hkv=2))
    o, lse = cca.forward(q, k, v, chunks, packed=True)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks, packed=True)
    torch.cuda.synchronize()
    grouped_check(q, k, v, do, o, lse, dq, dk, dv, cu, True, "gqa packed")
    o2, lse2 = cca.forward_streamed(q, k, v, chunks, packed=True)
    dq2, dk2, dv2, _, _ = cca.backward_streamed(q, k, v, o2, lse2, do, chunks, packed=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(lse2, lse)
    grouped_check(q, k, v, do, o2, lse2, dq2, dk2, dv2, cu, True, "gqa packed streamed")


def test_grouped_token_major_strides():
    """[B, L, H, D] storage for q/o/dout and [B, L, Hkv, D] for k/v (different
    token strides for the two groups of tensors) through the strided ABI."""
    B, L, H, Hkv, D = 1, 600, 4, 2, 128
    base = [x.cuda() for x in make_inputs(B, H, L, D, seed=502, Hkv=Hkv)]
    tm = [x.permute(0, 2, 1, 3).contiguous() for x in base]
    q, k, v, do = [x.permute(0, 2, 1, 3) for x in tm]
    chunks = P.plan(L, 2, P.FLOPS)
    o, lse = cca.forward(q, k, v, chunks)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    assert dk.stride() == k.stride()
    grouped_check(q, k, v, do, o, lse, dq, dk, dv, None, False, "gqa token-major")
    o2, lse2 = cca.forward(*base[:3], chunks)
    dq2, dk2, dv2 = cca.backward(*base[:3], o2, lse2, base[3], chunks)
    torch.cuda.synchronize()
    assert torch.equal(o.contiguous(), o2) and torch.equal(dk.contiguous(), dk2) and torch.equal(dv.contiguous(), dv2)


def test_gqa_128k_sampled():
    """The 128K grouped workload (32 query heads, 8 key/value heads): sampled
    query rows of every group, the last keys of two key/value heads summed
    over their query heads, and sum_j dV_j = sum over the group of sum_t dO_t."""
    w = WORKLOADS["gqa_128k"]
    q, k, v, do = (x.cuda() for x in workload_inputs(w))
    chunks = cca.attn_plan(w.L, w.N, w.mode)
    o, lse = cca.forward(q, k, v, chunks)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    G = w.H // w.Hkv
    rng = np.random.default_rng(31)
    go, gl, gq, ro, rl, rq = [], [], [], [], [], []
    for h in rng.choice(w.H, 8, replace=False):
        h = int(h)
        r = rng.integers(0, w.L, 256)
        qh, doh = head(q, 0, h, False), head(do, 0, h, False)
        kh, vh = head(k, 0, h // G, False), head(v, 0, h // G, False)
        o_ref, l_ref = A.forward_rows(qh, kh, vh, r, w.scale)
        ro.append(o_ref); rl.append(l_ref); rq.append(A.dq_rows(qh, kh, vh, doh, r, w.scale))
        go.append(head(o, 0, h, False)[r]); gl.append(lse_head(lse, 0, h)[r]); gq.append(head(dq, 0, h, False)[r])
    check_fwd(np.concatenate(go), np.concatenate(gl), np.concatenate(ro), np.concatenate(rl), "gqa 128k")
    check_grad(np.concatenate(gq), np.concatenate(rq), "gqa 128k dQ")
    keys = np.arange(w.L - 48, w.L)
    for hk in (0, 5):
        kh, vh = head(k, 0, hk, False), head(v, 0, hk, False)
        rdk = np.zeros((len(keys), w.D))
        rdv = np.zeros((len(keys), w.D))
        for h in range(hk * G, hk * G + G):
            a_, b_ = A.dkdv_keys(head(q, 0, h, False), kh, vh, head(do, 0, h, False), keys, w.scale)
            rdk += a_
            rdv += b_
        check_grad(head(dk, 0, hk, False)[keys], rdk, f"gqa 128k dK hk{hk}")
        check_grad(head(dv, 0, hk, False)[keys], rdv, f"gqa 128k dV hk{hk}")
        sdo = sum(head(do, 0, h, False).sum(axis=0) for h in range(hk * G, hk * G + G))
        sv = head(dv, 0, hk, False).sum(axis=0) - sdo
        norm = np.sqrt(sum((head(do, 0, h, False) ** 2).sum() for h in range(hk * G, hk * G + G)))
        assert np.linalg.norm(sv) / norm <= 5e-3


@pytest.mark.parametrize("D", [64, 128])
def test_grouped_p_part_plan(D):
    """Grouped key/value heads with a plan whose edge chunks are re-split into
    P key parts: the forward partials and their merge per query head, the
    backward's group sums."""
    L = 3000
    chunks = cca.attn_plan_multiplex(L, 6, 4)
    assert any(c[3] < 0 for c in chunks)
    q, k, v, do = (x.cuda() for x in make_inputs(2, 8, L, D, seed=520 + D, Hkv=2))
    o, lse = cca.forward(q, k, v, chunks)
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks)
    torch.cuda.synchronize()
    grouped_check(q, k, v, do, o, lse, dq, dk, dv, None, False, f"gqa multiplex D{D}")
