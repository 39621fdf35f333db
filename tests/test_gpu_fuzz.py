"""Seeded random cases across the cross product of the options, each checked
against the float64 oracle on every row and key: batch rows, heads and
grouped key/value heads, ragged lengths, head dims from 8 to 256, dense rows
or packed documents, the plan modes (uniform, FLOPs, edge re-split, P-part
multiplex), and a single call or chunk-streamed calls (forward in chunk
order, backward in reverse order with fp32 dK/dV accumulators). The cases are
drawn from a fixed seed, so a failure names a case that can be rerun."""
import numpy as np
import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300.workloads import make_inputs
from oracle import attention as A
from oracle import plan as P

from parity import check_fwd, check_grad, default_scale, head, lse_head

pytestmark = pytest.mark.gpu

N_CASES = 24
DIMS = [8, 16, 40, 64, 72, 96, 120, 128, 136, 160, 192, 248, 256]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(cca._lib.LIB_PATH):
        from chunked_causal_attention_gb300 import build
        build.build()


def dense_plan(rng, L):
    """A plan of L tokens in one of the four modes; falls back to fewer chunks
    where the drawn count is too large for L."""
    kind = int(rng.integers(0, 4))
    N = int(rng.integers(1, 7))
    while N >= 1:
        try:
            if kind == 3:
                return P.plan_multiplex(L, N, int(rng.integers(2, 5))), f"multiplex N{N}"
            mode = [P.UNIFORM, P.FLOPS, P.FLOPS_RESPLIT_EDGES][kind]
            return P.plan(L, N, mode), f"mode{mode} N{N}"
        except P.PlanError:
            N -= 1
            kind = min(kind, 2)
    return P.plan(L, 1, P.FLOPS), "N1"


def draw_case(seed):
    rng = np.random.default_rng(seed)
    D = int(rng.choice(DIMS))
    Hkv = int(rng.integers(1, 4))
    G = int(rng.choice([1, 1, 2, 3]))
    packed = bool(rng.integers(0, 2))
    L_max = 2000 if D <= 128 else 1200
    if packed:
        lens = [int(x) for x in rng.integers(1, L_max // 2, int(rng.integers(1, 6)))]
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        mode = int(rng.choice([P.UNIFORM, P.FLOPS, P.FLOPS_RESPLIT_EDGES]))
        mct = int(rng.choice([128, 256, 700]))
        while True:
            try:
                chunks = P.plan_varlen(cu, mct, mode)
                break
            except P.PlanError:                      # too many chunks for some document
                mct *= 2
        what = f"packed {lens} mode{mode} cap{mct}"
        B, L = 1, cu[-1]
    else:
        B = int(rng.integers(1, 3))
        L = int(rng.integers(1, L_max))
        chunks, what = dense_plan(rng, L)
        cu = None
    streamed = bool(rng.integers(0, 2))
    return dict(B=B, H=Hkv * G, Hkv=Hkv, L=L, D=D, packed=packed, cu=cu, chunks=chunks, streamed=streamed,
                what=f"seed {seed}: B{B} H{Hkv * G}/{Hkv} L{L} D{D} {what}{' streamed' if streamed else ''}")


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed):
    c = draw_case(7000 + seed)
    what = c["what"]
    q, k, v, do = (x.cuda() for x in make_inputs(c["B"], c["H"], c["L"], c["D"], seed=7100 + seed,
                                                 packed=c["packed"], Hkv=c["Hkv"]))
    chunks, packed = c["chunks"], c["packed"]
    if c["streamed"]:
        o, lse = cca.forward_streamed(q, k, v, chunks, packed=packed)
        dq, dk, dv, dk_acc, dv_acc = cca.backward_streamed(q, k, v, o, lse, do, chunks, packed=packed)
        torch.cuda.synchronize()
        assert torch.equal(dk, dk_acc.to(torch.bfloat16)) and torch.equal(dv, dv_acc.to(torch.bfloat16)), what
        o1, lse1 = cca.forward(q, k, v, chunks, packed=packed)
        torch.cuda.synchronize()
        assert torch.equal(o, o1) and torch.equal(lse, lse1), what
    else:
        o, lse = cca.forward(q, k, v, chunks, packed=packed)
        dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks, packed=packed)
        torch.cuda.synchronize()
    G = c["H"] // c["Hkv"]
    sc = default_scale(c["D"])
    for b in range(c["B"]):
        for hk in range(c["Hkv"]):
            hs = range(hk * G, hk * G + G)
            rdqs, rdk, rdv, ros, rls = A.grouped_backward([head(q, b, h, packed) for h in hs], head(k, b, hk, packed),
                                                          head(v, b, hk, packed), [head(do, b, h, packed) for h in hs],
                                                          sc, c["cu"])
            for g, h in enumerate(hs):
                check_fwd(head(o, b, h, packed), lse_head(lse, b, h), ros[g], rls[g], f"{what} b{b}h{h}")
                check_grad(head(dq, b, h, packed), rdqs[g], f"{what} dQ b{b}h{h}")
            check_grad(head(dk, b, hk, packed), rdk, f"{what} dK b{b}hk{hk}")
            check_grad(head(dv, b, hk, packed), rdv, f"{what} dV b{b}hk{hk}")
