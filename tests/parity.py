"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare against the float64 oracle with the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import chunked_causal_attention_gb300 as cca
from oracle import attention as A

# Tolerances (GPU bf16 outputs vs float64 oracle)
O_MAX_ABS = 1e-2
O_REL_L2 = 5e-3
LSE_ABS = 1e-3
GRAD_REL_L2 = 1e-2


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def head(x: torch.Tensor, b: int, h: int, packed: bool) -> np.ndarray:
    """[T, D] float64 slice of one (batch, head) of a dense [B,H,L,D] or packed [T,H,D] tensor."""
    s = x[:, h] if packed else x[b, h]
    return s.detach().float().cpu().numpy().astype(np.float64)


def lse_head(lse: torch.Tensor, b: int, h: int) -> np.ndarray:
    return lse[b, h].detach().cpu().numpy().astype(np.float64)


def run_gpu(q, k, v, do, chunks, packed=False, scale=None, backward=True):
    """Forward (and backward) through the C ABI on the inputs' device."""
    o, lse = cca.forward(q, k, v, chunks, scale=scale, packed=packed)
    if not backward:
        torch.cuda.synchronize()
        return o, lse, None, None, None
    dq, dk, dv = cca.backward(q, k, v, o, lse, do, chunks, scale=scale, packed=packed)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def check_fwd(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    err = np.abs(o_gpu - o_ref).max() if o_ref.size else 0.0
    assert err <= O_MAX_ABS, f"{what} O max-abs {err}"
    r = rel_l2(o_gpu, o_ref)
    assert r <= O_REL_L2, f"{what} O rel-L2 {r}"
    le = np.abs(lse_gpu - lse_ref).max() if lse_ref.size else 0.0
    assert le <= LSE_ABS, f"{what} LSE abs {le}"
    print(f"[parity] {what}: O max-abs {err:.3e} rel-L2 {r:.3e}, LSE max-abs {le:.3e}")
    return err, r, le


def check_grad(g, ref, what=""):
    r = rel_l2(g, ref)
    assert r <= GRAD_REL_L2, f"{what} rel-L2 {r}"
    print(f"[parity] {what}: rel-L2 {r:.3e}")
    return r


def docs_of(chunks):
    """Document boundaries (cu_seqlens) implied by a partitioning chunk table."""
    cu = [0]
    for i, (qb, qe, cb, _) in enumerate(chunks):
        if i > 0 and cb != chunks[i - 1][2]:
            cu.append(qb)
    cu.append(chunks[-1][1])
    return cu


def default_scale(D):
    return 1.0 / math.sqrt(D)


# ------------------------------------------------ full-size workloads (sampled)

def plan_of(w):
    if w.packed:
        return cca.attn_plan_varlen(w.cu_seqlens(), w.max_chunk_tokens, w.mode)
    return cca.attn_plan(w.L, w.N, w.mode)


def sampled_rows_check(w, q, k, v, do, o, lse, dq, n_rows, seed, what, backward=True):
    rng = np.random.default_rng(seed)
    heads = rng.integers(0, w.H, n_rows)
    rows = rng.integers(0, w.L, n_rows)
    cu = w.cu_seqlens()
    go, gl, gq, ro, rl, rq = [], [], [], [], [], []
    for h in np.unique(heads):
        r = rows[heads == h]
        qh, kh, vh, doh = (head(x, 0, int(h), w.packed) for x in (q, k, v, do))
        o_ref, l_ref = A.forward_rows(qh, kh, vh, r, w.scale, cu)
        go.append(head(o, 0, int(h), w.packed)[r]); gl.append(lse_head(lse, 0, int(h))[r])
        ro.append(o_ref); rl.append(l_ref)
        if backward:
            rq.append(A.dq_rows(qh, kh, vh, doh, r, w.scale, cu))
            gq.append(head(dq, 0, int(h), w.packed)[r])
    check_fwd(np.concatenate(go), np.concatenate(gl), np.concatenate(ro), np.concatenate(rl), what)
    if backward:
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
