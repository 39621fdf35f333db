"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare against the float64 oracle with the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import chunked_causal_attention_gb300 as cca

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
