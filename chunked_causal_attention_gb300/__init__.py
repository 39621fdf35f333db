"""Chunked causal self-attention for GB300 (sm_103a).

The compute lives in libattn.so (C ABI in include/attn.h, CUDA kernels in
csrc/); this package is its thin binding. PyTorch provides device memory and
streams only. ``forward`` / ``backward`` allocate outputs and the workspace
with torch and call the library; the ``attn_*`` functions mirror the C entry
points one to one.
"""
from __future__ import annotations

from typing import Optional, Sequence

from ._lib import (AttnError, EXPORTS, PASS_BWD, PASS_BWD_CHUNK, PASS_FWD, PLAN_FLOPS, PLAN_FLOPS_RESPLIT_EDGES,
                   PLAN_UNIFORM, attn_bwd, attn_bwd_chunk, attn_bwd_dq, attn_bwd_prep, attn_bwd_tiles, attn_fwd,
                   attn_fwd_merge, attn_fwd_noalloc, attn_fwd_tiles, attn_noalloc_status, attn_plan,
                   attn_plan_infinipipe, attn_plan_multiplex, attn_plan_varlen, attn_shape, attn_status,
                   attn_workspace_size, lib, make_shape, shape_of, strerror, version,
                   kernel_launches)

__all__ = ["AttnError", "EXPORTS", "PLAN_UNIFORM", "PLAN_FLOPS", "PLAN_FLOPS_RESPLIT_EDGES", "attn_plan",
           "attn_plan_varlen", "attn_plan_infinipipe", "attn_plan_multiplex", "attn_workspace_size", "attn_fwd", "attn_fwd_tiles", "attn_fwd_merge", "attn_bwd",
           "attn_bwd_prep", "attn_bwd_tiles", "attn_bwd_dq", "attn_bwd_chunk", "attn_fwd_noalloc",
           "attn_noalloc_status", "attn_status", "attn_shape",
           "make_shape", "shape_of", "workspace", "forward", "backward", "forward_streamed", "backward_streamed",
           "PASS_FWD", "PASS_BWD", "PASS_BWD_CHUNK", "plan_infinipipe", "lib", "strerror", "version",
           "kernel_launches"]


def workspace(shape: attn_shape, chunks: Sequence, pass_: int, device="cuda", per_chunk: bool = False):
    """A uint8 device buffer of the size the library asks for (pass 0 forward,
    1 backward, 2 chunk-streamed backward), with its 256-byte status header
    zeroed. per_chunk: ``chunks`` is a list of calls (each a chunk or a list
    of chunks) and the buffer fits any one of them."""
    import torch
    if per_chunk:
        calls = [c if isinstance(c[0], (list, tuple)) else [c] for c in chunks]
        n = max(attn_workspace_size(shape, c, pass_) for c in calls)
    else:
        n = attn_workspace_size(shape, chunks, pass_)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def _like(x):
    """An uninitialised tensor with x's sizes and strides (so that one attn_shape
    describes both), also when x is a view with gaps, such as the first D dims
    of a wider buffer."""
    import torch
    return torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)


def forward(q, k, v, chunks: Sequence, scale: Optional[float] = None, packed: bool = False, ws=None, stream=None):
    """(o, lse) of chunked causal attention; q, k, v bf16 [B, H, L, D] (or packed [T, H, D])."""
    import torch
    shape = shape_of(q, scale, packed, k)
    o = _like(q)
    lse = torch.empty((shape.B, shape.H, shape.T), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, chunks, 0, q.device)
    attn_fwd(q, k, v, chunks, shape, o, lse, ws, stream)
    return o, lse


def backward(q, k, v, o, lse, dout, chunks: Sequence, scale: Optional[float] = None, packed: bool = False,
             ws=None, stream=None):
    """(dq, dk, dv) for upstream gradient dout, given the forward's o and lse."""
    import torch
    shape = shape_of(q, scale, packed, k)
    dq, dk, dv = _like(q), _like(k), _like(v)
    if ws is None:
        ws = workspace(shape, chunks, 1, q.device)
    attn_bwd(q, k, v, o, lse, dout, chunks, shape, dq, dk, dv, ws, stream)
    return dq, dk, dv


def forward_streamed(q, k, v, chunks: Sequence, scale: Optional[float] = None, packed: bool = False, stream=None):
    """The forward one call at a time, in order: each entry of ``chunks`` is a
    chunk or a list of chunks (one call, e.g. an InfiniPipe batched or hybrid
    chunk); each call computes its rows against the keys before them, which
    are resident in k, v."""
    import torch
    shape = shape_of(q, scale, packed, k)
    o = _like(q)
    lse = torch.empty((shape.B, shape.H, shape.T), dtype=torch.float32, device=q.device)
    calls = [c if isinstance(c[0], (list, tuple)) else [c] for c in chunks]
    ws = workspace(shape, calls, PASS_FWD, q.device, per_chunk=True)
    for c in calls:
        attn_fwd(q, k, v, c, shape, o, lse, ws, stream)
    return o, lse


def backward_streamed(q, k, v, o, lse, dout, chunks: Sequence, scale: Optional[float] = None, packed: bool = False,
                      stream=None):
    """The backward one call at a time, in reverse order (entries of
    ``chunks`` as forward_streamed), with fp32 dK/dV accumulators shared by
    the calls (attn_bwd_chunk). Returns (dq, dk, dv, dk_acc, dv_acc)."""
    import torch
    shape = shape_of(q, scale, packed, k)
    dq, dk, dv = _like(q), _like(k), _like(v)
    # fp32 accumulators at the same element offsets as k and v
    dk_acc = torch.empty_strided(k.shape, k.stride(), dtype=torch.float32, device=k.device).zero_()
    dv_acc = torch.empty_strided(v.shape, v.stride(), dtype=torch.float32, device=v.device).zero_()
    calls = [c if isinstance(c[0], (list, tuple)) else [c] for c in chunks]
    ws = workspace(shape, calls, PASS_BWD_CHUNK, q.device, per_chunk=True)
    for c in reversed(calls):
        attn_bwd_chunk(q, k, v, o, lse, dout, c, shape, dq, dk, dv, dk_acc, dv_acc, ws, stream)
    return dq, dk, dv, dk_acc, dv_acc


def plan_infinipipe(seq_lens: Sequence[int], K: int, token_cap: int, cost=None):
    """InfiniPipe Algorithm 1 (attn_plan_infinipipe) with the Eq. (1) costs
    fitted on a GB300 (cost_gb300.json, from ``python -m
    chunked_causal_attention_gb300.costfit fit``) unless ``cost`` =
    (alpha1, alpha2, beta1) is given. Returns a list of calls for
    forward_streamed / backward_streamed (packed layout of seq_lens)."""
    if cost is None:
        from .costfit import load_cost
        cost = load_cost()
    return attn_plan_infinipipe(seq_lens, K, token_cap, *cost)
