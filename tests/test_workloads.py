"""The synthetic input recipe (no GPU): workload shapes and plans, seeds,
bf16 rounding of the N(0, 1) draws, and the skewed packed document lengths."""
import math
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from chunked_causal_attention_gb300 import workloads as W  # noqa: E402


def test_workload_shapes_and_seeds():
    """Shapes and plans of the five configurations, seed = 1234 + index, plus the grouped-head variant."""
    want = {
        "tiny": (1, 2, 64, 1024, 4, W.PLAN_UNIFORM, 1234),
        "7b_32k": (1, 32, 128, 32768, 8, W.PLAN_FLOPS, 1235),
        "7b_128k": (1, 32, 128, 131072, 16, W.PLAN_FLOPS_RESPLIT_EDGES, 1236),
        "13b_1m": (1, 40, 128, 1 << 20, 64, W.PLAN_FLOPS, 1238),
    }
    for name, (B, H, D, L, N, mode, seed) in want.items():
        w = W.WORKLOADS[name]
        assert (w.B, w.H, w.D, w.L, w.N, w.mode, w.seed) == (B, H, D, L, N, mode, seed), name
        assert w.scale == 1.0 / math.sqrt(D) and not w.packed and w.cu_seqlens() is None
    p = W.WORKLOADS["packed_256k"]
    assert (p.B, p.H, p.D, p.L, p.seed, p.max_chunk_tokens, p.packed) == (1, 32, 128, 262144, 1237, 16384, True)
    cu = p.cu_seqlens()
    assert cu[0] == 0 and cu[-1] == 262144 and len(cu) == len(p.doc_lens) + 1
    g = W.WORKLOADS["gqa_128k"]
    assert (g.H, g.Hkv, g.L, g.N, g.mode) == (32, 8, 131072, 16, W.PLAN_FLOPS_RESPLIT_EDGES)


def test_skewed_document_lengths():
    lens = W.skewed_doc_lengths()
    assert lens == W.skewed_doc_lengths()                 # seeded
    assert sum(lens) == 262144
    assert lens[0] > 65536                                 # the rejection-sampled first document
    assert all(128 <= n <= 131072 for n in lens)
    assert lens == W.WORKLOADS["packed_256k"].doc_lens
    # another seed gives another mix with the same guarantees
    other = W.skewed_doc_lengths(seed=99)
    assert other != lens and sum(other) == 262144 and other[0] > 65536 and min(other) >= 128


def test_skewed_lengths_follow_the_lognormal():
    """Over many documents the log-lengths of the draws after the first have the
    recipe's median (ln 4096) and spread (sigma 1.2) up to clipping."""
    lens = W.skewed_doc_lengths(total=40_000_000, seed=2)[1:-1]
    x = np.log(np.array(lens, dtype=np.float64))
    se_median = 1.2533 * 1.2 / math.sqrt(len(x))          # standard error of a normal sample's median
    assert abs(np.median(x) - math.log(4096.0)) < 4 * se_median
    assert 1.1 < np.std(x) < 1.25                          # clipping to [128, 131072] trims the tails a little


def test_bf16_draws():
    a = W.randn_bf16((4096,), seed=3)
    assert a.dtype == torch.bfloat16
    assert torch.equal(a, W.randn_bf16((4096,), seed=3)) and not torch.equal(a, W.randn_bf16((4096,), seed=4))
    # the bf16 values are the float32 draws rounded to nearest even
    g = torch.Generator()
    g.manual_seed(3)
    f = torch.randn(4096, generator=g, dtype=torch.float32)
    assert torch.equal(a, f.to(torch.bfloat16))
    af = a.float()
    assert abs(af.mean().item()) < 0.06 and abs(af.std().item() - 1.0) < 0.05


def test_make_inputs_layouts_and_streams():
    q, k, v, do = W.make_inputs(2, 4, 300, 64, seed=10)
    assert [tuple(x.shape) for x in (q, k, v, do)] == [(2, 4, 300, 64)] * 4
    assert not torch.equal(q, k) and not torch.equal(v, do)
    assert torch.equal(q, W.randn_bf16((2, 4, 300, 64), 40))   # tensor i draws from seed*4 + i
    assert torch.equal(do, W.randn_bf16((2, 4, 300, 64), 43))
    q, k, v, do = W.make_inputs(1, 6, 500, 128, seed=11, packed=True, Hkv=2)
    assert tuple(q.shape) == (500, 6, 128) and tuple(k.shape) == (500, 2, 128) and tuple(do.shape) == (500, 6, 128)
