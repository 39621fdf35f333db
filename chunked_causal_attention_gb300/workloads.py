"""Seeded synthetic inputs shaped like the long-sequence training workloads.

This module holds input generation only: shapes, seeds, random draws and the
document-length mix. It contains none of the attention arithmetic, so both the
CUDA path and the float64 oracle can be fed from it.

Workloads (the pages train GPT/LLaMA 7B and 13B models on 128K to 4M tokens;
no dataset is available here, so all tensors are i.i.d. N(0, 1) cast to bf16):

* ``tiny``       B=1 H=2  D=64  L=1024, UNIFORM plan of 4 chunks of 256.
* ``7b_32k``     B=1 H=32 D=128 L=32768, FLOPS plan N=8.
* ``7b_128k``    B=1 H=32 D=128 L=131072, FLOPS plan N=16 with the first and
                 last chunk re-split (the throughput workload).
* ``packed_256k`` 262144 packed tokens, H=32 D=128, document lengths drawn
                 lognormal(mu=ln 4096, sigma=1.2) clipped to [128, 131072], at
                 least one document longer than 64K (InfiniPipe's skewed
                 real-world length distribution, Fig. 1(b)); documents longer
                 than 16K are cut into FLOPs-balanced chunks.
* ``13b_1m``     B=1 H=40 D=128 L=1048576, FLOPS plan N=64.
* ``gqa_128k``   B=1 H=32 with 8 key/value heads (grouped-query attention,
                 4 query heads per key/value head), D=128 L=131072, the same
                 plan as 7b_128k.
* ``d256_32k``   B=1 H=16 D=256 L=32768 (the 7B hidden size of 4096 as 16
                 heads of 256 dims), FLOPS plan N=8 with the edges re-split.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

PLAN_UNIFORM = 0
PLAN_FLOPS = 1
PLAN_FLOPS_RESPLIT_EDGES = 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    L: int                     # tokens per batch row (dense) or total packed tokens
    N: int = 1                 # chunks (dense plans)
    mode: int = PLAN_FLOPS
    seed: int = 1234
    packed: bool = False
    max_chunk_tokens: int = 16384
    doc_lens: Optional[List[int]] = field(default=None, compare=False)
    Hkv: Optional[int] = None  # key/value heads (grouped-query attention); None: H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def cu_seqlens(self) -> Optional[List[int]]:
        if not self.packed:
            return None
        cu = [0]
        for n in self.doc_lens:
            cu.append(cu[-1] + n)
        return cu


def skewed_doc_lengths(total: int = 262144, seed: int = 1237, mu: float = math.log(4096.0),
                       sigma: float = 1.2, lo: int = 128, hi: int = 131072,
                       first_min: int = 65536) -> List[int]:
    """Document lengths summing to ``total``: the first draw is rejection-sampled
    above ``first_min`` (so one document is longer than 64K), the rest are
    round(lognormal) clipped to [lo, hi]; the last document is truncated so the
    lengths sum to ``total`` and a remainder under ``lo`` joins the previous one."""
    rng = np.random.Generator(np.random.PCG64(seed))
    while True:
        x = rng.lognormal(mu, sigma)
        if x > first_min:
            break
    lens = [int(min(round(x), hi))]
    while sum(lens) < total:
        lens.append(int(min(max(round(rng.lognormal(mu, sigma)), lo), hi)))
    excess = sum(lens) - total
    lens[-1] -= excess
    if lens[-1] < lo and len(lens) > 1:
        tail = lens.pop()
        lens[-1] += tail
    assert sum(lens) == total
    return lens


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 64, 1024, N=4, mode=PLAN_UNIFORM, seed=1234),
    "7b_32k": Workload("7b_32k", 1, 32, 128, 32768, N=8, mode=PLAN_FLOPS, seed=1235),
    "7b_128k": Workload("7b_128k", 1, 32, 128, 131072, N=16, mode=PLAN_FLOPS_RESPLIT_EDGES, seed=1236),
    "packed_256k": Workload("packed_256k", 1, 32, 128, 262144, mode=PLAN_FLOPS, seed=1237, packed=True,
                            max_chunk_tokens=16384, doc_lens=skewed_doc_lengths()),
    "13b_1m": Workload("13b_1m", 1, 40, 128, 1048576, N=64, mode=PLAN_FLOPS, seed=1238),
    "gqa_128k": Workload("gqa_128k", 1, 32, 128, 131072, N=16, mode=PLAN_FLOPS_RESPLIT_EDGES, seed=1239, Hkv=8),
    "d256_32k": Workload("d256_32k", 1, 16, 256, 32768, N=8, mode=PLAN_FLOPS_RESPLIT_EDGES, seed=1240),
}


def randn_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """i.i.d. N(0,1) drawn in float32 from a seeded generator, rounded to bf16 (RNE)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_inputs(B: int, H: int, L: int, D: int, seed: int, device="cpu", packed: bool = False,
                Hkv: Optional[int] = None):
    """(q, k, v, do) bf16 tensors; dense layout [B, H, L, D], packed [L, H, D];
    k and v have Hkv heads when given (grouped key/value heads).

    Each tensor has its own stream: seeds seed*4 + {0,1,2,3}."""
    hk = H if Hkv is None else Hkv
    shapes = [(L, h, D) if packed else (B, h, L, D) for h in (H, hk, hk, H)]
    return tuple(randn_bf16(shapes[i], seed * 4 + i, device) for i in range(4))


def workload_inputs(w: Workload, device="cpu"):
    return make_inputs(w.B, w.H, w.L, w.D, w.seed, device=device, packed=w.packed, Hkv=w.Hkv)
