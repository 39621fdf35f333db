"""Writes tests/golden/plans.json: the oracle's chunk plans for the five
workloads (tiny, 7b_32k, 7b_128k, packed_256k, 13b_1m). Expected values come
from oracle/ only; the packed document lengths come from the seeded input
generator. Run from the repository root: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import plan as P  # noqa: E402
from chunked_causal_attention_gb300.workloads import WORKLOADS  # noqa: E402


def main():
    out = {}
    for name, w in WORKLOADS.items():
        if w.packed:
            cu = w.cu_seqlens()
            out[name] = {"cu_seqlens": cu, "max_chunk_tokens": w.max_chunk_tokens, "mode": w.mode,
                         "chunks": [list(c) for c in P.plan_varlen(cu, w.max_chunk_tokens, w.mode)]}
        else:
            out[name] = {"L": w.L, "N": w.N, "mode": w.mode,
                         "chunks": [list(c) for c in P.plan(w.L, w.N, w.mode)]}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "plans.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
