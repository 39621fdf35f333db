"""Cost model of a chunk on this GPU (InfiniPipe Eq. (1)) and the chunk-streamed
execution of the plans built on it.

    python -m chunked_causal_attention_gb300.costfit fit      # time calls, fit, write cost_gb300.json
    python -m chunked_causal_attention_gb300.costfit report   # run plans of the packed 256K documents

Eq. (1) on one GPU (N = d_p = 1, no all-to-all): a call holding slices s with
contexts C costs beta1 + alpha1 * sum((C+s)^2 - C^2) + alpha2 * sum(s). ``fit``
times one forward call (attn_fwd) plus one backward call (attn_bwd_chunk) for
split slices of a long sequence and for batches of short sequences, at the
7B attention shape (32 heads of 128), and fits the three constants by
non-negative least squares on relative error (each point weighted by 1/time,
since a plan compares calls of very different sizes). ``report`` plans the packed 256K documents with
InfiniPipe Algorithm 1 (attn_plan_infinipipe, fitted costs) and with the
per-document FLOPs chunks of attn_plan_varlen, runs each plan one call at a
time (forward in call order, backward in reverse), and prints per-call
times, their balance, the model's error and the throughput as one JSON line.
"""
from __future__ import annotations

import json
import os
import statistics
import sys
from typing import List, Sequence, Tuple

COST_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cost_gb300.json")

H, D = 32, 128
T_BUF = 262144


def load_cost():
    """(alpha1, alpha2, beta1) in milliseconds, fitted on a GB300 by ``fit``."""
    with open(COST_PATH) as f:
        c = json.load(f)
    return c["alpha1_ms"], c["alpha2_ms"], c["beta1_ms"]


def model_terms(call: Sequence[Tuple[int, int, int, int]]):
    """(sum of (C+s)^2 - C^2, sum of s) of a call's chunks."""
    quad = lin = 0
    for qb, qe, cb, _ in call:
        C, s = qb - cb, qe - qb
        quad += (C + s) * (C + s) - C * C
        lin += s
    return quad, lin


class Runner:
    """Packed [T, H, D] inputs on the GPU and one workspace per pass large enough for any call."""

    def __init__(self, calls_list: Sequence[Sequence], seed: int = 4321):
        import torch
        import chunked_causal_attention_gb300 as cca
        from chunked_causal_attention_gb300.workloads import make_inputs
        self.torch, self.cca = torch, cca
        self.q, self.k, self.v, self.do = (x.cuda() for x in make_inputs(1, H, T_BUF, D, seed=seed, packed=True))
        self.shape = cca.shape_of(self.q, packed=True)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((1, H, T_BUF), dtype=torch.float32, device="cuda")
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.dk_acc = torch.zeros(self.k.shape, dtype=torch.float32, device="cuda")
        self.dv_acc = torch.zeros(self.v.shape, dtype=torch.float32, device="cuda")
        all_calls = [c for calls in calls_list for c in calls]
        self.ws_f = cca.workspace(self.shape, all_calls, cca.PASS_FWD, per_chunk=True)
        self.ws_b = cca.workspace(self.shape, all_calls, cca.PASS_BWD_CHUNK, per_chunk=True)
        self.stream = torch.cuda.current_stream()

    def fwd(self, call):
        self.cca.attn_fwd(self.q, self.k, self.v, call, self.shape, self.o, self.lse, self.ws_f, self.stream)

    def bwd(self, call):
        self.cca.attn_bwd_chunk(self.q, self.k, self.v, self.o, self.lse, self.do, call, self.shape, self.dq, self.dk,
                                self.dv, self.dk_acc, self.dv_acc, self.ws_b, self.stream)

    def time_call(self, call, reps: int = 3) -> Tuple[float, float]:
        """Median forward and backward milliseconds of one call (events on the stream)."""
        torch = self.torch
        self.fwd(call)
        self.bwd(call)
        fw, bw = [], []
        for _ in range(reps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(self.stream)
            self.fwd(call)
            e[1].record(self.stream)
            self.bwd(call)
            e[2].record(self.stream)
            torch.cuda.synchronize()
            fw.append(e[0].elapsed_time(e[1]))
            bw.append(e[1].elapsed_time(e[2]))
        self.check()
        return statistics.median(fw), statistics.median(bw)

    def run_plan(self, calls) -> Tuple[List[float], List[float]]:
        """One pass of a plan: forward per call in order, backward per call in reverse."""
        torch = self.torch
        self.dk_acc.zero_()
        self.dv_acc.zero_()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(2 * len(calls))]
        for i, c in enumerate(calls):
            ev[i][0].record(self.stream)
            self.fwd(c)
            ev[i][1].record(self.stream)
        for j, c in enumerate(reversed(calls)):
            i = len(calls) + j
            ev[i][0].record(self.stream)
            self.bwd(c)
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        self.check()
        f = [ev[i][0].elapsed_time(ev[i][1]) for i in range(len(calls))]
        b = [ev[len(calls) + j][0].elapsed_time(ev[len(calls) + j][1]) for j in range(len(calls))][::-1]
        return f, b

    def check(self):
        st = self.cca.attn_status(self.ws_f) or self.cca.attn_status(self.ws_b)
        if st:
            raise RuntimeError(f"device status: {self.cca.strerror(st)}")


def fit_calls():
    """Calls of the fitting grid: slices of one 128K sequence at [0, 131072)
    and batches of short sequences in [131072, 262144)."""
    calls = []
    for C in (0, 16384, 49152, 98304):
        for s in (1024, 4096, 8192, 16384, 32768):
            if C + s <= 131072:
                calls.append([(C, C + s, 0, 0)])
    base = 131072
    for n, s in ((2, 16384), (8, 8192), (4, 2048), (16, 1024), (64, 512), (128, 256), (32, 4096)):
        calls.append([(base + j * s, base + (j + 1) * s, base + j * s, 0) for j in range(n)])
    return calls


def fit_constants(rows, ms):
    """(alpha1, alpha2, beta1) >= 0 minimising the squared relative error of
    alpha1 quad + alpha2 tokens + beta1 against the measured times ``ms``
    (rows: [quad, tokens, 1] per call), and the relative errors per call."""
    import numpy as np
    from scipy.optimize import nnls
    A = np.array(rows, dtype=np.float64)
    y = np.array(ms, dtype=np.float64)
    W = A / y[:, None]                         # relative residuals: (pred - y) / y
    scale = W.max(axis=0)
    x, _ = nnls(W / scale, np.ones_like(y))
    a1, a2, b1 = (x / scale).tolist()
    pred = A @ np.array([a1, a2, b1])
    return a1, a2, b1, np.abs(pred - y) / y


def fit():
    import numpy as np
    calls = fit_calls()
    r = Runner([calls])
    rows, ms, fw_ms, bw_ms = [], [], [], []
    for c in calls:
        f, b = r.time_call(c)
        quad, lin = model_terms(c)
        rows.append([quad, lin, 1.0])
        ms.append(f + b)
        fw_ms.append(f)
        bw_ms.append(b)
    a1, a2, b1, rel = fit_constants(rows, ms)
    out = {"alpha1_ms": a1, "alpha2_ms": a2, "beta1_ms": b1, "unit": "ms per call (forward + backward)",
           "shape": f"H{H} D{D} bf16", "calls": len(calls), "max_rel_err": float(rel.max()),
           "median_rel_err": float(np.median(rel)),
           "points": [{"chunks": len(c), "quad": int(q), "tokens": int(l), "fwd_ms": f, "bwd_ms": b}
                      for c, (q, l, _), f, b in zip(calls, rows, fw_ms, bw_ms)],
           "command": "python -m chunked_causal_attention_gb300.costfit fit"}
    with open(COST_PATH, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps({k: out[k] for k in ("alpha1_ms", "alpha2_ms", "beta1_ms", "max_rel_err", "median_rel_err")}))


def report(settings=((4, 65536), (8, 65536), (16, 32768))):
    import chunked_causal_attention_gb300 as cca
    from chunked_causal_attention_gb300.workloads import WORKLOADS
    a1, a2, b1 = load_cost()
    cu = WORKLOADS["packed_256k"].cu_seqlens()
    lengths = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    pairs = sum(L * (L + 1) // 2 for L in lengths) * H
    flops = 14 * D * pairs
    plans = {f"infinipipe_K{K}_cap{cap}": cca.attn_plan_infinipipe(lengths, K, cap, a1, a2, b1) for K, cap in settings}
    plans["flops_per_document_16k"] = [[c] for c in cca.attn_plan_varlen(cu, 16384, cca.PLAN_FLOPS)]
    r = Runner(list(plans.values()))
    res = {}
    for name, calls in plans.items():
        r.run_plan(calls)                                   # warm-up pass
        f, b = r.run_plan(calls)
        t = [x + y for x, y in zip(f, b)]
        pred = [b1 + a1 * model_terms(c)[0] + a2 * model_terms(c)[1] for c in calls]
        res[name] = {"calls": len(calls), "total_ms": sum(t), "fwd_ms": sum(f), "bwd_ms": sum(b),
                     "tflops": flops / (sum(t) * 1e-3) / 1e12,
                     "call_ms_max": max(t), "call_ms_mean": statistics.mean(t),
                     "imbalance_max_over_mean": max(t) / statistics.mean(t),
                     "model_max_rel_err": max(abs(p - m) / m for p, m in zip(pred, t)),
                     "model_median_rel_err": statistics.median(abs(p - m) / m for p, m in zip(pred, t)),
                     "per_call": [{"chunks": len(c), "tokens": model_terms(c)[1], "ms": m, "pred_ms": p}
                                  for c, m, p in zip(calls, t, pred)]}
    print(json.dumps({"workload": "packed_256k", "cost_ms": [a1, a2, b1], "plans": res}))


if __name__ == "__main__":
    {"fit": fit, "report": report}[sys.argv[1] if len(sys.argv) > 1 else "report"]()
