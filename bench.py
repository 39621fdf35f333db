"""Benchmark: causal attention fwd+bwd TFLOP/s (bf16) at L=128K on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 7b_128k] [--impl ours|reference]

A step is one pass of the whole hot path over the workload: forward tile
kernel, LSE merge of the re-split edge chunks, backward preprocess, backward
key-tile kernel, dQ finalize. `value` counts algorithmic FLOPs only: 14*D per
visible (query, key) pair (2 forward GEMMs, 5 backward GEMMs). Inputs (1 GiB
per tensor) are far larger than the 129 MB L2, so no flush is needed between
steps. Under torchrun every rank runs its own replica of the workload (the
heads are independent; no data-path collective) and rank 0 prints one JSON
line with the whole-job throughput (weak scaling).

--impl reference times the float64 CPU oracle on the same workload, metric
and unit, each step a bounded sample (a causal prefix of one head).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
METRIC = "causal attn fwd+bwd TFLOP/s (bf16) at L=128K, % of GB300 dense BF16 peak"
CPU_SAMPLE_TOKENS = 40960     # causal prefix of one head timed on the host cores


TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic_7b_128k.json")
KERNEL_SOURCES = ["bwd_tc.cu", "device_common.cuh", "tc_common.cuh"]
# the parts of attn_api.cpp that set the backward's work list, order and launch
API_SECTIONS = [("// --------------------------------------------------------------- backward layout", "\n}  // namespace"),
                ("constexpr int32_t kGroupBwd", "\n"),
                ("int bwd_launch(", "\nint bwd_common(")]


def kernel_source_hash():
    """SHA-256 over what sets the backward tile kernel's memory traffic: its
    source and device headers, and the backward work-list layout, head-group
    constant and launch code of attn_api.cpp."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_causal_attention_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(csrc, "attn_api.cpp")) as fh:
        api = fh.read()
    for start, end in API_SECTIONS:
        i = api.index(start)
        h.update(api[i:api.index(end, i + len(start))].encode())
    return h.hexdigest()


def measured_traffic(workload):
    """DRAM bytes per launch of the backward tile kernel from the committed ncu
    capture, or None when the kernel sources changed since it was taken."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("workload") != workload or t.get("source_sha256") != kernel_source_hash():
        return None
    return t["dram_bytes_read"] + t["dram_bytes_write"]


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def causal_pairs_total(w, chunks):
    from chunked_causal_attention_gb300.workloads import Workload  # noqa: F401
    if w.packed:
        lens = w.doc_lens
        per = sum(n * (n + 1) // 2 for n in lens)
    else:
        per = w.L * (w.L + 1) // 2
    return per * w.B * w.H


# ----------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, path=None):
        self.proc = None
        self.path = path
        self.lines = []
        self.bus = None
        try:
            import torch
            p = torch.cuda.get_device_properties(device_index)
            self.bus = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            self.bus = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.bus:
            cmd += ["-i", self.bus]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]
        if self.path:
            with open(self.path, "w") as f:
                f.write(self.QUERY + "\n" + "\n".join(self.lines) + "\n")
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- oracle arm
def time_oracle_sample(w, tokens, seed):
    """Oracle fwd+bwd (float64, host cores) on a causal prefix of one head."""
    import numpy as np
    from chunked_causal_attention_gb300.workloads import make_inputs
    from oracle import attention as A
    D = w.D
    q, k, v, do = (x[0, 0].float().numpy() for x in make_inputs(1, 1, tokens, D, seed=seed))
    t0 = time.perf_counter()
    A.backward(q, k, v, do, w.scale, None, row_block=1024)
    dt = time.perf_counter() - t0
    pairs = tokens * (tokens + 1) // 2
    return 14 * D * pairs / dt / 1e12, dt


def row_kernel_bytes(w, chunks):
    """Algorithmic HBM bytes per launch of the three row kernels of one step.

    attn_bwd_prep reads O and dO (bf16) and writes D_t (fp32) and the zeroed
    fp32 dQ accumulator row; attn_bwd_dq reads that accumulator and writes bf16
    dQ: 4D + 4 + 4D and 4D + 2D bytes per (row, query head). attn_fwd_merge reads
    (4D + 4) bytes of every key-range partial a re-split row can see and writes
    its bf16 O and fp32 LSE (2D + 4). The partial rows of a two-part split run
    from the 128-row tile holding the split point m to the chunk's end; rows
    before m see the first part only. The merge figure is None for plans with
    P-part splits (kv_split < 0), whose boundaries only the library computes,
    and 0 when no chunk is split."""
    D, rows = w.D, w.B * w.H * w.L
    merge = 0
    for qb, qe, cb, m in chunks:
        if m < 0:
            merge = None
            break
        if m == 0:
            continue
        pr0 = qb + 128 * ((m - qb) // 128) if m > qb else qb
        seen = 2 * (qe - max(pr0, m)) + max(0, m - pr0)
        merge += w.B * w.H * (seen * (4 * D + 4) + (qe - pr0) * (2 * D + 4))
    return {"bwd_prep": rows * (8 * D + 4), "bwd_dq": rows * 6 * D, "fwd_merge": merge}


def hbm_kernels(w, chunks, stage_ms, peak_gbs):
    """Achieved GB/s of the HBM-bound row kernels: algorithmic bytes per launch
    over the launch's mean event time on the launching stream."""
    out = {}
    for name, nbytes in row_kernel_bytes(w, chunks).items():
        if not nbytes or stage_ms[name] <= 0:
            out[name] = None
            continue
        gbs = nbytes / (stage_ms[name] * 1e-3) / 1e9
        out[name] = {"bytes": nbytes, "ms": stage_ms[name], "achieved": gbs, "peak": peak_gbs,
                     "unit": "GB/s", "frac": gbs / peak_gbs}
    return out


def workload_flops(w):
    """Algorithmic fwd+bwd FLOPs of a workload: 14 D per visible pair (per document when packed)."""
    return 14 * w.D * causal_pairs_total(w, None)


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from chunked_causal_attention_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    n_tok = args.cpu_sample_tokens
    for i in range(args.warmup):
        time_oracle_sample(w, max(128, n_tok // 4), 7000 + i)
    vals, secs = [], []
    for i in range(args.steps):
        v, dt = time_oracle_sample(w, n_tok, 8000 + i)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    sample = (f"oracle.attention.backward (float64 fwd+bwd) on a causal prefix of {n_tok} tokens "
              f"of one head (D={w.D}) per step; TFLOP/s = 14*D*pairs/time")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, args),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample,
                             "extrapolated_full_step_s": workload_flops(w) / (value * 1e12),
                             "extrapolation": "the workload's fwd+bwd FLOPs at the sample's rate (not measured)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w, args):
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "D": w.D, "tokens": w.L, "plan_chunks": w.N,
           "plan_mode": ["uniform", "flops", "flops_resplit_edges"][w.mode], "packed": w.packed,
           "l2": f"inputs of {w.B * w.H * w.L * w.D * 2 / 2**30:.3g} GiB per tensor, q/k/v/dO together larger "
                 "than the 129 MB L2; no flush", "parallelism": f"replicas x{args.gpus}"}
    if getattr(args, "heads", 0):
        cfg["heads_override"] = args.heads
    if w.Hkv is not None:
        cfg["Hkv"] = w.Hkv
    if args.plan != "default" and not w.packed:
        cfg["plan_mode"] = args.plan
    return cfg


# ----------------------------------------------------------------- GPU arm
def max_over_ranks(ms, world, device):
    """The slowest rank's time: a job of replicas ends when its last rank does."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_replica_step, steps, world, ms):
    """Whole-job throughput: the FLOPs of every replica's steps over the slowest rank's time."""
    return world * flops_per_replica_step * steps / (ms * 1e-3) / 1e12


def run_ours(args):
    import torch
    import torch.distributed as dist

    import chunked_causal_attention_gb300 as cca
    from chunked_causal_attention_gb300.workloads import WORKLOADS, workload_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    w = WORKLOADS[args.workload]
    if args.heads:
        # fewer heads of the same sequence: a small case for profiler captures (the
        # backward walks heads one after another, so its traffic per head carries over)
        import dataclasses
        g = w.H // (w.Hkv or w.H)
        w = dataclasses.replace(w, H=args.heads, Hkv=None if w.Hkv is None else max(1, args.heads // g))
    if w.packed:
        chunks = cca.attn_plan_varlen(w.cu_seqlens(), w.max_chunk_tokens, w.mode)
    elif args.plan.startswith("multiplex:"):
        chunks = cca.attn_plan_multiplex(w.L, w.N, int(args.plan.split(":")[1]))
    else:
        chunks = cca.attn_plan(w.L, w.N, w.mode)
    q, k, v, do = workload_inputs(w, device=dev)
    shape = cca.shape_of(q, w.scale, w.packed, k)
    o = torch.empty_like(q)
    lse = torch.empty((shape.B, shape.H, shape.T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_f = cca.workspace(shape, chunks, 0, dev)
    ws_b = cca.workspace(shape, chunks, 1, dev)
    stream = torch.cuda.current_stream(dev)
    stages = ["fwd_tiles", "fwd_merge", "bwd_prep", "bwd_tiles", "bwd_dq"]

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        cca.attn_fwd_tiles(q, k, v, chunks, shape, o, lse, ws_f, stream)
        mark(1)
        cca.attn_fwd_merge(chunks, shape, o, lse, ws_f, stream)
        mark(2)
        cca.attn_bwd_prep(o, do, chunks, shape, ws_b, stream)
        mark(3)
        cca.attn_bwd_tiles(q, k, v, lse, do, chunks, shape, dk, dv, ws_b, stream)
        mark(4)
        cca.attn_bwd_dq(chunks, shape, dq, ws_b, stream)
        mark(5)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = cca.attn_status(ws_f, stream) or cca.attn_status(ws_b, stream)
    if st:
        raise RuntimeError(f"device status after warm-up: {cca.strerror(st)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(local, args.clock_log)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    launches0 = cca.kernel_launches()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    launches = cca.kernel_launches() - launches0   # the library's own count of its enqueued kernels
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    stage_ms = {s: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, s in enumerate(stages)}
    st = cca.attn_status(ws_f, stream) or cca.attn_status(ws_b, stream)
    if st:
        raise RuntimeError(f"device status after timed steps: {cca.strerror(st)}")

    total_ms = max_over_ranks(total_ms, world, dev)

    pairs = causal_pairs_total(w, chunks)
    flops_fwd = 4 * w.D * pairs
    flops_bwd = 10 * w.D * pairs
    flops_step = flops_fwd + flops_bwd
    ms_step = total_ms / args.steps
    value = job_tflops(flops_step, args.steps, world, total_ms)

    def streamed_leg():
        # Chunk-streamed calls, as SPPO and InfiniPipe invoke attention: the forward
        # one chunk at a time in chunk order (attn_fwd on a single chunk against the
        # resident keys before it), the backward one chunk at a time in reverse
        # order (attn_bwd_chunk) with fp32 dK/dV accumulators that the calls share.
        ws_fc = cca.workspace(shape, chunks, cca.PASS_FWD, dev, per_chunk=True)
        ws_bc = cca.workspace(shape, chunks, cca.PASS_BWD_CHUNK, dev, per_chunk=True)
        dk_acc = torch.empty_strided(k.shape, k.stride(), dtype=torch.float32, device=dev)
        dv_acc = torch.empty_strided(v.shape, v.stride(), dtype=torch.float32, device=dev)

        def streamed_step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            for c in chunks:
                cca.attn_fwd(q, k, v, [c], shape, o, lse, ws_fc, stream)
            if ev is not None:
                ev[1].record(stream)
            dk_acc.zero_()
            dv_acc.zero_()
            for c in reversed(chunks):
                cca.attn_bwd_chunk(q, k, v, o, lse, do, [c], shape, dq, dk, dv, dk_acc, dv_acc, ws_bc, stream)
            if ev is not None:
                ev[2].record(stream)

        s_steps = max(1, min(args.steps, 3))
        streamed_step()
        s_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(s_steps)]
        barrier()
        torch.cuda.synchronize(dev)
        for i in range(s_steps):
            streamed_step(s_ev[i])
        torch.cuda.synchronize(dev)
        barrier()
        st = cca.attn_status(ws_fc, stream) or cca.attn_status(ws_bc, stream)
        if st:
            raise RuntimeError(f"device status after streamed steps: {cca.strerror(st)}")
        s_fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in s_ev)
        s_bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in s_ev)
        s_job_ms = max_over_ranks(s_fwd_ms + s_bwd_ms, world, dev)
        streamed = {"value": job_tflops(flops_step, 1, world, s_job_ms), "unit": "TFLOP/s",
                    "steps": s_steps, "calls_per_step": 2 * len(chunks),
                    "fwd_tflops": flops_fwd / (s_fwd_ms * 1e-3) / 1e12,
                    "bwd_tflops": flops_bwd / (s_bwd_ms * 1e-3) / 1e12,
                    "ms_per_step": s_fwd_ms + s_bwd_ms,
                    "note": "attn_fwd per chunk in order, attn_bwd_chunk in reverse order; zeroing of the fp32 "
                            "dK/dV accumulators included"}
        del dk_acc, dv_acc, ws_fc, ws_bc
        return streamed

    def e2e_leg():
        # End to end through the public API: every step uploads its inputs from pinned
        # host memory and reads its results back. Uploads and read-backs run on two
        # copy streams of their own with two sets of device buffers, so step i+1's
        # upload and step i-1's read-back overlap step i's kernels and each other;
        # each step still moves all of its own bytes. Within a step the forward waits
        # only for q, k, v (dO's upload overlaps it), and o, lse are read back while
        # the backward runs.
        # enough steps that the pipeline's fill (the first upload) and drain (the last
        # read-back), which no kernel can overlap, stay a small share of the leg
        e2e_steps = max(8, min(4 * args.steps, 24))
        hin = [x.cpu().pin_memory() for x in (q, k, v, do)]
        hout = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (o, lse, dq, dk, dv)]
        bufs = []
        for _ in range(2):
            din = [torch.empty_like(x) for x in (q, k, v, do)]
            dout_ = [torch.empty_like(x) for x in (o, lse, dq, dk, dv)]
            bufs.append((din, dout_))
        h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        tev = lambda: torch.cuda.Event(enable_timing=True)
        h2d_start = [tev() for _ in range(e2e_steps)]
        qkv_done = [tev() for _ in range(e2e_steps)]
        h2d_done = [tev() for _ in range(e2e_steps)]
        fwd_done = [tev() for _ in range(e2e_steps)]
        comp_done = [tev() for _ in range(e2e_steps)]
        d2h_start = [tev() for _ in range(e2e_steps)]
        d2h_fwd_done = [tev() for _ in range(e2e_steps)]
        d2h_bwd_start = [tev() for _ in range(e2e_steps)]
        d2h_done = [tev() for _ in range(e2e_steps)]

        def e2e_upload(i):
            din, _ = bufs[i % 2]
            with torch.cuda.stream(h2d_stream):
                if i >= 2:
                    h2d_stream.wait_event(comp_done[i - 2])       # step i-2 no longer reads these inputs
                h2d_start[i].record(h2d_stream)
                for d_, h_ in zip(din[:3], hin[:3]):
                    d_.copy_(h_, non_blocking=True)
                qkv_done[i].record(h2d_stream)
                din[3].copy_(hin[3], non_blocking=True)
                h2d_done[i].record(h2d_stream)

        barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        d2h_stream.wait_event(e0)
        e2e_upload(0)
        for i in range(e2e_steps):
            din, dout_ = bufs[i % 2]
            q2, k2, v2, do2 = din
            o2, lse2, dq2, dk2, dv2 = dout_
            stream.wait_event(qkv_done[i])
            if i >= 2:
                stream.wait_event(d2h_done[i - 2])               # step i-2's results are read back
            cca.attn_fwd(q2, k2, v2, chunks, shape, o2, lse2, ws_f, stream)
            fwd_done[i].record(stream)
            stream.wait_event(h2d_done[i])                       # dO is in
            cca.attn_bwd(q2, k2, v2, o2, lse2, do2, chunks, shape, dq2, dk2, dv2, ws_b, stream)
            comp_done[i].record(stream)
            if i + 1 < e2e_steps:
                e2e_upload(i + 1)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(fwd_done[i])               # o, lse while the backward runs
                d2h_start[i].record(d2h_stream)
                for h_, d_ in zip(hout[:2], dout_[:2]):
                    h_.copy_(d_, non_blocking=True)
                d2h_fwd_done[i].record(d2h_stream)
                d2h_stream.wait_event(comp_done[i])
                d2h_bwd_start[i].record(d2h_stream)
                for h_, d_ in zip(hout[2:], dout_[2:]):
                    h_.copy_(d_, non_blocking=True)
                d2h_done[i].record(d2h_stream)
        stream.wait_event(d2h_done[e2e_steps - 1])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = e0.elapsed_time(e1)
        # the copies' own time: the dO upload and the dq/dk/dv read-back may wait for
        # compute, so each group of copies is timed from its own start
        h2d_ms = sum(h2d_start[i].elapsed_time(h2d_done[i]) for i in range(e2e_steps))
        d2h_ms = sum(d2h_start[i].elapsed_time(d2h_fwd_done[i]) + d2h_bwd_start[i].elapsed_time(d2h_done[i])
                     for i in range(e2e_steps))
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        nbytes = lambda x: x.numel() * x.element_size()
        h2d = sum(nbytes(x) for x in (q, k, v, do))
        d2h = sum(nbytes(x) for x in (o, lse, dq, dk, dv))
        e2e_value = job_tflops(flops_step, e2e_steps, world, e2e_ms)
        return {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "copies": "pinned host buffers; upload and read-back streams overlapped with compute; the forward "
                          "waits for q, k, v only, and o, lse are read back during the backward",
                "h2d_gbs": h2d * e2e_steps / (h2d_ms * 1e-3) / 1e9,
                "d2h_gbs": d2h * e2e_steps / (d2h_ms * 1e-3) / 1e9}

    # --device-only (large workloads whose second set of e2e buffers would not fit,
    # or whose chunk-streamed leg would take minutes) reports the device leg alone
    skipped = {"skipped": "--device-only"}
    streamed = skipped if args.device_only else streamed_leg()
    e2e = skipped if args.device_only else e2e_leg()

    peaks, peak_src = load_peaks()
    fwd_tflops = flops_fwd / ((stage_ms["fwd_tiles"] + stage_ms["fwd_merge"]) * 1e-3) / 1e12
    bwd_tflops = flops_bwd / ((stage_ms["bwd_prep"] + stage_ms["bwd_tiles"] + stage_ms["bwd_dq"]) * 1e-3) / 1e12
    dom = "bwd_tiles"
    dom_ms = stage_ms[dom]
    achieved = flops_bwd / (dom_ms * 1e-3) / 1e12
    peak_sus = peaks["bf16_tflops_sustained"]
    peak_burst = peaks["bf16_tflops"]

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(w, args),
            "pct_of_peak": {"burst": 100 * value / world / peak_burst, "sustained": 100 * value / world / peak_sus,
                            "fwd_burst": 100 * fwd_tflops / peak_burst, "bwd_burst": 100 * bwd_tflops / peak_burst,
                            "peak_source": peak_src},
            "fwd_tflops": fwd_tflops,
            "bwd_tflops": bwd_tflops,
            "stage_ms": stage_ms,
            "roofline": {"kernel": "bwd key-tile kernel (attn_bwd_tiles)", "bound": "tensor",
                         "achieved": achieved, "peak": peak_sus, "unit": "TFLOP/s", "frac": achieved / peak_sus,
                         "peak_kind": f"bf16_tflops_sustained ({peak_src})",
                         "frac_of_burst": achieved / peak_burst, "traffic": None if args.heads else measured_traffic(w.name),
                         "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"},
            "hbm_kernels": hbm_kernels(w, chunks, stage_ms, peaks["hbm_gbs"]),
            "gpu_launches": launches,
            "e2e": e2e,
            "clocks": clk,
            "streamed": streamed,
        }
        if world == 1 and not args.no_cpu_baseline:
            v_cpu, dt = time_oracle_sample(w, args.cpu_sample_tokens, 9000)
            line["cpu_baseline"] = {
                "value": v_cpu, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                "sample": f"oracle.attention.backward (float64 fwd+bwd) on a causal prefix of "
                          f"{args.cpu_sample_tokens} tokens of one head, {dt:.1f} s",
                "extrapolated_full_step_s": flops_step / (v_cpu * 1e12),
                "extrapolation": "the workload's fwd+bwd FLOPs at the sample's rate (not measured)"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="7b_128k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=CPU_SAMPLE_TOKENS,
                    help="causal prefix that the oracle (cpu_baseline, reference arm) is timed on")
    ap.add_argument("--device-only", action="store_true",
                    help="report the device-timed leg only (no chunk-streamed and no end-to-end leg)")
    ap.add_argument("--plan", default="default",
                    help="default (the workload's plan) or multiplex:PP (SPPO Table 3 edge re-splits)")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the workload with this many heads instead of its own (small profiler captures)")
    ap.add_argument("--clock-log", default=None,
                    help="also write the raw nvidia-smi clock samples of the timed region to this CSV file")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
