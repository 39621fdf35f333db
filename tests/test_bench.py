"""Host-side checks of bench.py (no GPU): the oracle arm's JSON line, the
gating of the committed ncu traffic record by the kernel sources' hash, the
workload config keys, the replicas' timing over gloo with two ranks, the
row kernels' algorithmic bytes, and the GPU arm's whole JSON line on a fake
device (torch.cuda and the compute calls replaced by stand-ins)."""
import json
import os
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "7b_32k", "--cpu-sample-tokens", "2048"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["dtype"] == "f64"
    assert d["config"]["workload"] == "7b_32k"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    from chunked_causal_attention_gb300.workloads import WORKLOADS
    w = WORKLOADS["7b_32k"]
    full = 14 * w.D * w.H * w.L * (w.L + 1) // 2
    assert abs(d["cpu_baseline"]["extrapolated_full_step_s"] - full / (d["value"] * 1e12)) < 1e-6 * full / (d["value"] * 1e12)
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_record_is_gated_by_source_hash(tmp_path, monkeypatch):
    rec = {"workload": "7b_128k", "dram_bytes_read": 3.0, "dram_bytes_write": 4.0,
           "source_sha256": bench.kernel_source_hash()}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(p))
    assert bench.measured_traffic("7b_128k") == 7.0
    assert bench.measured_traffic("7b_32k") is None              # another workload
    rec["source_sha256"] = "0" * 64                               # kernel changed since the capture
    p.write_text(json.dumps(rec))
    assert bench.measured_traffic("7b_128k") is None
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(tmp_path / "missing.json"))
    assert bench.measured_traffic("7b_128k") is None


def test_source_hash_follows_the_backward_kernel_only(tmp_path, monkeypatch):
    """The traffic record's hash covers the backward tile kernel, its device
    headers and the backward's layout, order and launch code in attn_api.cpp:
    an edit there changes it, an edit of the forward kernel or of forward-only
    host code does not."""
    import shutil
    src = os.path.join(ROOT, "chunked_causal_attention_gb300", "csrc")
    dst = tmp_path / "chunked_causal_attention_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()

    def edited(name, old, new):
        path = dst / name
        text = path.read_text()
        assert old in text
        path.write_text(text.replace(old, new, 1))
        h = bench.kernel_source_hash()
        path.write_text(text)
        return h

    assert edited("fwd_tc.cu", "namespace attn {", "namespace attn {\n") == h0
    assert edited("attn_api.cpp", "constexpr int32_t kGroupFwd", "constexpr int32_t kGroupFwd ") == h0
    assert edited("bwd_tc.cu", "namespace attn {", "namespace attn {\n") != h0
    assert edited("attn_api.cpp", "constexpr int32_t kGroupBwd", "constexpr int32_t kGroupBwd ") != h0
    assert edited("attn_api.cpp", "void bwd_layout(", "void  bwd_layout(") != h0
    assert edited("attn_api.cpp", "        a.group = kGroupBwd;", "        a.group = kGroupBwd; ") != h0
    assert bench.kernel_source_hash() == h0


def test_committed_traffic_record_names_its_kernel_and_command():
    with open(os.path.join(ROOT, "profiles", "traffic_7b_128k.json")) as f:
        rec = json.load(f)
    assert rec["workload"] == "7b_128k" and len(rec["source_sha256"]) == 64
    assert rec["dram_bytes_read"] > 0 and rec["dram_bytes_write"] > 0
    assert "--clock-control none" in rec["command"] and "bwd_tc_kernel" in rec["kernel"]


@pytest.mark.parametrize("name", ["tiny", "7b_32k", "7b_128k", "packed_256k", "13b_1m", "gqa_128k"])
def test_workload_config(name):
    from chunked_causal_attention_gb300.workloads import WORKLOADS
    w = WORKLOADS[name]
    args = types.SimpleNamespace(gpus=1, plan="default")
    cfg = bench.workload_config(w, args)
    assert cfg["workload"] == name and cfg["D"] == w.D and cfg["H"] == w.H and cfg["packed"] == w.packed
    assert "model" not in cfg
    if w.Hkv is not None:
        assert cfg["Hkv"] == w.Hkv
    assert "heads_override" not in cfg
    small = bench.workload_config(w, types.SimpleNamespace(gpus=1, plan="default", heads=2))
    assert small["heads_override"] == 2


def test_reference_arm_under_torchrun_prints_from_rank_0_only():
    """The driver launches N > 1 through torchrun: rank 0 alone runs the oracle
    arm and prints its line, the other ranks exit 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "7b_32k",
                        "--cpu-sample-tokens", "2048"],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def _replica_rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 100.0 + 50.0 * rank                 # rank 1 is the slow one
        job_ms = bench.max_over_ranks(ms, world, "cpu")
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"job_ms": job_ms, "tflops": bench.job_tflops(1e12, 4, world, job_ms)}, f)
    finally:
        dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_over_gloo(tmp_path):
    """N > 1 runs one replica per rank: every rank times the job by the slowest
    rank, and the whole-job value counts the work of all ranks."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_replica_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["job_ms"] == 150.0
        # 2 replicas x 4 steps x 1e12 FLOP in 0.15 s
        assert abs(g["tflops"] - 2 * 4 * 1.0 / 0.15) < 1e-9
    assert bench.max_over_ranks(7.0, 1, "cpu") == 7.0


def test_row_kernel_bytes():
    """Algorithmic bytes of the HBM-bound row kernels, counted by hand."""
    import chunked_causal_attention_gb300 as cca
    from chunked_causal_attention_gb300.workloads import WORKLOADS, Workload
    w = WORKLOADS["7b_128k"]
    rows = 32 * 131072
    got = bench.row_kernel_bytes(w, cca.attn_plan(w.L, w.N, w.mode))
    assert got["bwd_prep"] == rows * (2 * 256 + 4 + 512)       # O, dO in; D_t and the zeroed accumulator out
    assert got["bwd_dq"] == rows * (512 + 256)                  # fp32 accumulator in, bf16 dQ out
    # first chunk [0, 32768) split at 16384, last [126848, 131072) at 129024: every
    # partial row lies past its split point and reads both parts
    assert got["fwd_merge"] == 32 * (16384 + 2048) * (2 * (4 * 128 + 4) + 2 * 128 + 4)
    assert bench.row_kernel_bytes(w, cca.attn_plan_multiplex(w.L, w.N, 3))["fwd_merge"] is None
    assert bench.row_kernel_bytes(w, cca.attn_plan(w.L, w.N, cca.PLAN_FLOPS))["fwd_merge"] == 0
    # a split point inside a tile: partial rows from 256, rows 256..299 see the first part only
    small = Workload("s", 1, 2, 64, 1000)
    got = bench.row_kernel_bytes(small, [(0, 1000, 0, 300)])
    assert got["fwd_merge"] == 2 * ((44 + 2 * 700) * (4 * 64 + 4) + 744 * (2 * 64 + 4))
    hk = bench.hbm_kernels(small, [(0, 1000, 0, 0)], {"bwd_prep": 1.0, "bwd_dq": 0.5, "fwd_merge": 0.01}, 1000.0)
    assert hk["fwd_merge"] is None
    assert hk["bwd_prep"]["achieved"] == pytest.approx(2000 * (8 * 64 + 4) / 1e-3 / 1e9)
    assert hk["bwd_dq"]["frac"] == pytest.approx(2000 * 6 * 64 / 0.5e-3 / 1e9 / 1000.0)


class _FakeEvent:
    """A CUDA event stand-in: every record advances a clock by 1 ms."""
    clock = [0.0]

    def __init__(self, enable_timing=False):
        self.t = None

    def record(self, stream=None):
        _FakeEvent.clock[0] += 1.0
        self.t = _FakeEvent.clock[0]

    def elapsed_time(self, other):
        return other.t - self.t


class _FakeStream:
    def wait_event(self, event):
        pass


def test_gpu_arm_json_line_with_a_fake_device(monkeypatch, capsys):
    """The GPU arm's host logic end to end, with torch.cuda, the device and the
    compute calls replaced by stand-ins (no kernel runs): the JSON line has
    every key the bench contract asks for, on a small plan with re-split edges."""
    import contextlib

    import torch
    import chunked_causal_attention_gb300 as cca
    from chunked_causal_attention_gb300 import workloads as W

    real_torch = torch

    class TorchProxy(types.ModuleType):
        def __init__(self):
            super().__init__("torch")
            self.cuda = types.SimpleNamespace(
                set_device=lambda *a: None, Event=_FakeEvent, synchronize=lambda *a: None,
                current_stream=lambda *a: _FakeStream(), Stream=lambda *a: _FakeStream(),
                stream=lambda s: contextlib.nullcontext())

        def __getattr__(self, name):
            return getattr(real_torch, name)

        def device(self, *args, **kwargs):
            return real_torch.device("cpu")

        def empty(self, *args, pin_memory=False, **kwargs):
            return real_torch.empty(*args, **kwargs)

    calls = []
    for name in ("attn_fwd_tiles", "attn_fwd_merge", "attn_bwd_prep", "attn_bwd_tiles", "attn_bwd_dq", "attn_fwd",
                 "attn_bwd", "attn_bwd_chunk"):
        monkeypatch.setattr(cca, name, lambda *a, _n=name: calls.append(_n))
    monkeypatch.setattr(cca, "attn_status", lambda *a: 0)
    monkeypatch.setattr(cca, "kernel_launches", lambda: len(calls))   # one launch per stand-in call
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    monkeypatch.setitem(sys.modules, "torch", TorchProxy())
    monkeypatch.setitem(W.WORKLOADS, "mini_resplit",
                        W.Workload("mini_resplit", 1, 2, 64, 2048, N=4, mode=W.PLAN_FLOPS_RESPLIT_EDGES, seed=5))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "2", "--warmup", "3", "--workload", "mini_resplit",
                                      "--cpu-sample-tokens", "256"])
    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
                "hbm_kernels", "streamed"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["n_gpus"] == 1 and d["steps"] == 2 and d["value"] > 0
    assert d["config"]["workload"] == "mini_resplit"
    assert d["roofline"]["bound"] == "tensor" and 0 < d["roofline"]["frac"]
    assert d["e2e"]["h2d_bytes_per_step"] == 4 * 2 * 2048 * 64 * 2
    assert d["e2e"]["d2h_bytes_per_step"] == 4 * 2 * 2048 * 64 * 2 + 2 * 2048 * 4
    assert d["hbm_kernels"]["fwd_merge"]["bytes"] > 0 and d["hbm_kernels"]["bwd_prep"]["frac"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert d["gpu_launches"] == 5 * 2
    for key in ("burst", "sustained", "fwd_burst", "bwd_burst"):
        assert d["pct_of_peak"][key] > 0
    # one step = the five stage calls; warm-up and timed steps, then the streamed and e2e legs
    assert calls[:5] == ["attn_fwd_tiles", "attn_fwd_merge", "attn_bwd_prep", "attn_bwd_tiles", "attn_bwd_dq"]
    assert calls.count("attn_bwd_tiles") == 3 + 2
