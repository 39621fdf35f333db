"""attn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Those callers (code hosted by a runtime that owns all device memory and
exposes no allocator, or code that must not allocate once it is running)
cannot provide the workspace that attn_fwd needs. attn_fwd_noalloc uses
scratch memory that lives inside the library instead; attn_noalloc_status
reads that path's device error word. This file checks it through the C ABI:

- against attn_fwd with its own workspace on the same inputs, bit for bit
  (the same kernels and work list, and no order-dependent reduction), over a
  sequence of calls with different shapes and plans run in one order and then
  in the reverse order, so that no call is disturbed by what an earlier one
  left in the shared scratch (work list, merge segments, partials);
- once against the float64 oracle;
- that a bounded wait that gives up is reported by attn_noalloc_status and
  that the read clears it;
- that a request larger than the scratch is refused on the host;
- that a call after the caller resets the device (cudaDeviceReset) finds the
  scratch in the new context (a child process, with no framework holding
  device memory across the reset).

pytest collects this file last.
"""
import ctypes

import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300 import _lib
from chunked_causal_attention_gb300.workloads import make_inputs
from oracle import attention as A
from oracle import plan as P

from parity import check_fwd, head, lse_head

pytestmark = pytest.mark.gpu

ATTN_E_WORKSPACE = 4
ATTN_E_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(_lib.LIB_PATH):
        from chunked_causal_attention_gb300 import build
        build.build()


def call_noalloc(q, k, v, chunks, shape, o, lse):
    arr, n = _lib.chunk_array(chunks)
    stream = torch.cuda.current_stream().cuda_stream
    return cca.lib().attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), arr, n, ctypes.byref(shape),
                                      o.data_ptr(), lse.data_ptr(), stream)


def noalloc_status():
    return cca.lib().attn_noalloc_status(torch.cuda.current_stream().cuda_stream)


# (B, H, L, D, plan, seed): a two-part edge re-split (partials and a merge), an
# unsplit plan (no partials), P-part re-splits (a wider partial layout and more
# merge segments) and another two-part re-split with a different partial layout
CASES = [
    (1, 4, 4096, 128, P.plan(4096, 3, P.FLOPS_RESPLIT_EDGES), 901),
    (2, 3, 1000, 64, P.plan(1000, 2, P.UNIFORM), 902),
    (1, 4, 4096, 128, P.plan_multiplex(4096, 4, 3), 903),
    (1, 2, 3000, 96, P.plan(3000, 4, P.FLOPS_RESPLIT_EDGES), 904),
]


def run_case(case):
    B, H, L, D, chunks, seed = case
    q, k, v, _ = (x.cuda() for x in make_inputs(B, H, L, D, seed=seed))
    shape = cca.shape_of(q)
    assert cca.attn_workspace_size(shape, chunks, 0) <= _lib.NOALLOC_SCRATCH_BYTES
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, L), float("nan"), device="cuda")
    st = call_noalloc(q, k, v, chunks, shape, o, lse)
    assert st == 0, cca.strerror(st)
    assert noalloc_status() == 0
    return (q, k, v), o, lse


def test_noalloc_equals_attn_fwd_bit_for_bit_in_both_orders():
    refs = {}
    for i, case in enumerate(CASES):
        B, H, L, D, chunks, seed = case
        q, k, v, _ = (x.cuda() for x in make_inputs(B, H, L, D, seed=seed))
        refs[i] = cca.forward(q, k, v, chunks)
    torch.cuda.synchronize()
    order = list(range(len(CASES)))
    for i in order + order[::-1] + [0, 2, 3]:
        _, o, lse = run_case(CASES[i])
        o_ref, lse_ref = refs[i]
        assert torch.equal(o, o_ref), f"case {i}: O differs from attn_fwd"
        assert torch.equal(lse, lse_ref), f"case {i}: LSE differs from attn_fwd"


def test_noalloc_matches_the_oracle():
    (q, k, v), o, lse = run_case(CASES[0])
    B, H, L, D, chunks, _ = CASES[0]
    for h in range(H):
        ro, rl = A.forward(head(q, 0, h, False), head(k, 0, h, False), head(v, 0, h, False), D ** -0.5)
        check_fwd(head(o, 0, h, False), lse_head(lse, 0, h), ro, rl, f"noalloc h{h}")


def test_noalloc_status_reports_a_wait_that_gave_up(monkeypatch):
    """With the test-only producer stall no tile is loaded, so the forward's
    bounded waits give up; the error lands in the library scratch's status
    word, which attn_noalloc_status reads and clears. A normal call afterwards
    in the same context still equals attn_fwd."""
    B, H, L, D, chunks, seed = CASES[0]
    q, k, v, _ = (x.cuda() for x in make_inputs(B, H, L, D, seed=seed))
    shape = cca.shape_of(q)
    o = torch.zeros_like(q)
    lse = torch.zeros((B, H, L), device="cuda")
    monkeypatch.setenv("ATTN_WAIT_LIMIT_MS", "200")
    monkeypatch.setenv("ATTN_TEST_STALL_PRODUCER", "1")
    assert call_noalloc(q, k, v, chunks, shape, o, lse) == 0    # enqueued; the error is on the device
    assert noalloc_status() == ATTN_E_TIMEOUT
    assert noalloc_status() == 0                                 # the read cleared it
    monkeypatch.delenv("ATTN_TEST_STALL_PRODUCER")
    monkeypatch.delenv("ATTN_WAIT_LIMIT_MS")
    o_ref, lse_ref = cca.forward(q, k, v, chunks)
    _, o, lse = run_case(CASES[0])
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_noalloc_refuses_requests_beyond_its_scratch():
    B, H, L, D = 1, 32, 32768, 128
    chunks = P.plan(L, 8, P.FLOPS_RESPLIT_EDGES)              # the partials need ~1 GB
    shape = cca.make_shape(B, H, L, D, H * L * D, D, L * D, D ** -0.5)
    assert cca.attn_workspace_size(shape, chunks, 0) > _lib.NOALLOC_SCRATCH_BYTES
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never read: refused on the host
    st = call_noalloc(q, q, q, chunks, shape, q, q)
    assert st == ATTN_E_WORKSPACE, cca.strerror(st)


def test_noalloc_after_a_device_reset():
    import glob
    import os
    import subprocess
    import sys
    libs = sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
    if not libs:
        pytest.skip("no CUDA runtime library to reset the device through")
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "noalloc_reset_child.py")
    r = subprocess.run([sys.executable, child, libs[0]], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(line.split(" ", 1) for line in r.stdout.splitlines() if " " in line)
    assert lines["status"].split() == ["0", "0", "0", "0"], r.stdout
    assert lines["equal"] == "1" and lines["finite"] == "1", r.stdout
