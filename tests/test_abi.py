"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/attn.h declares, its planner equals the oracle's bit for bit, and
argument errors are reported on the host before anything is enqueued."""
import ctypes
import os
import random
import re

import pytest

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300 import _lib
from oracle import plan as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "attn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", txt)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(_lib.LIB_PATH):
        from chunked_causal_attention_gb300 import build
        build.build()


def test_exports_every_declared_symbol():
    syms = header_symbols()
    assert len(syms) >= 13
    L = cca.lib()
    for s in syms:
        assert hasattr(L, s), s
    assert set(syms) == set(_lib.EXPORTS)
    assert "sm_103a" in cca.version()


def test_plan_matches_oracle_exactly():
    rng = random.Random(11)
    cases = [(1024, 4, 0), (32768, 8, 1), (131072, 16, 2), (1 << 20, 64, 1), (1000, 3, 0), (2688, 4, 1)]
    cases += [(rng.randint(1, 1 << 21), rng.randint(1, 64), rng.randint(0, 2)) for _ in range(400)]
    for L, N, mode in cases:
        try:
            want = P.plan(L, N, mode)
        except P.PlanError:
            with pytest.raises(cca.AttnError) as e:
                cca.attn_plan(L, N, mode)
            assert e.value.status == 1
            continue
        assert cca.attn_plan(L, N, mode) == want, (L, N, mode)


def test_plan_varlen_matches_oracle_exactly():
    rng = random.Random(12)
    for _ in range(100):
        nd = rng.randint(1, 12)
        lens = [rng.choice([0, 1, 5, 127, 128, 129, rng.randint(1, 70000)]) for _ in range(nd)]
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        if cu[-1] == 0:
            continue
        mct = rng.choice([128, 1000, 16384])
        for mode in (0, 1, 2):
            try:
                want = P.plan_varlen(cu, mct, mode)
            except P.PlanError:
                with pytest.raises(cca.AttnError):
                    cca.attn_plan_varlen(cu, mct, mode)
                continue
            assert cca.attn_plan_varlen(cu, mct, mode) == want


def test_plan_errors():
    L = cca.lib()
    out = (_lib.attn_chunk * 4)()
    n = ctypes.c_int32(0)
    assert L.attn_plan(0, 4, 1, out, 4, ctypes.byref(n)) == 1
    assert L.attn_plan(1024, 0, 1, out, 4, ctypes.byref(n)) == 1
    assert L.attn_plan(1024, 4, 7, out, 4, ctypes.byref(n)) == 1
    assert L.attn_plan(1024, 16, 1, out, 4, ctypes.byref(n)) == 1         # collapsing boundaries
    assert L.attn_plan(1024, 4, 1, out, 2, ctypes.byref(n)) == 8          # capacity
    assert L.attn_plan(1024, 4, 1, out, 4, None) == 1


def shape(B=1, H=2, T=1024, D=64, scale=0.125):
    return cca.make_shape(B, H, T, D, H * T * D, D, T * D, scale)


def test_workspace_size_validation():
    ch = cca.attn_plan(1024, 4, 0)
    assert cca.attn_workspace_size(shape(), ch, 0) >= 256
    assert cca.attn_workspace_size(shape(), ch, 1) >= 2 * 1024 * 64 * 4
    # head dims: multiples of 8 from 8 to 256, forward and backward
    for D in (8, 40, 80, 96, 120, 136, 192, 256):
        assert cca.attn_workspace_size(shape(D=D), ch, 0) >= 256
        assert cca.attn_workspace_size(shape(D=D), ch, 1) >= 2 * 1024 * D * 4
        assert cca.attn_workspace_size(shape(D=D), ch[:1], 2) >= 256
    for D in (4, 100, 264, 512):
        for pass_ in (0, 1, 2):
            with pytest.raises(cca.AttnError) as e:
                cca.attn_workspace_size(shape(D=D), ch if pass_ < 2 else ch[:1], pass_)
            assert e.value.status == 3
    bad = [(0, 600, 0, 0), (500, 1024, 0, 0)]                  # overlapping
    with pytest.raises(cca.AttnError):
        cca.attn_workspace_size(shape(), bad, 0)
    gap = [(0, 500, 0, 0), (600, 1024, 0, 0)]                  # fine forward, not a partition
    cca.attn_workspace_size(shape(), gap, 0)
    with pytest.raises(cca.AttnError):
        cca.attn_workspace_size(shape(), gap, 1)
    badsplit = [(0, 1024, 0, 1024)]
    with pytest.raises(cca.AttnError):
        cca.attn_workspace_size(shape(), badsplit, 0)
    baddoc = [(0, 512, 0, 0), (512, 1024, 100, 0)]             # ctx neither continues nor starts a doc
    with pytest.raises(cca.AttnError):
        cca.attn_workspace_size(shape(), baddoc, 1)
    with pytest.raises(cca.AttnError) as e:
        cca.attn_workspace_size(cca.make_shape(1, 2, 1024, 64, 2 * 1024 * 64, 60, 1024 * 64, 0.1), ch, 0)
    assert e.value.status == 2                                  # token stride not a multiple of 8


def test_workspace_partials_sized_for_split_rows():
    s = cca.make_shape(1, 32, 131072, 128, 32 * 131072 * 128, 128, 131072 * 128, 0.088)
    ch = cca.attn_plan(131072, 16, 2)
    unsplit = [(a, b, c, 0) for a, b, c, _ in ch]
    rows = (32768 - 16384) + (131072 - 129024)
    extra = cca.attn_workspace_size(s, ch, 0) - cca.attn_workspace_size(s, unsplit, 0)
    assert extra >= 2 * rows * 32 * (128 + 1) * 4


def test_grouped_heads_shape_validation():
    """Hkv must divide H; key/value strides follow the same alignment rule."""
    ch = cca.attn_plan(1024, 4, 0)
    ok = cca.make_shape(1, 8, 1024, 64, 8 * 1024 * 64, 64, 1024 * 64, 0.1, 2, 2 * 1024 * 64, 64, 1024 * 64)
    assert cca.attn_workspace_size(ok, ch, 1) > 0
    for bad, st in [((3, 3 * 1024 * 64, 64, 1024 * 64), 1),        # 8 % 3 != 0
                    ((16, 16 * 1024 * 64, 64, 1024 * 64), 1),      # more key/value heads than query heads
                    ((2, 2 * 1024 * 64, 60, 1024 * 64), 2),        # key/value token stride not a multiple of 8
                    ((2, 0, 64, 1024 * 64), 1),
                    ((-1, 0, 0, 0), 1)]:
        s = cca.make_shape(1, 8, 1024, 64, 8 * 1024 * 64, 64, 1024 * 64, 0.1, *bad)
        with pytest.raises(cca.AttnError) as e:
            cca.attn_workspace_size(s, ch, 0)
        assert e.value.status == st, bad


def test_compute_calls_reject_bad_arguments_on_host():
    """Validation happens before any CUDA call, so these run without a GPU."""
    L = cca.lib()
    launches0 = cca.kernel_launches()
    ch, n = _lib.chunk_array(cca.attn_plan(1024, 4, 0))
    s = shape()
    fake = ctypes.c_void_p(4096)
    ws = ctypes.c_void_p(1 << 20)
    # D unsupported (not a multiple of 8, or above 256)
    for D in (100, 264):
        sD = cca.make_shape(1, 2, 1024, D, 2 * 1024 * D, D, 1024 * D, 0.1)
        assert L.attn_fwd(fake, fake, fake, ch, n, ctypes.byref(sD), fake, fake, ws, 1 << 30, None) == 3
        assert L.attn_bwd(fake, fake, fake, fake, fake, fake, ch, n, ctypes.byref(sD), fake, fake, fake, ws,
                          1 << 30, None) == 3
        one, n1 = _lib.chunk_array(cca.attn_plan(1024, 4, 0)[:1])
        assert L.attn_bwd_chunk(fake, fake, fake, fake, fake, fake, one, n1, ctypes.byref(sD), fake, fake, fake,
                                fake, fake, ws, 1 << 30, None) == 3
    # misaligned q
    assert L.attn_fwd(ctypes.c_void_p(4098), fake, fake, ch, n, ctypes.byref(s), fake, fake, ws, 1 << 30, None) == 2
    # workspace too small / missing
    assert L.attn_fwd(fake, fake, fake, ch, n, ctypes.byref(s), fake, fake, ws, 16, None) == 4
    assert L.attn_bwd(fake, fake, fake, fake, fake, fake, ch, n, ctypes.byref(s), fake, fake, fake, None, 0,
                      None) == 4
    # null output
    assert L.attn_fwd(fake, fake, fake, ch, n, ctypes.byref(s), None, fake, ws, 1 << 30, None) == 1
    # bad chunk table
    bad, nb = _lib.chunk_array([(0, 2000, 0, 0)])
    assert L.attn_fwd(fake, fake, fake, bad, nb, ctypes.byref(s), fake, fake, ws, 1 << 30, None) == 1
    assert L.attn_status(None, None) == 1
    assert cca.strerror(4).startswith("workspace")
    assert cca.kernel_launches() == launches0   # a call refused on the host enqueues nothing


def test_chunk_backward_workspace_and_host_errors():
    """attn_bwd_chunk (pass 2): delta and the dQ accumulator sized for the
    chunks' rows; chunks of one call must have disjoint key ranges; argument
    errors found before any CUDA call."""
    s = shape()                                                 # B1 H2 T1024 D64
    with pytest.raises(cca.AttnError) as e:
        cca.attn_workspace_size(s, cca.attn_plan(1024, 4, 0), 2)   # later chunks' contexts overlap earlier ones
    assert e.value.status == 1
    two = cca.attn_workspace_size(s, [(0, 100, 0, 0), (300, 400, 100, 0)], 2)   # two documents
    assert two >= 2 * 200 * (64 + 1) * 4
    n1 = cca.attn_workspace_size(s, [(256, 512, 0, 0)], 2)
    n2 = cca.attn_workspace_size(s, [(256, 1024, 0, 0)], 2)
    assert n1 >= 2 * 256 * (64 + 1) * 4 and n2 - n1 >= 2 * 512 * (64 + 1) * 4 - 1024
    with pytest.raises(cca.AttnError):
        cca.attn_workspace_size(s, [(512, 256, 0, 0)], 2)
    L = cca.lib()
    fake = ctypes.c_void_p(4096)
    ws = ctypes.c_void_p(1 << 20)
    one, _ = _lib.chunk_array([(256, 512, 0, 0)])
    args = [fake] * 6

    def call(chunk=one, dk_acc=fake, dv_acc=fake, ws_bytes=1 << 30, n=1):
        return L.attn_bwd_chunk(*args, chunk, n, ctypes.byref(s), fake, fake, fake, dk_acc, dv_acc, ws, ws_bytes,
                                None)
    assert call(dk_acc=None) == 1
    assert call(dv_acc=ctypes.c_void_p(4100)) == 2
    assert call(ws_bytes=n1 - 1) == 4
    bad, _ = _lib.chunk_array([(256, 2000, 0, 0)])
    assert call(chunk=bad) == 1
    nested, _ = _lib.chunk_array([(256, 512, 300, 0)])            # ctx_begin after q_begin
    assert call(chunk=nested) == 1
    overlap, _ = _lib.chunk_array([(0, 100, 0, 0), (100, 200, 0, 0)])   # second context covers the first chunk
    assert call(chunk=overlap, n=2) == 1
    assert call(n=0) == 1


def test_plan_infinipipe_matches_oracle_exactly():
    """attn_plan_infinipipe (C++) against oracle.infinipipe on random inputs:
    the same calls, chunk for chunk, including float64 threshold decisions."""
    from oracle import infinipipe as IP
    rng = random.Random(11)
    checked = 0
    for it in range(600):
        n = rng.randint(1, 40)
        top = rng.choice([300, 5000, 40000, 300000])
        lengths = [rng.choice([0, rng.randint(1, 128), rng.randint(1, top)]) for _ in range(n)]
        K = rng.randint(1, 10)
        a1 = rng.choice([1.0, 3.3e-10, 1e-9, 7.1e-11])
        a2 = rng.choice([0.0, 2.2e-5, 1e-3, 31.0])
        b1 = rng.choice([0.0, 1e-4, 2.5])
        cap = rng.choice([1000, 20000, 70000, 400000])
        try:
            want, _ = IP.plan(lengths, K, cap, IP.Cost(a1, a2, b1))
        except IP.PlanError:
            with pytest.raises(cca.AttnError) as e:
                cca.attn_plan_infinipipe(lengths, K, cap, a1, a2, b1)
            assert e.value.status == 1
            continue
        got = cca.attn_plan_infinipipe(lengths, K, cap, a1, a2, b1)
        assert got == [list(c) for c in want], (lengths, K, cap, a1, a2, b1)
        checked += 1
    assert checked > 300
    # the hand-worked cases of the oracle's pins (bucket packing, the starting threshold)
    for lengths, cap in (([1024, 300, 256, 200, 128, 100], 1024), ([1024, 800, 700, 100], 2048)):
        want, _ = IP.plan(lengths, 2, cap, IP.Cost(1.0, 0.0, 0.0))
        assert cca.attn_plan_infinipipe(lengths, 2, cap, 1.0, 0.0, 0.0) == [list(c) for c in want]


def test_plan_infinipipe_workload_lengths():
    """The packed 256K workload's document lengths (one 128K document and 15
    shorter ones) with the costs and K used by the streamed measurement."""
    from oracle import infinipipe as IP
    from chunked_causal_attention_gb300.workloads import WORKLOADS
    cu = WORKLOADS["packed_256k"].cu_seqlens()
    lengths = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    for K, cap in [(4, 65536), (8, 65536), (16, 131072)]:
        got = cca.attn_plan_infinipipe(lengths, K, cap, 1.0, 2000.0, 0.0)
        want, info = IP.plan(lengths, K, cap, IP.Cost(1.0, 2000.0, 0.0))
        assert got == [list(c) for c in want]
        assert sum(qe - qb for call in got for qb, qe, _, _ in call) == cu[-1]


def test_plan_infinipipe_errors():
    with pytest.raises(cca.AttnError) as e:
        cca.attn_plan_infinipipe([1000], 16, 10 ** 6, 1.0, 0.0, 0.0)       # mesh collapses
    assert e.value.status == 1
    with pytest.raises(cca.AttnError):
        cca.attn_plan_infinipipe([4096, 10], 2, 1000, 1.0, 0.0, 0.0)        # capacity below the first slice
    with pytest.raises(cca.AttnError):
        cca.attn_plan_infinipipe([4096], 2, 4096, 0.0, 0.0, 1.0)            # no per-token cost
    with pytest.raises(cca.AttnError):
        cca.attn_plan_infinipipe([4096], 2, 4096, float("nan"), 0.0, 1.0)
    with pytest.raises(cca.AttnError):
        cca.attn_plan_infinipipe([4096, -1], 2, 4096, 1.0, 0.0, 0.0)
    assert cca.attn_plan_infinipipe([0, 0], 2, 100, 1.0, 0.0, 0.0) == []
    L = cca.lib()
    lens = (ctypes.c_int64 * 3)(5000, 300, 200)
    out = (_lib.attn_chunk * 1)()
    off = (ctypes.c_int32 * 1)()
    n, nc = ctypes.c_int32(0), ctypes.c_int32(0)
    assert L.attn_plan_infinipipe(lens, 3, 2, 10000, 1.0, 0.0, 0.0, out, 1, ctypes.byref(n), off, 1,
                                  ctypes.byref(nc)) == 8
    assert n.value >= 3 and nc.value >= 2


def test_plan_multiplex_matches_oracle_exactly():
    for L in (1024, 4096, 32768, 131072, 1 << 20, 100000):
        for N in (1, 2, 4, 8, 16):
            for PP in (1, 2, 3, 4, 8):
                try:
                    want = P.plan_multiplex(L, N, PP)
                except P.PlanError:
                    with pytest.raises(cca.AttnError):
                        cca.attn_plan_multiplex(L, N, PP)
                    continue
                assert cca.attn_plan_multiplex(L, N, PP) == want, (L, N, PP)


def test_p_part_resplit_validation_and_workspace():
    """kv_split = -P: accepted when the P equal-pair boundaries are strictly
    increasing; the forward workspace grows by one partial block per part."""
    s = shape()                                                 # B1 H2 T1024 D64
    base = cca.attn_workspace_size(s, [(0, 1024, 0, 0)], 0)
    w2 = cca.attn_workspace_size(s, [(0, 1024, 0, -2)], 0)
    w4 = cca.attn_workspace_size(s, [(0, 1024, 0, -4)], 0)
    assert base < w2 < w4
    for bad in ([(0, 200, 0, -4)], [(0, 1024, 0, -1)], [(0, 1024, 0, -65)]):
        with pytest.raises(cca.AttnError) as e:
            cca.attn_workspace_size(s, bad, 0)
        assert e.value.status == 1
    # the backward ignores kv_split but validates it like the forward
    assert cca.attn_workspace_size(s, [(0, 1024, 0, -4)], 1) > 0


def test_tensor_layout_check():
    """The binding checks every tensor against the attn_shape before a call:
    the C ABI takes one set of strides and raw pointers, so a tensor with
    another layout would be read or written at the shape's offsets."""
    import torch
    from chunked_causal_attention_gb300._lib import _layout_ok
    x = torch.zeros(2, 3, 50, 64)
    s = cca.shape_of(x)
    assert _layout_ok(x, s.B, s.H, s.T, s.D, s.sb, s.st, s.sh)
    tm = torch.zeros(2, 50, 3, 64).permute(0, 2, 1, 3)                 # token-major storage
    s = cca.shape_of(tm)
    assert _layout_ok(tm, s.B, s.H, s.T, s.D, s.sb, s.st, s.sh)
    assert not _layout_ok(x, s.B, s.H, s.T, s.D, s.sb, s.st, s.sh)      # same sizes, other strides
    wide = torch.zeros(2, 3, 50, 128)[..., :80]                          # first 80 dims of a wider buffer
    s = cca.shape_of(wide)
    assert (s.D, s.st) == (80, 128) and _layout_ok(wide, s.B, s.H, s.T, s.D, s.sb, s.st, s.sh)
    assert not _layout_ok(torch.zeros(2, 3, 50, 80), s.B, s.H, s.T, s.D, s.sb, s.st, s.sh)
    p = torch.zeros(70, 4, 32)                                           # packed [T, H, D]
    s = cca.shape_of(p, packed=True)
    assert _layout_ok(p, s.B, s.H, s.T, s.D, s.sb, s.st, s.sh)
    assert not _layout_ok(p[:69], s.B, s.H, s.T, s.D, s.sb, s.st, s.sh)


def test_compute_wrappers_reject_cpu_and_mismatched_tensors():
    """Rejected on the host with ATTN_E_INVAL before the library is called."""
    import torch
    q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16)
    s = cca.shape_of(q)
    ch = cca.attn_plan(256, 1, 0)
    lse = torch.zeros(1, 2, 256)
    ws = torch.zeros(1, dtype=torch.uint8)
    with pytest.raises(cca.AttnError) as e:
        cca.attn_fwd(q, q, q, ch, s, q, lse, ws)                        # host tensors
    assert e.value.status == 1
    with pytest.raises(cca.AttnError) as e:
        cca.attn_bwd_chunk(q, q, q, q, lse, q, ch, s, q, q, q, q.float(), q.float(), ws)
    assert e.value.status == 1


def test_header_is_plain_c(tmp_path):
    """include/attn.h is a C header: a C99 program that includes it, links
    libattn.so and calls the host-only entry points (planner, workspace size,
    error strings, version) compiles and gives the same plan as the binding;
    its compute calls without buffers return ATTN_E_INVAL from the host."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(ROOT, "include")
    src = tmp_path / "use_attn.c"
    src.write_text(r'''
#include <stdio.h>
#include "attn.h"
int main(void) {
    attn_chunk c[16];
    int32_t n = 0;
    if (attn_plan(131072, 16, ATTN_PLAN_FLOPS_RESPLIT_EDGES, c, 16, &n) != ATTN_OK) return 1;
    attn_shape s = {1, 32, 131072, 128, 32LL * 131072 * 128, 128, 131072LL * 128, 0.08838834764831845f, 0, 0, 0, 0};
    size_t bytes = 0;
    if (attn_workspace_size(&s, c, n, 1, &bytes) != ATTN_OK || bytes == 0) return 2;
    /* compute calls with missing buffers are refused on the host, before any CUDA call */
    if (attn_fwd(NULL, NULL, NULL, c, n, &s, NULL, NULL, NULL, 0, NULL) != ATTN_E_INVAL) return 4;
    if (attn_bwd(NULL, NULL, NULL, NULL, NULL, NULL, c, n, &s, NULL, NULL, NULL, NULL, 0, NULL) != ATTN_E_INVAL)
        return 5;
    s.D = 100;
    if (attn_workspace_size(&s, c, n, 1, &bytes) != ATTN_E_UNSUPPORTED) return 3;
    printf("%d", (int)n);
    for (int32_t i = 0; i < n; ++i) printf(" %d,%d,%d,%d", c[i].q_begin, c[i].q_end, c[i].ctx_begin, c[i].kv_split);
    printf("\n%s\n%s\n", attn_strerror(ATTN_E_UNSUPPORTED), attn_version());
    return 0;
}
''')
    exe = tmp_path / "use_attn"
    libdir = os.path.dirname(_lib.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-L", libdir, "-lattn",
                        f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    lines = out.stdout.splitlines()
    fields = lines[0].split()
    got = [tuple(int(x) for x in f.split(",")) for f in fields[1:]]
    assert int(fields[0]) == len(got) == 16
    assert got == cca.attn_plan(131072, 16, cca.PLAN_FLOPS_RESPLIT_EDGES)
    assert lines[1] == cca.strerror(3) and lines[2]
