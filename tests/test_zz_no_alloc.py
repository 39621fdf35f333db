"""attn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Those callers (code hosted by a runtime that owns all device memory and
exposes no allocator, or code that must not allocate once it is running)
cannot provide the workspace that attn_fwd needs. attn_fwd_noalloc uses
scratch memory that lives inside the library instead. This file checks it,
through the C ABI, against attn_fwd on the same inputs, for two calls in a
row with different shapes and plans (the second call must not be disturbed by
what the first left in the shared scratch), and checks that a request larger
than the scratch is refused. pytest collects this file last.
"""
import ctypes

import pytest
import torch

import chunked_causal_attention_gb300 as cca
from chunked_causal_attention_gb300 import _lib
from chunked_causal_attention_gb300.workloads import make_inputs
from oracle import plan as P

from parity import LSE_ABS, O_MAX_ABS

pytestmark = pytest.mark.gpu


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


def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row():
    cases = [
        (1, 4, 4096, 128, P.plan(4096, 3, P.FLOPS_RESPLIT_EDGES), 901),   # re-split: uses the partial area
        (2, 3, 1000, 64, P.plan(1000, 2, P.UNIFORM), 902),
    ]
    for B, H, L, D, chunks, seed in cases:
        q, k, v, _ = (x.cuda() for x in make_inputs(B, H, L, D, seed=seed))
        shape = cca.shape_of(q)
        assert cca.attn_workspace_size(shape, chunks, 0) <= _lib.NOALLOC_SCRATCH_BYTES
        o_ref, lse_ref = cca.forward(q, k, v, chunks)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, L), float("nan"), device="cuda")
        st = call_noalloc(q, k, v, chunks, shape, o, lse)
        assert st == 0, cca.strerror(st)
        torch.cuda.synchronize()
        assert (o.float() - o_ref.float()).abs().max().item() <= O_MAX_ABS
        assert (lse - lse_ref).abs().max().item() <= LSE_ABS


def test_noalloc_refuses_requests_beyond_its_scratch():
    B, H, L, D = 1, 32, 32768, 128
    chunks = P.plan(L, 8, P.FLOPS_RESPLIT_EDGES)              # the partials need ~1 GB
    shape = cca.make_shape(B, H, L, D, H * L * D, D, L * D, D ** -0.5)
    assert cca.attn_workspace_size(shape, chunks, 0) > _lib.NOALLOC_SCRATCH_BYTES
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never read: refused on the host
    st = call_noalloc(q, q, q, chunks, shape, q, q)
    assert st == 4, cca.strerror(st)                            # ATTN_E_WORKSPACE
