"""Child process of tests/test_zz_no_alloc.py::test_noalloc_after_a_device_reset.

Runs attn_fwd_noalloc, resets the device (cudaDeviceReset through the CUDA
runtime library, as a caller would), allocates fresh buffers and runs the
same problem again; prints the two calls' status codes and whether their
outputs are equal. It uses no torch, so that no framework holds device
memory across the reset. Device memory is allocated and copied with the
runtime's own calls; inputs are seeded N(0, 1) rounded to bf16."""
import ctypes
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), ".."))
from chunked_causal_attention_gb300 import _lib  # noqa: E402

H2D, D2H = 1, 2


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even."""
    u = x.astype(np.float32).view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def main():
    rt = ctypes.CDLL(sys.argv[1])
    rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
    rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    rt.cudaFree.argtypes = [ctypes.c_void_p]
    L = _lib.lib()
    B, H, T, D = 1, 4, 2048, 128
    chunks = _lib.attn_plan(T, 2, _lib.PLAN_FLOPS_RESPLIT_EDGES)   # edge re-splits: partials and a merge
    assert all(c[3] > 0 for c in chunks)
    rng = np.random.default_rng(5)
    host = [bf16_bits(rng.standard_normal((B, H, T, D)).astype(np.float32)) for _ in range(3)]
    shape = _lib.make_shape(B, H, T, D, H * T * D, D, T * D, 1.0 / np.sqrt(D))
    arr, n = _lib.chunk_array(chunks)
    results = []
    for call in range(2):
        ptrs = []
        for x in host + [np.zeros_like(host[0]), np.zeros((B, H, T), np.float32)]:
            p = ctypes.c_void_p()
            assert rt.cudaMalloc(ctypes.byref(p), x.nbytes) == 0
            assert rt.cudaMemcpy(p, x.ctypes.data, x.nbytes, H2D) == 0
            ptrs.append(p)
        q, k, v, o, lse = ptrs
        st = L.attn_fwd_noalloc(q, k, v, arr, n, ctypes.byref(shape), o, lse, None)
        st2 = L.attn_noalloc_status(None)
        out_o = np.zeros_like(host[0])
        out_l = np.zeros((B, H, T), np.float32)
        assert rt.cudaMemcpy(out_o.ctypes.data, o, out_o.nbytes, D2H) == 0
        assert rt.cudaMemcpy(out_l.ctypes.data, lse, out_l.nbytes, D2H) == 0
        results.append((st, st2, out_o, out_l))
        for p in ptrs:
            rt.cudaFree(p)
        if call == 0:
            assert rt.cudaDeviceReset() == 0
    (s0, t0, o0, l0), (s1, t1, o1, l1) = results
    print(f"status {s0} {t0} {s1} {t1}")
    print(f"equal {int(np.array_equal(o0, o1) and np.array_equal(l0, l1))}")
    print(f"finite {int(np.isfinite(l0).all())}")


if __name__ == "__main__":
    main()
