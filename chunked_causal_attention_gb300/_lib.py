"""ctypes binding of libattn (include/attn.h): argument marshalling only.

Every function here converts Python/torch arguments to the C ABI's plain
pointers and sizes and calls the entry point of the same name. All compute
runs in the library's CUDA kernels; there is no Python or CPU fallback: if
libattn.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_OK = 0
ATTN_E_INVAL = 1
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_E_INVAL", 2: "ATTN_E_ALIGN", 3: "ATTN_E_UNSUPPORTED",
                4: "ATTN_E_WORKSPACE", 5: "ATTN_E_CUDA", 6: "ATTN_E_TIMEOUT", 7: "ATTN_E_BOUNDS",
                8: "ATTN_E_CAPACITY"}

PLAN_UNIFORM = 0
PLAN_FLOPS = 1
PLAN_FLOPS_RESPLIT_EDGES = 2

# Every symbol include/attn.h declares.
EXPORTS = ("attn_plan", "attn_plan_varlen", "attn_plan_multiplex", "attn_plan_infinipipe", "attn_workspace_size", "attn_fwd", "attn_fwd_tiles",
           "attn_fwd_merge", "attn_bwd", "attn_bwd_prep", "attn_bwd_tiles", "attn_bwd_dq",
           "attn_bwd_chunk", "attn_fwd_noalloc", "attn_noalloc_status", "attn_status", "attn_strerror",
           "attn_version", "attn_kernel_launches")

# attn_workspace_size passes
PASS_FWD = 0
PASS_BWD = 1
PASS_BWD_CHUNK = 2

# Size of the library-held scratch area of attn_fwd_noalloc (ATTN_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 64 << 20


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({strerror(status)})")


class attn_chunk(ctypes.Structure):
    _fields_ = [("q_begin", ctypes.c_int32), ("q_end", ctypes.c_int32),
                ("ctx_begin", ctypes.c_int32), ("kv_split", ctypes.c_int32)]


class attn_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64), ("D", ctypes.c_int64),
                ("sb", ctypes.c_int64), ("st", ctypes.c_int64), ("sh", ctypes.c_int64),
                ("scale", ctypes.c_float),
                ("Hkv", ctypes.c_int64), ("sb_kv", ctypes.c_int64), ("st_kv", ctypes.c_int64), ("sh_kv", ctypes.c_int64)]


_lib: Optional[ctypes.CDLL] = None

_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_CP = ctypes.POINTER(attn_chunk)
_SP = ctypes.POINTER(attn_shape)
_SIG = {
    "attn_plan": ([_I64, _I32, _I32, _CP, _I32, ctypes.POINTER(_I32)], ctypes.c_int),
    "attn_plan_varlen": ([ctypes.POINTER(_I64), _I32, _I32, _I32, _CP, _I32, ctypes.POINTER(_I32)], ctypes.c_int),
    "attn_plan_multiplex": ([_I64, _I32, _I32, _CP, _I32, ctypes.POINTER(_I32)], ctypes.c_int),
    "attn_plan_infinipipe": ([ctypes.POINTER(_I64), _I32, _I32, _I64, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                              _CP, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32), _I32, ctypes.POINTER(_I32)],
                             ctypes.c_int),
    "attn_workspace_size": ([_SP, _CP, _I32, _I32, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "attn_fwd": ([_VP, _VP, _VP, _CP, _I32, _SP, _VP, _VP, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "attn_fwd_tiles": ([_VP, _VP, _VP, _CP, _I32, _SP, _VP, _VP, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "attn_fwd_merge": ([_CP, _I32, _SP, _VP, _VP, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "attn_bwd": ([_VP, _VP, _VP, _VP, _VP, _VP, _CP, _I32, _SP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP],
                 ctypes.c_int),
    "attn_bwd_prep": ([_VP, _VP, _CP, _I32, _SP, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "attn_bwd_tiles": ([_VP, _VP, _VP, _VP, _VP, _CP, _I32, _SP, _VP, _VP, _VP, ctypes.c_size_t, _VP],
                       ctypes.c_int),
    "attn_bwd_dq": ([_CP, _I32, _SP, _VP, _VP, ctypes.c_size_t, _VP], ctypes.c_int),
    "attn_bwd_chunk": ([_VP, _VP, _VP, _VP, _VP, _VP, _CP, _I32, _SP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t,
                        _VP], ctypes.c_int),
    "attn_fwd_noalloc": ([_VP, _VP, _VP, _CP, _I32, _SP, _VP, _VP, _VP], ctypes.c_int),
    "attn_noalloc_status": ([_VP], ctypes.c_int),
    "attn_status": ([_VP, _VP], ctypes.c_int),
    "attn_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "attn_version": ([], ctypes.c_char_p),
    "attn_kernel_launches": ([], ctypes.c_uint64),
}


def lib() -> ctypes.CDLL:
    """Load libattn.so (built in-tree by chunked_causal_attention_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libattn.so not built ({LIB_PATH}); run `python -m "
                               "chunked_causal_attention_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIG.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().attn_strerror(status).decode()


def version() -> str:
    return lib().attn_version().decode()


def kernel_launches() -> int:
    """Kernels the library has enqueued since it was loaded."""
    return int(lib().attn_kernel_launches())


def _check(fn: str, st: int) -> None:
    if st != ATTN_OK:
        raise AttnError(fn, st)


def chunk_array(chunks: Sequence[Sequence[int]]):
    arr = (attn_chunk * max(1, len(chunks)))()
    for i, c in enumerate(chunks):
        arr[i] = attn_chunk(*[int(x) for x in c])
    return arr, len(chunks)


# ------------------------------------------------------------------ planning

def attn_plan(L: int, N: int, mode: int) -> List[Tuple[int, int, int, int]]:
    out = (attn_chunk * max(1, N))()
    n = _I32(0)
    _check("attn_plan", lib().attn_plan(L, N, mode, out, N, ctypes.byref(n)))
    return [(c.q_begin, c.q_end, c.ctx_begin, c.kv_split) for c in out[:n.value]]


def attn_plan_multiplex(L: int, N: int, PP: int) -> List[Tuple[int, int, int, int]]:
    """FLOPS chunks with SPPO Table 3 edge re-splits for PP stages (kv_split = -P)."""
    out = (attn_chunk * max(1, N))()
    n = _I32(0)
    _check("attn_plan_multiplex", lib().attn_plan_multiplex(L, N, PP, out, N, ctypes.byref(n)))
    return [(c.q_begin, c.q_end, c.ctx_begin, c.kv_split) for c in out[:n.value]]


def attn_plan_varlen(cu_seqlens: Sequence[int], max_chunk_tokens: int, mode: int):
    nd = len(cu_seqlens) - 1
    cu = (_I64 * len(cu_seqlens))(*[int(x) for x in cu_seqlens])
    n = _I32(0)
    cap = 16
    while True:
        out = (attn_chunk * cap)()
        st = lib().attn_plan_varlen(cu, nd, max_chunk_tokens, mode, out, cap, ctypes.byref(n))
        if st == 8 and n.value > cap:       # ATTN_E_CAPACITY reports the needed count
            cap = n.value
            continue
        _check("attn_plan_varlen", st)
        return [(c.q_begin, c.q_end, c.ctx_begin, c.kv_split) for c in out[:n.value]]


def attn_plan_infinipipe(seq_lens: Sequence[int], K: int, token_cap: int, alpha1: float, alpha2: float,
                         beta1: float) -> List[List[Tuple[int, int, int, int]]]:
    """InfiniPipe Algorithm 1: a list of calls, each a list of chunks in the
    packed layout of ``seq_lens`` (see include/attn.h)."""
    lens = (_I64 * max(1, len(seq_lens)))(*[int(x) for x in seq_lens])
    n, nc = _I32(0), _I32(0)
    cap, ccap = 16, 16
    while True:
        out = (attn_chunk * cap)()
        off = (_I32 * ccap)()
        st = lib().attn_plan_infinipipe(lens, len(seq_lens), K, token_cap, alpha1, alpha2, beta1, out, cap,
                                        ctypes.byref(n), off, ccap, ctypes.byref(nc))
        if st == 8:                          # ATTN_E_CAPACITY reports the needed counts
            cap, ccap = max(cap, n.value), max(ccap, nc.value + 1)
            continue
        _check("attn_plan_infinipipe", st)
        return [[(c.q_begin, c.q_end, c.ctx_begin, c.kv_split) for c in out[off[i]:off[i + 1]]]
                for i in range(nc.value)]


# ------------------------------------------------------------------ shapes

def make_shape(B, H, T, D, sb, st, sh, scale, Hkv=0, sb_kv=0, st_kv=0, sh_kv=0) -> attn_shape:
    return attn_shape(B, H, T, D, sb, st, sh, float(scale), Hkv, sb_kv, st_kv, sh_kv)


def _bths(x, packed: bool):
    """(B, heads, T, sb, st, sh) of a dense [B, H, L, D] or packed [T, H, D] tensor."""
    if packed:
        T, H, _ = x.shape
        return 1, H, T, x.stride(0) * T, x.stride(0), x.stride(1)
    B, H, L, _ = x.shape
    return B, H, L, x.stride(0), x.stride(2), x.stride(1)


def shape_of(x, scale: Optional[float] = None, packed: bool = False, k=None) -> attn_shape:
    """attn_shape of a query tensor: dense [B, H, L, D] or packed [T, H, D].
    Given k with fewer heads than x (grouped key/value heads), the shape also
    carries k's head count and strides (used for k, v, dk, dv)."""
    D = x.shape[-1]
    sc = (1.0 / D ** 0.5) if scale is None else scale
    B, H, T, sb, st, sh = _bths(x, packed)
    if k is None or k.shape == x.shape and k.stride() == x.stride():
        return make_shape(B, H, T, D, sb, st, sh, sc)
    _, Hkv, _, sbk, stk, shk = _bths(k, packed)
    return make_shape(B, H, T, D, sb, st, sh, sc, Hkv, sbk, stk, shk)


def attn_workspace_size(shape: attn_shape, chunks, pass_: int) -> int:
    arr, n = chunk_array(chunks)
    out = ctypes.c_size_t(0)
    _check("attn_workspace_size", lib().attn_workspace_size(ctypes.byref(shape), arr, n, pass_, ctypes.byref(out)))
    return out.value


# ------------------------------------------------------------------ compute

def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _layout_ok(t, B: int, H: int, T: int, D: int, sb: int, st: int, sh: int) -> bool:
    """t addresses element (b, t, h, d) at b*sb + t*st + h*sh + d: a dense
    [B, H, T, D] view, or a packed [T, H, D] one when B == 1 (strides of size-1
    dims are free)."""
    if t.dim() == 4:
        want_size, want_stride = (B, H, T, D), (sb, sh, st, 1)
    elif t.dim() == 3 and B == 1:
        want_size, want_stride = (T, H, D), (st, sh, 1)
    else:
        return False
    if tuple(t.shape) != want_size:
        return False
    return all(n == 1 or got == want for n, got, want in zip(want_size, t.stride(), want_stride))


def _expect(fn: str, shape: attn_shape, kind: str, *tensors) -> None:
    """The C ABI takes one set of strides per kind of tensor and raw pointers,
    so it cannot see a tensor whose layout differs from the shape's; such a
    tensor would be read or written at the shape's offsets. Every tensor
    argument must therefore have the shape's sizes and strides: kind 'q'
    (q, o, dout, dq: bf16, query strides), 'kv' (k, v, dk, dv: bf16,
    key/value strides), 'acc' (fp32 dK/dV accumulators: key/value strides),
    'lse' (fp32 [B, H, T] contiguous). None is passed through (the library
    rejects null pointers itself). Raises AttnError(ATTN_E_INVAL)."""
    import torch
    grouped = kind in ("kv", "acc") and shape.Hkv > 0
    H = shape.Hkv if grouped else shape.H
    sb, st, sh = (shape.sb_kv, shape.st_kv, shape.sh_kv) if grouped else (shape.sb, shape.st, shape.sh)
    for t in tensors:
        if t is None:
            continue
        if kind == "lse":
            ok = (t.dtype == torch.float32 and t.is_cuda and t.is_contiguous()
                  and t.numel() == shape.B * shape.H * shape.T)
        else:
            dt = torch.float32 if kind == "acc" else torch.bfloat16
            ok = t.dtype == dt and t.is_cuda and _layout_ok(t, shape.B, H, shape.T, shape.D, sb, st, sh)
        if not ok:
            raise AttnError(fn, ATTN_E_INVAL)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def attn_fwd(q, k, v, chunks, shape, o, lse, ws, stream=None) -> None:
    _expect("attn_fwd", shape, "q", q, o)
    _expect("attn_fwd", shape, "kv", k, v)
    _expect("attn_fwd", shape, "lse", lse)
    arr, n = chunk_array(chunks)
    _check("attn_fwd", lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), arr, n, ctypes.byref(shape), _ptr(o), _ptr(lse),
                                      _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def attn_fwd_tiles(q, k, v, chunks, shape, o, lse, ws, stream=None) -> None:
    _expect("attn_fwd_tiles", shape, "q", q, o)
    _expect("attn_fwd_tiles", shape, "kv", k, v)
    _expect("attn_fwd_tiles", shape, "lse", lse)
    arr, n = chunk_array(chunks)
    _check("attn_fwd_tiles", lib().attn_fwd_tiles(_ptr(q), _ptr(k), _ptr(v), arr, n, ctypes.byref(shape), _ptr(o),
                                                  _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(),
                                                  _stream(stream)))


def attn_fwd_merge(chunks, shape, o, lse, ws, stream=None) -> None:
    _expect("attn_fwd_merge", shape, "q", o)
    _expect("attn_fwd_merge", shape, "lse", lse)
    arr, n = chunk_array(chunks)
    _check("attn_fwd_merge", lib().attn_fwd_merge(arr, n, ctypes.byref(shape), _ptr(o), _ptr(lse), _ptr(ws),
                                                  ws.numel() * ws.element_size(), _stream(stream)))


def attn_bwd(q, k, v, o, lse, dout, chunks, shape, dq, dk, dv, ws, stream=None) -> None:
    _expect("attn_bwd", shape, "q", q, o, dout, dq)
    _expect("attn_bwd", shape, "kv", k, v, dk, dv)
    _expect("attn_bwd", shape, "lse", lse)
    arr, n = chunk_array(chunks)
    _check("attn_bwd", lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), arr, n,
                                      ctypes.byref(shape), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)))


def attn_bwd_prep(o, dout, chunks, shape, ws, stream=None) -> None:
    _expect("attn_bwd_prep", shape, "q", o, dout)
    arr, n = chunk_array(chunks)
    _check("attn_bwd_prep", lib().attn_bwd_prep(_ptr(o), _ptr(dout), arr, n, ctypes.byref(shape), _ptr(ws),
                                                ws.numel() * ws.element_size(), _stream(stream)))


def attn_bwd_tiles(q, k, v, lse, dout, chunks, shape, dk, dv, ws, stream=None) -> None:
    _expect("attn_bwd_tiles", shape, "q", q, dout)
    _expect("attn_bwd_tiles", shape, "kv", k, v, dk, dv)
    _expect("attn_bwd_tiles", shape, "lse", lse)
    arr, n = chunk_array(chunks)
    _check("attn_bwd_tiles", lib().attn_bwd_tiles(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(dout), arr, n,
                                                  ctypes.byref(shape), _ptr(dk), _ptr(dv), _ptr(ws),
                                                  ws.numel() * ws.element_size(), _stream(stream)))


def attn_bwd_dq(chunks, shape, dq, ws, stream=None) -> None:
    _expect("attn_bwd_dq", shape, "q", dq)
    arr, n = chunk_array(chunks)
    _check("attn_bwd_dq", lib().attn_bwd_dq(arr, n, ctypes.byref(shape), _ptr(dq), _ptr(ws),
                                            ws.numel() * ws.element_size(), _stream(stream)))


def attn_bwd_chunk(q, k, v, o, lse, dout, chunks, shape, dq, dk, dv, dk_acc, dv_acc, ws, stream=None) -> None:
    """Backward of the rows of a set of chunks (chunk-streamed; see include/attn.h)."""
    _expect("attn_bwd_chunk", shape, "q", q, o, dout, dq)
    _expect("attn_bwd_chunk", shape, "kv", k, v, dk, dv)
    _expect("attn_bwd_chunk", shape, "acc", dk_acc, dv_acc)
    _expect("attn_bwd_chunk", shape, "lse", lse)
    arr, n = chunk_array(chunks)
    _check("attn_bwd_chunk", lib().attn_bwd_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), arr, n,
                                                  ctypes.byref(shape), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dk_acc),
                                                  _ptr(dv_acc), _ptr(ws), ws.numel() * ws.element_size(),
                                                  _stream(stream)))


def attn_fwd_noalloc(q, k, v, chunks, shape, o, lse, stream=None) -> None:
    """Forward without a workspace argument: for callers that cannot allocate
    device memory; uses the library's own scratch (see include/attn.h)."""
    _expect("attn_fwd_noalloc", shape, "q", q, o)
    _expect("attn_fwd_noalloc", shape, "kv", k, v)
    _expect("attn_fwd_noalloc", shape, "lse", lse)
    arr, n = chunk_array(chunks)
    _check("attn_fwd_noalloc", lib().attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), arr, n, ctypes.byref(shape),
                                                      _ptr(o), _ptr(lse), _stream(stream)))


def attn_status(ws, stream=None) -> int:
    return lib().attn_status(_ptr(ws), _stream(stream))


def attn_noalloc_status(stream=None) -> int:
    """Device error word of attn_fwd_noalloc (synchronises the stream; read clears it)."""
    return lib().attn_noalloc_status(_stream(stream))
