"""ctypes binding over libattn.so (the C-ABI in include/attn.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the launch stream, and non-zero status codes become
``AttnError``.  Every step of the computation runs in the library's kernels.
The library is loaded on first use; if it is missing or cannot be loaded the
call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

ATTN_F16 = 0
ATTN_BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libattn.so"
_lock = threading.Lock()
_lib = None

# The symbols include/attn.h declares (checked by the CPU test-suite).
EXPORTS = (
    "attn_fwd",
    "attn_fwd_visited",
    "attn_fwd_noalloc",
    "attn_fwd_ex",
    "attn_check",
    "attn_release_workspace",
    "attn_debug_counters",
    "attn_strerror",
    "attn_tile_shape",
    "attn_set_wait_timeout_ns",
    "attn_debug_inject",
    "attn_version",
)


class FwdParams(ctypes.Structure):
    """attn_fwd_params_t of include/attn.h."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("o", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("mask_bits", ctypes.c_void_p), ("mask_per_head", ctypes.c_int),
                ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("Sq", ctypes.c_int),
                ("Sk", ctypes.c_int), ("d", ctypes.c_int), ("causal", ctypes.c_int), ("window_left", ctypes.c_int),
                ("window_right", ctypes.c_int), ("scale", ctypes.c_float), ("dtype", ctypes.c_int),
                ("stream", ctypes.c_void_p), ("visited", ctypes.c_void_p), ("seqlens_q", ctypes.c_void_p),
                ("seqlens_k", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
                ("max_seqlen_q", ctypes.c_int), ("max_seqlen_k", ctypes.c_int)]


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_strerror(status)} ({status})")


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def library():
    """Load libattn.so (built in-tree by __graft_entry__.build()); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fwd_args = [p, p, p, p, p, p, i, i, i, i, i, i, f, i, p]
        lib.attn_fwd.argtypes = fwd_args
        lib.attn_fwd.restype = i
        lib.attn_fwd_visited.argtypes = fwd_args + [p]
        lib.attn_fwd_visited.restype = i
        lib.attn_fwd_noalloc.argtypes = fwd_args
        lib.attn_fwd_noalloc.restype = i
        lib.attn_fwd_ex.argtypes = [ctypes.POINTER(FwdParams)]
        lib.attn_fwd_ex.restype = i
        lib.attn_check.argtypes = [p]
        lib.attn_check.restype = i
        lib.attn_release_workspace.argtypes = [p]
        lib.attn_release_workspace.restype = i
        lib.attn_debug_counters.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i]
        lib.attn_debug_counters.restype = i
        lib.attn_strerror.argtypes = [i]
        lib.attn_strerror.restype = ctypes.c_char_p
        lib.attn_tile_shape.argtypes = [i, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.attn_tile_shape.restype = i
        lib.attn_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        lib.attn_set_wait_timeout_ns.restype = i
        lib.attn_debug_inject.argtypes = [i]
        lib.attn_debug_inject.restype = i
        lib.attn_version.argtypes = []
        lib.attn_version.restype = i
        _lib = lib
        return lib


def attn_strerror(status: int) -> str:
    return library().attn_strerror(int(status)).decode()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; fp16 or bf16 expected")


def _lens_ptr(t, B):
    import torch
    if t.dtype != torch.int32 or t.numel() != B or not t.is_contiguous():
        raise ValueError("sequence lengths must be a contiguous int32 tensor of B entries")
    return t.data_ptr()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _call(fn, q, k, v, o, lse, mask_bits, causal, scale, stream, extra=()):
    """q/o: [B,Hq,S,d]; k/v: [B,Hkv,S,d]; lse: fp32 [B,Hq,S] or None;
    mask_bits: int32/uint32 [B,S,ceil(S/32)] or None.  Shapes are taken from q and k."""
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(mask_bits), int(B), int(Hq), int(Hkv),
            int(S), int(d), int(bool(causal)), ctypes.c_float(scale), _dtype_code(q), _stream_handle(stream),
            *extra)
    if rc != 0:
        raise AttnError(rc, fn.__name__)


def attn_fwd(q, k, v, o, lse=None, mask_bits=None, causal=False, scale=None, stream=None):
    """Launch the fused forward on `stream` (default: torch's current stream).

    The caller owns every tensor (device memory, contiguous, [B,H,S,d]); the
    call is asynchronous; use attn_check() to collect in-kernel errors."""
    lib = library()
    _call(lib.attn_fwd, q, k, v, o, lse, mask_bits, causal, scale, stream)


def attn_fwd_visited(q, k, v, o, lse, mask_bits, causal, scale, visited, stream=None):
    """attn_fwd that also sets visited[b, hq, qtile, ktile] = 1 (uint8) for every
    (query tile, key tile) block the kernel computed; the caller zeroes it first."""
    lib = library()
    _call(lib.attn_fwd_visited, q, k, v, o, lse, mask_bits, causal, scale, stream, extra=(_ptr(visited),))


def attn_fwd_noalloc(q, k, v, o, lse=None, mask_bits=None, causal=False, scale=None, stream=None):
    """attn_fwd for callers that may not allocate device memory: a custom mask's
    pre-pass output goes into a fixed array the library reserves per GPU (see
    include/attn.h for the size limit and the rules on sharing it)."""
    lib = library()
    _call(lib.attn_fwd_noalloc, q, k, v, o, lse, mask_bits, causal, scale, stream)


def attn_fwd_ex(q, k, v, o, lse=None, mask_bits=None, mask_per_head=False, causal=False, window_left=-1,
                window_right=-1, scale=None, visited=None, stream=None, seqlens_q=None, seqlens_k=None):
    """Generalised forward: q/o [B,Hq,Sq,d], k/v [B,Hkv,Sk,d] with Sk >= Sq (bottom-right
    aligned), a band of kept keys (window_left / window_right, -1 = unbounded), custom masks
    [B,Sq,ceil(Sk/32)] or per head [B,Hq,Sq,ceil(Sk/32)], per-entry lengths seqlens_q /
    seqlens_k (int32 device tensors [B]); see include/attn.h."""
    B, Hq, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    prm = FwdParams(q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(), o=o.data_ptr(),
                    lse=None if lse is None else lse.data_ptr(),
                    mask_bits=None if mask_bits is None else mask_bits.data_ptr(),
                    mask_per_head=int(bool(mask_per_head)), B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=d,
                    causal=int(bool(causal)), window_left=int(window_left), window_right=int(window_right),
                    scale=float(scale), dtype=_dtype_code(q), stream=_stream_handle(stream).value,
                    visited=None if visited is None else visited.data_ptr(),
                    seqlens_q=None if seqlens_q is None else _lens_ptr(seqlens_q, B),
                    seqlens_k=None if seqlens_k is None else _lens_ptr(seqlens_k, B))
    rc = library().attn_fwd_ex(ctypes.byref(prm))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_ex")


def attn_fwd_packed(q, k, v, o, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, lse=None, causal=False,
                    window_left=-1, window_right=-1, scale=None, visited=None, stream=None):
    """attn_fwd_ex over packed variable-length batches: q/o [Hq, total_q, d], k/v [Hkv, total_k, d],
    lse [Hq, total_q]; cu_seqlens_q / cu_seqlens_k int32 device tensors [B+1] of row offsets;
    max_seqlen_q / max_seqlen_k bound the entries' lengths.  See include/attn.h."""
    Hq, Sq, d = q.shape
    Hkv, Sk = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    prm = FwdParams(q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(), o=o.data_ptr(),
                    lse=None if lse is None else lse.data_ptr(), mask_bits=None, mask_per_head=0,
                    B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=d, causal=int(bool(causal)),
                    window_left=int(window_left), window_right=int(window_right), scale=float(scale),
                    dtype=_dtype_code(q), stream=_stream_handle(stream).value,
                    visited=None if visited is None else visited.data_ptr(),
                    cu_seqlens_q=_lens_ptr(cu_seqlens_q, B + 1), cu_seqlens_k=_lens_ptr(cu_seqlens_k, B + 1),
                    max_seqlen_q=int(max_seqlen_q), max_seqlen_k=int(max_seqlen_k))
    rc = library().attn_fwd_ex(ctypes.byref(prm))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_ex")


def attn_check(stream=None) -> int:
    """Synchronise `stream` and return the library status (0 = OK); raises on error."""
    rc = library().attn_check(_stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_check")
    return rc


def attn_release_workspace(stream=None) -> None:
    """Free the custom-mask workspace the library holds for `stream` (stream-ordered)."""
    rc = library().attn_release_workspace(_stream_handle(stream))
    if rc != 0:
        raise AttnError(rc, "attn_release_workspace")


def debug_counters() -> dict:
    """Host-side counters: workspace allocations, tensor maps encoded, tensor-map cache hits."""
    out = (ctypes.c_ulonglong * 3)()
    rc = library().attn_debug_counters(out, 3)
    if rc != 0:
        raise AttnError(rc, "attn_debug_counters")
    return {"workspace_allocs": out[0], "map_encodes": out[1], "map_hits": out[2]}


def attn_tile_shape(d: int):
    """(rows per query tile, columns per key tile) the kernel uses for head dim d."""
    bm, bn = ctypes.c_int(0), ctypes.c_int(0)
    rc = library().attn_tile_shape(int(d), ctypes.byref(bm), ctypes.byref(bn))
    if rc != 0:
        raise AttnError(rc, "attn_tile_shape")
    return bm.value, bn.value
