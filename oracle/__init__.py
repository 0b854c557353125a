"""fp64 CPU oracle for masked attention forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library path never does, and the
two implementations share no code: this package wraps ``attn_oracle.c``
(plain C, double precision) through ctypes.

What the oracle computes and which passages of the pages it follows is stated
in the header of ``attn_oracle.c``.  Every function here takes host numpy
arrays:

* ``q``, ``k``, ``v``: ``uint16`` views of fp16 / bf16 words, shaped
  ``[B, H, S, d]``;
* ``mask_bits``: ``uint32`` ``[B, S, ceil(S/32)]`` or ``None``.

Parity pins: see ``tests/test_oracle_pins.py`` (brute force against library
routines, closed forms and invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p = ctypes.c_void_p
            i = ctypes.c_int
            i64 = ctypes.c_int64
            d = ctypes.c_double
            lib.oracle_attn_rows.argtypes = [p, p, p, i, p, i, i, i, i, i, i, d, p, i64, p, p, i]
            lib.oracle_attn_rows.restype = i
            lib.oracle_attn_fwd.argtypes = [p, p, p, i, p, i, i, i, i, i, i, d, p, p, i]
            lib.oracle_attn_fwd.restype = i
            lib.oracle_skip_map.argtypes = [p, i, i, i, i, i, p]
            lib.oracle_skip_map.restype = i
            lib.oracle_attn_rows_ex.argtypes = [p, p, p, i, p, i, i, i, i, i, i, i, i, i, i, p, p, d, p, i64, p, p, i]
            lib.oracle_attn_rows_ex.restype = i
            lib.oracle_skip_map_ex.argtypes = [p, i, i, i, i, i, i, i, i, p, p, i, i, p]
            lib.oracle_skip_map_ex.restype = i
            lib.oracle_widen.argtypes = [ctypes.c_uint16, i]
            lib.oracle_widen.restype = d
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check_inputs(q, k, v, mask_bits):
    for name, a in (("q", q), ("k", k), ("v", v)):
        if a.dtype != np.uint16 or a.ndim != 4 or not a.flags.c_contiguous:
            raise ValueError(f"{name} must be a C-contiguous uint16 [B,H,S,d] array")
    B, Hq, S, d = q.shape
    Bk, Hkv, Sk, dk = k.shape
    if (Bk, Sk, dk) != (B, S, d) or v.shape != k.shape:
        raise ValueError("q/k/v shapes disagree")
    if mask_bits is not None:
        W = (S + 31) // 32
        if mask_bits.dtype != np.uint32 or mask_bits.shape != (B, S, W) or not mask_bits.flags.c_contiguous:
            raise ValueError("mask_bits must be C-contiguous uint32 [B,S,ceil(S/32)]")
    return B, Hq, Hkv, S, d


def attn_fwd(q, k, v, dtype, mask_bits=None, causal=False, scale=None, nthreads=0):
    """Every row of O (float64 [B,Hq,S,d]) and LSE (float64 [B,Hq,S])."""
    B, Hq, Hkv, S, d = _check_inputs(q, k, v, mask_bits)
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    o = np.empty((B, Hq, S, d), np.float64)
    lse = np.empty((B, Hq, S), np.float64)
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), int(dtype), _ptr(mask_bits), B, Hq, Hkv, S, d,
                                 int(bool(causal)), float(scale), _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    return o, lse


def attn_rows(q, k, v, dtype, rows, mask_bits=None, causal=False, scale=None, nthreads=0):
    """Selected rows: ``rows`` are flat ids (b*Hq + hq)*S + i.  Returns O [n,d], LSE [n]."""
    B, Hq, Hkv, S, d = _check_inputs(q, k, v, mask_bits)
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_attn_rows(_ptr(q), _ptr(k), _ptr(v), int(dtype), _ptr(mask_bits), B, Hq, Hkv, S, d,
                                  int(bool(causal)), float(scale), _ptr(rows), n, _ptr(o), _ptr(lse),
                                  int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed ({rc})")
    return o, lse


def skip_map(mask_bits, B, S, causal, bm, bn):
    """uint8 [B, ceil(S/bm), ceil(S/bn)]: 1 where the block holds a kept entry."""
    if mask_bits is not None:
        mask_bits = np.ascontiguousarray(mask_bits, dtype=np.uint32)
    nqt, nkt = (S + bm - 1) // bm, (S + bn - 1) // bn
    out = np.zeros((B, nqt, nkt), np.uint8)
    rc = _load().oracle_skip_map(_ptr(mask_bits), B, S, int(bool(causal)), bm, bn, _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_skip_map failed ({rc})")
    return out


def _lens(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.int32)


def attn_rows_ex(q, k, v, dtype, rows=None, mask_bits=None, mask_per_head=False, causal=False,
                 window_left=-1, window_right=-1, scale=None, nthreads=0, seqlens_q=None, seqlens_k=None):
    """Extended definition (see attn_oracle.c): q [B,Hq,Sq,d], k/v [B,Hkv,Sk,d] with Sq <= Sk,
    bottom-right aligned; optional key band; masks [B,Sq,W] or per head [B,Hq,Sq,W].
    rows=None evaluates every row and returns O [B,Hq,Sq,d], LSE [B,Hq,Sq].  seqlens_q / seqlens_k
    (int [B]) give each batch entry its own lengths; rows past them come back as NaN."""
    for name, a in (("q", q), ("k", k), ("v", v)):
        if a.dtype != np.uint16 or a.ndim != 4 or not a.flags.c_contiguous:
            raise ValueError(f"{name} must be a C-contiguous uint16 [B,H,S,d] array")
    B, Hq, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if mask_bits is not None:
        mask_bits = np.ascontiguousarray(mask_bits, dtype=np.uint32)
        want = (B, Hq, Sq, (Sk + 31) // 32) if mask_per_head else (B, Sq, (Sk + 31) // 32)
        if mask_bits.shape != want:
            raise ValueError(f"mask_bits shape {mask_bits.shape}, expected {want}")
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    full = rows is None
    if full:
        rows = np.arange(B * Hq * Sq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    lq, lk = _lens(seqlens_q), _lens(seqlens_k)
    rc = _load().oracle_attn_rows_ex(_ptr(q), _ptr(k), _ptr(v), int(dtype), _ptr(mask_bits), int(bool(mask_per_head)),
                                     B, Hq, Hkv, Sq, Sk, d, int(bool(causal)), int(window_left), int(window_right),
                                     _ptr(lq), _ptr(lk), float(scale), _ptr(rows), n, _ptr(o), _ptr(lse),
                                     int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows_ex failed ({rc})")
    if full:
        return o.reshape(B, Hq, Sq, d), lse.reshape(B, Hq, Sq)
    return o, lse


def skip_map_ex(mask_bits, mask_per_head, B, Hq, Sq, Sk, causal, window_left, window_right, bm, bn,
                seqlens_q=None, seqlens_k=None):
    """uint8 [B*Hm, ceil(Sq/bm), ceil(Sk/bn)], Hm = Hq for per-head masks else 1."""
    if mask_bits is not None:
        mask_bits = np.ascontiguousarray(mask_bits, dtype=np.uint32)
    Hm = Hq if (mask_bits is not None and mask_per_head) else 1
    out = np.zeros((B * Hm, (Sq + bm - 1) // bm, (Sk + bn - 1) // bn), np.uint8)
    lq, lk = _lens(seqlens_q), _lens(seqlens_k)
    rc = _load().oracle_skip_map_ex(_ptr(mask_bits), int(bool(mask_per_head)), B, Hq, Sq, Sk, int(bool(causal)),
                                    int(window_left), int(window_right), _ptr(lq), _ptr(lk), bm, bn, _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_skip_map_ex failed ({rc})")
    return out


def widen(word: int, dtype: int) -> float:
    return _load().oracle_widen(int(word), int(dtype))


def num_threads() -> int:
    return _load().oracle_num_threads()
