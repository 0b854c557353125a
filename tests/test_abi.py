"""The C-ABI library without a GPU: it loads, exports every symbol include/attn.h
declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest
import torch

import attention_forward_07_gb300 as af
from attention_forward_07_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from attention_forward_07_gb300 import build
    build.build()
    return af.library()


def _declared():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "attn_fwd" in names and len(names) >= 6
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_binding.EXPORTS) == names


def test_no_vendor_gemm_or_attention_library_linked(lib):
    """Our own build's dynamic dependencies and undefined symbols name no cuBLAS, cuDNN or
    CUTLASS: the contractions are this library's own tcgen05 code."""
    import subprocess
    path = _binding.library_path()
    needed = subprocess.run(["readelf", "-d", path], capture_output=True, text=True).stdout
    undef = subprocess.run(["nm", "-D", "--undefined-only", path], capture_output=True, text=True).stdout
    for banned in ("cublas", "cudnn", "cutlass", "cute"):
        assert banned not in needed.lower() and banned not in undef.lower(), banned


def test_strings_and_tile_shape(lib):
    assert af.attn_strerror(0) == "ok"
    assert af.attn_strerror(-4) == "kernel barrier wait timed out"
    assert af.attn_tile_shape(64) == (128, 128)
    assert af.attn_tile_shape(128) == (128, 128)
    with pytest.raises(af.AttnError):
        af.attn_tile_shape(96)
    assert lib.attn_version() >= 100


# Fake, never-dereferenced device pointers: validation must fail before any access.
P = 0x10000


def _fwd(lib, q=P, k=P, v=P, o=P, lse=None, mask=None, B=1, Hq=2, Hkv=2, S=128, d=64, causal=0,
         scale=0.125, dtype=0, stream=None):
    vp = ctypes.c_void_p
    return lib.attn_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse) if lse else None, vp(mask) if mask else None,
                        B, Hq, Hkv, S, d, causal, ctypes.c_float(scale), dtype, stream)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), -1), (dict(k=0), -1), (dict(v=0), -1), (dict(o=0), -1),
    (dict(B=0), -1), (dict(S=0), -1), (dict(Hq=0), -1), (dict(Hkv=0), -1), (dict(Hq=3, Hkv=2), -1),
    (dict(d=96), -2), (dict(d=32), -2), (dict(dtype=2), -2),
    (dict(scale=0.0), -1), (dict(scale=-1.0), -1), (dict(scale=float("inf")), -1), (dict(scale=float("nan")), -1),
    (dict(q=P + 8), -1), (dict(o=P + 2), -1), (dict(lse=P + 2), -1), (dict(mask=P + 1), -1),
    (dict(B=1 << 16, Hq=1 << 8, Hkv=1 << 8, S=1 << 16), -1),
])
def test_validation_before_launch(lib, kw, status):
    assert _fwd(lib, **kw) == status


def test_visited_requires_buffer(lib):
    vp = ctypes.c_void_p
    rc = lib.attn_fwd_visited(vp(P), vp(P), vp(P), vp(P), None, None, 1, 1, 1, 8, 64, 0,
                              ctypes.c_float(0.1), 0, None, None)
    assert rc == -1


def test_hooks(lib):
    assert lib.attn_set_wait_timeout_ns(123456789) == 0
    assert lib.attn_set_wait_timeout_ns(0) == 0
    assert lib.attn_debug_inject(2) == -1
    assert lib.attn_debug_inject(0) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_device_error(lib):
    assert _fwd(lib) == -5


def test_fwd_ex_validation(lib):
    from attention_forward_07_gb300._binding import FwdParams
    assert lib.attn_fwd_ex(None) == -1
    base = dict(q=P, k=P, v=P, o=P, B=1, Hq=2, Hkv=2, Sq=128, Sk=256, d=64, causal=1, window_left=-1,
                window_right=-1, scale=0.125, dtype=0)
    for kw, status in ((dict(Sk=64), -1), (dict(window_left=-2), -1), (dict(window_right=-5), -1),
                       (dict(mask_per_head=2), -1), (dict(d=80), -2), (dict(Sq=0), -1),
                       (dict(seqlens_q=P + 2), -1), (dict(seqlens_k=P + 1), -1),
                       # packed layouts: both offset arrays, no padded lengths, no custom mask
                       (dict(cu_seqlens_q=P, max_seqlen_q=8, max_seqlen_k=8), -1),
                       (dict(cu_seqlens_q=P, cu_seqlens_k=P, max_seqlen_q=0, max_seqlen_k=8), -1),
                       (dict(cu_seqlens_q=P, cu_seqlens_k=P, seqlens_q=P, max_seqlen_q=8, max_seqlen_k=8), -1),
                       (dict(cu_seqlens_q=P, cu_seqlens_k=P, mask_bits=P, max_seqlen_q=8, max_seqlen_k=8), -2),
                       (dict(cu_seqlens_q=P + 2, cu_seqlens_k=P, max_seqlen_q=8, max_seqlen_k=8), -1)):
        args = dict(base, **kw)
        assert lib.attn_fwd_ex(ctypes.byref(FwdParams(**args))) == status, kw
