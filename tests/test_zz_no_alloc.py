"""attn_fwd_noalloc: the entry point for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: an allocator or memory-pool hook would re-enter
itself, a real-time path may not wait on the allocator, a host may hand out a fixed
budget up front.  For them the custom-mask pre-pass writes into a fixed array the
library reserves per GPU.  Its results are checked against the fp64 oracle and against
attn_fwd on the same inputs, over calls in a row whose shapes differ, so that nothing a
previous call left in the shared array can leak into the next.  This file is collected
last so that, if it fails, a run stopping at the first failure has already run every
other test; it passes alone in a fresh process (the first call then loads the device
code) and after the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_forward_07_gb300 as af
from attention_forward_07_gb300 import inputs as inp

from gpu_util import assert_close, oracle_full

pytestmark = pytest.mark.gpu

LIMIT = 4 << 20  # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def scratch_bytes(nm, Sq, Sk):
    """The custom-mask scratch size as include/attn.h states it."""
    r256 = lambda x: -(-x // 256) * 256  # noqa: E731
    R, T, U, N = -(-Sq // 16), -(-Sq // 128), -(-Sq // 256), -(-Sk // 128)
    return r256(nm * Sq * N * 16) + r256(nm * R * N) + r256(nm * R) + r256(nm * U * 64) + r256(nm * T * N)


def _case(B, H, S, d, dtype, seed, mask):
    q, k, v = inp.qkv(B, H, H, S, d, dtype, seed)
    if mask == "bernoulli":
        bits = inp.pack_bits(inp.bernoulli_mask(B, S, seed))
    else:
        bits = inp.pack_bits(inp.block_sparse_mask(B, S, seed))
    return q, k, v, bits


def _run(entry, q, k, v, bits, causal):
    dev = "cuda"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = torch.from_numpy(bits.view(np.int32)).to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    entry(qd, kd, vd, o, lse, md, causal=causal, scale=1.0 / q.shape[-1] ** 0.5)
    af.attn_check()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(case, causal, what):
    q, k, v, bits = case
    got = _run(af.attn_fwd_noalloc, q, k, v, bits, causal)
    dtype = inp.F16 if q.dtype == torch.float16 else inp.BF16
    o_ref, lse_ref = oracle_full(q, k, v, bits, causal, 1.0 / q.shape[-1] ** 0.5, dtype)
    assert_close(got[0], got[1], o_ref, lse_ref, what)
    return got


def test_noalloc_against_the_oracle_on_calls_in_a_row():
    # a large dense-mask call, then smaller and sparser ones of other shapes, then the
    # large one again: every call is checked against the oracle
    big = _case(4, 2, 1024, 64, inp.F16, 31, "bernoulli")
    small = _case(3, 2, 300, 128, inp.BF16, 32, "block90")
    tiny = _case(1, 1, 77, 64, inp.F16, 33, "block90")
    first = _check(big, False, "big")
    _check(small, True, "small after big")
    _check(tiny, False, "tiny after small")
    again = _check(big, False, "big again")
    assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])
    # and it gives what attn_fwd gives on the same inputs
    ref = _run(af.attn_fwd, *small, True)
    got = _run(af.attn_fwd_noalloc, *small, True)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_noalloc_just_under_the_limit():
    B, H, S, d = 1, 1, 5760, 64
    need = scratch_bytes(B, S, S)
    assert 0.99 * LIMIT < need <= LIMIT
    case = _case(B, H, S, d, inp.F16, 34, "block90")
    _check(case, True, "S=5760")
    _check(case, True, "S=5760 second call")


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = af.library()
    B, H, S, d = 1, 1, 5888, 64
    assert scratch_bytes(B, S, S) > LIMIT
    q = torch.zeros((B, H, S, d), dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    m = torch.zeros((B, S, S // 32), dtype=torch.int32, device="cuda")
    vp = ctypes.c_void_p
    rc = lib.attn_fwd_noalloc(vp(q.data_ptr()), vp(q.data_ptr()), vp(q.data_ptr()), vp(o.data_ptr()), None,
                              vp(m.data_ptr()), B, H, H, S, d, 0, ctypes.c_float(0.125), 0, None)
    assert rc == -1
    # without a custom mask nothing goes into the array, so any size works
    af.attn_fwd_noalloc(q, q, q, o)
    af.attn_check()
