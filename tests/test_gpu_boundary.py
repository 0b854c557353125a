"""The C-ABI's ownership rules on the GPU: a custom-mask workspace per stream that repeated
calls reuse (no allocation after the first call of a shape), cached tensor maps (no
re-encoding for the same buffers), and a status word per stream (a timeout on one stream is
not reported on another)."""
import numpy as np
import pytest
import torch

import attention_forward_07_gb300 as af
from attention_forward_07_gb300 import inputs as inp

from gpu_util import assert_close, oracle_full

pytestmark = pytest.mark.gpu


def _dev_inputs(B, H, S, d, dtype, seed, mask=True):
    q, k, v = inp.qkv(B, H, H, S, d, dtype, seed)
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, seed)) if mask else None
    md = None if bits is None else torch.from_numpy(bits.view(np.int32)).cuda()
    return (q, k, v, bits), (q.cuda(), k.cuda(), v.cuda(), md)


def test_repeated_custom_mask_calls_allocate_and_encode_nothing():
    (q, k, v, bits), (qd, kd, vd, md) = _dev_inputs(2, 2, 300, 64, inp.F16, 21)
    o = torch.empty_like(qd)
    lse = torch.empty((2, 2, 300), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    af.attn_release_workspace(s)  # streams come from a pool: start from no workspace
    with torch.cuda.stream(s):
        af.attn_fwd(qd, kd, vd, o, lse, md, causal=True, scale=0.125)
        af.attn_check(s)
        c1 = af.debug_counters()
        for _ in range(3):
            af.attn_fwd(qd, kd, vd, o, lse, md, causal=True, scale=0.125)
        af.attn_check(s)
        c2 = af.debug_counters()
    assert c2["workspace_allocs"] == c1["workspace_allocs"]
    assert c2["map_encodes"] == c1["map_encodes"]
    assert c2["map_hits"] >= c1["map_hits"] + 3 * 6
    o_ref, lse_ref = oracle_full(q, k, v, bits, True, 0.125, inp.F16)
    assert_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                 "reused workspace")
    # a call that needs more grows the workspace once, then reuses it
    (q2, k2, v2, bits2), (qd2, kd2, vd2, md2) = _dev_inputs(4, 2, 2000, 64, inp.F16, 22)
    o2 = torch.empty_like(qd2)
    lse2 = torch.empty((4, 2, 2000), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        af.attn_fwd(qd2, kd2, vd2, o2, lse2, md2, scale=0.125)
        af.attn_fwd(qd2, kd2, vd2, o2, lse2, md2, scale=0.125)
        af.attn_check(s)
    c3 = af.debug_counters()
    assert c3["workspace_allocs"] == c2["workspace_allocs"] + 1
    af.attn_release_workspace(s)
    s.synchronize()


def test_timeout_is_reported_only_on_its_own_stream():
    lib = af.library()
    (q, k, v, _), (qd, kd, vd, _) = _dev_inputs(1, 2, 300, 64, inp.F16, 23, mask=False)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    oa, ob = torch.empty_like(qd), torch.empty_like(qd)
    la = torch.empty((1, 2, 300), dtype=torch.float32, device="cuda")
    lb = torch.empty_like(la)
    # both streams have run once, so each has its own status word
    af.attn_fwd(qd, kd, vd, oa, la, causal=True, stream=sa)
    af.attn_fwd(qd, kd, vd, ob, lb, causal=True, stream=sb)
    af.attn_check(sa)
    af.attn_check(sb)
    assert lib.attn_set_wait_timeout_ns(50_000_000) == 0
    try:
        assert lib.attn_debug_inject(1) == 0
        af.attn_fwd(qd, kd, vd, ob, lb, causal=True, stream=sb)   # this launch times out
        af.attn_fwd(qd, kd, vd, oa, la, causal=True, stream=sa)   # this one does not
        sb.synchronize()
        af.attn_check(sa)                                          # stream A: clean
        with pytest.raises(af.AttnError) as ei:
            af.attn_check(sb)
        assert ei.value.status == -4
        af.attn_check(sb)                                          # cleared by the read
    finally:
        lib.attn_debug_inject(0)
        lib.attn_set_wait_timeout_ns(0)
    o_ref, lse_ref = oracle_full(q, k, v, None, True, 1.0 / 8, inp.F16)
    assert_close(oa.float().cpu().numpy().astype(np.float64), la.cpu().numpy().astype(np.float64), o_ref, lse_ref,
                 "stream A")
