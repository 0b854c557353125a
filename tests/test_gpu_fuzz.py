"""Seeded random configurations across the whole option space of attn_fwd_ex, each checked
row by row against the oracle: padded and packed layouts, per-entry lengths, windows, GQA,
shared / per-head / mostly-empty masks, both dtypes and both head dims, ragged sizes."""
import numpy as np
import pytest
import torch

import attention_forward_07_gb300 as af
import oracle
from attention_forward_07_gb300 import inputs as inp

from gpu_util import assert_close, expected_visited

pytestmark = pytest.mark.gpu

N_CASES = 24


def _config(seed, short_queries=False):
    """short_queries: at most 128 queries and an even GQA group (query-head pairs), lengths and
    packed layouts more often (the variable-length work order)."""
    g = np.random.default_rng((5000 if short_queries else 1000) + seed)
    d = int(g.choice([64, 128]))
    dtype = int(g.choice([inp.F16, inp.BF16]))
    Hkv = int(g.choice([1, 2, 3]))
    Hq = Hkv * int(g.choice([2, 4] if short_queries else [1, 2, 4]))
    B = int(g.integers(1, 6 if short_queries else 4))
    Sq = int(g.integers(1, 129 if short_queries else 420))
    Sk = int(g.integers(Sq, Sq + 300))
    causal = bool(g.random() < 0.5)
    wl = int(g.choice([-1, -1, int(g.integers(0, 200))]))
    wr = -1 if causal else int(g.choice([-1, -1, int(g.integers(0, 100))]))
    mask = str(g.choice(["none", "none", "shared", "head", "sparse"]))
    packed = mask == "none" and bool(g.random() < (0.6 if short_queries else 0.4))
    lens = bool(g.random() < (0.6 if short_queries else 0.4)) or packed
    lq = g.integers(0, Sq + 1, size=B).astype(np.int32) if lens else None
    lk = g.integers(0, Sk + 1, size=B).astype(np.int32) if lens else None
    return dict(d=d, dtype=dtype, Hkv=Hkv, Hq=Hq, B=B, Sq=Sq, Sk=Sk, causal=causal, wl=wl, wr=wr, mask=mask,
                packed=packed, lq=lq, lk=lk)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_configuration(seed):
    _check(_config(seed), seed)


@pytest.mark.parametrize("seed", range(12))
def test_random_short_query_configuration(seed):
    _check(_config(seed, short_queries=True), 100 + seed)


def _check(c, seed):
    B, Hq, Hkv, Sq, Sk, d, dtype = c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["d"], c["dtype"]
    q, k, v = inp.qkv(B, Hq, Hkv, Sk, d, dtype, 77 * seed + 5)
    q = q[:, :, :Sq].contiguous()
    per_head = c["mask"] == "head"
    bits = None
    if c["mask"] == "shared":
        bits = inp.pack_bits(inp.bernoulli_mask(B, Sk, seed)[:, :Sq])
    elif c["mask"] == "head":
        bits = inp.pack_bits(inp.bernoulli_mask(B * Hq, Sk, seed)[:, :Sq]).reshape(B, Hq, Sq, -1)
    elif c["mask"] == "sparse":
        bits = inp.pack_bits(inp.block_sparse_mask(B, Sk, seed)[:, :Sq])
    scale = 1.0 / d ** 0.5
    dev = "cuda"
    lq, lk = c["lq"], c["lk"]
    o_ref, lse_ref = oracle.attn_rows_ex(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), dtype, None, bits, per_head,
                                         c["causal"], c["wl"], c["wr"], float(np.float32(scale)),
                                         seqlens_q=lq, seqlens_k=lk)
    what = str({key: (val.tolist() if isinstance(val, np.ndarray) else val) for key, val in c.items()})
    if c["packed"]:
        cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
        qp = torch.cat([q[b, :, :lq[b]] for b in range(B)] + [torch.zeros(Hq, 1, d, dtype=q.dtype)], dim=1).contiguous()
        kp = torch.cat([k[b, :, :lk[b]] for b in range(B)] + [torch.zeros(Hkv, 1, d, dtype=k.dtype)], dim=1).contiguous()
        vp = torch.cat([v[b, :, :lk[b]] for b in range(B)] + [torch.zeros(Hkv, 1, d, dtype=v.dtype)], dim=1).contiguous()
        o = torch.full((Hq, qp.shape[1], d), float("nan"), dtype=q.dtype, device=dev)
        lse = torch.full((Hq, qp.shape[1]), float("nan"), dtype=torch.float32, device=dev)
        af.attn_fwd_packed(qp.to(dev), kp.to(dev), vp.to(dev), o, torch.from_numpy(cq).to(dev),
                           torch.from_numpy(ck).to(dev), Sq, Sk, lse=lse, causal=c["causal"],
                           window_left=c["wl"], window_right=c["wr"], scale=scale)
        af.attn_check()
        o = o.cpu().float().numpy().astype(np.float64)
        lse = lse.cpu().numpy().astype(np.float64)
        for b in range(B):
            n = int(lq[b])
            if n:
                rows = slice(int(cq[b]), int(cq[b + 1]))
                assert_close(o[:, rows], lse[:, rows], o_ref[b, :, :n], lse_ref[b, :, :n], f"{what} entry {b}")
        assert np.all(np.isnan(o[:, cq[-1]:]))
        return
    md = None if bits is None else torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(dev)
    o = torch.full((B, Hq, Sq, d), float("nan"), dtype=q.dtype, device=dev)
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device=dev)
    vis = torch.zeros((B, Hq, -(-Sq // 128), -(-Sk // 128)), dtype=torch.uint8, device=dev)
    af.attn_fwd_ex(q.to(dev), k.to(dev), v.to(dev), o, lse, md, per_head, c["causal"], c["wl"], c["wr"], scale, vis,
                   seqlens_q=None if lq is None else torch.from_numpy(lq).to(dev),
                   seqlens_k=None if lk is None else torch.from_numpy(lk).to(dev))
    af.attn_check()
    o = o.cpu().float().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    for b in range(B):
        n = Sq if lq is None else int(lq[b])
        if n:
            assert_close(o[b, :, :n], lse[b, :, :n], o_ref[b, :, :n], lse_ref[b, :, :n], f"{what} entry {b}")
        assert np.all(np.isnan(o[b, :, n:]))
    assert np.array_equal(vis.cpu().numpy(), expected_visited(bits, per_head, B, Hq, Sq, Sk, c["causal"], c["wl"],
                                                              c["wr"], seqlens_q=lq, seqlens_k=lk))
