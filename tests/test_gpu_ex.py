"""attn_fwd_ex against the oracle's extended definition: Sq < Sk bottom-right aligned,
sliding-window bands, per-head custom masks, and the tile-skip map under them."""
import numpy as np
import pytest
import torch

import attention_forward_07_gb300 as af
import oracle
from attention_forward_07_gb300 import inputs as inp

from gpu_util import assert_close, expected_visited

pytestmark = pytest.mark.gpu


def _run(q, k, v, bits, per_head, causal, wl, wr, scale, visited=False):
    dev = "cuda"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if bits is None else torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(dev)
    B, Hq, Sq, d = q.shape
    Sk = k.shape[2]
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device=dev)
    vis = torch.zeros((B, Hq, -(-Sq // 128), -(-Sk // 128)), dtype=torch.uint8, device=dev) if visited else None
    af.attn_fwd_ex(qd, kd, vd, o, lse, md, per_head, causal, wl, wr, scale, vis)
    af.attn_check()
    out = (o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))
    return out + ((vis.cpu().numpy(),) if visited else ())


CASES = [
    # B, Hq, Hkv, Sq, Sk, d, dtype, causal, wl, wr, mask
    (2, 4, 2, 200, 500, 128, inp.BF16, True, -1, -1, None),        # prefill against a cache
    (1, 2, 2, 1, 300, 64, inp.F16, True, -1, -1, None),            # one new query
    (1, 3, 3, 257, 257, 128, inp.BF16, True, 100, -1, None),       # causal sliding window
    (2, 2, 1, 700, 700, 64, inp.F16, False, 50, 30, None),         # symmetric-ish band
    (1, 2, 2, 300, 900, 128, inp.BF16, False, 200, 40, None),      # band with Sq < Sk
    (2, 4, 2, 256, 384, 64, inp.F16, True, -1, -1, "shared"),      # custom mask, Sq < Sk
    (2, 4, 2, 300, 300, 128, inp.BF16, True, 120, -1, "head"),     # per-head mask + window
    (1, 4, 4, 129, 640, 64, inp.F16, False, -1, -1, "head"),       # per-head, ragged
    # masks with whole empty 16-row blocks: the rows are compacted before the tiles are formed
    (2, 4, 2, 512, 512, 64, inp.F16, False, -1, -1, "sparse"),
    (2, 2, 2, 700, 900, 128, inp.BF16, True, -1, -1, "sparse"),
    (1, 4, 4, 333, 333, 64, inp.F16, True, 90, -1, "sparse_head"),
    (2, 2, 1, 1100, 1100, 128, inp.BF16, False, 200, 100, "sparse"),
    # at most 128 queries and an even group size: a unit pairs two query heads of a K/V head
    (2, 8, 2, 100, 700, 128, inp.BF16, True, -1, -1, None),
    (1, 4, 1, 128, 300, 64, inp.F16, False, -1, -1, None),
    (2, 8, 4, 1, 513, 128, inp.BF16, True, 50, -1, None),
    (3, 6, 3, 77, 77, 64, inp.BF16, True, -1, -1, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_Sq{}_Sk{}_d{}_c{}_w{}_{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], int(c[7]), c[8], c[9], c[10]))
def test_extended_parity_and_skip_map(case):
    B, Hq, Hkv, Sq, Sk, d, dtype, causal, wl, wr, mask = case
    q, k, v = inp.qkv(B, Hq, Hkv, Sk, d, dtype, Sq + Sk)
    q = q[:, :, :Sq].contiguous()
    per_head = mask == "head"
    bits = None
    if mask == "shared":
        bits = inp.pack_bits(inp.bernoulli_mask(B, Sk, 3)[:, :Sq])
    elif mask == "head":
        keep = inp.bernoulli_mask(B * Hq, Sk, 4)[:, :Sq]
        bits = inp.pack_bits(keep).reshape(B, Hq, Sq, -1)
    elif mask == "sparse":
        bits = inp.pack_bits(inp.block_sparse_mask(B, Sk, 7)[:, :Sq])
    elif mask == "sparse_head":
        per_head = True
        bits = inp.pack_bits(inp.block_sparse_mask(B * Hq, Sk, 8)[:, :Sq]).reshape(B, Hq, Sq, -1)
    scale = 1.0 / d ** 0.5
    o, lse, vis = _run(q, k, v, bits, per_head, causal, wl, wr, scale, visited=True)
    o_ref, lse_ref = oracle.attn_rows_ex(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), dtype, None, bits,
                                         per_head, causal, wl, wr, float(np.float32(scale)))
    assert_close(o, lse, o_ref, lse_ref, str(case))
    assert np.array_equal(vis, expected_visited(bits, per_head, B, Hq, Sq, Sk, causal, wl, wr))


def test_ex_defaults_are_attn_fwd():
    B, Hq, Hkv, S, d = 2, 4, 2, 333, 128
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, inp.BF16, 1)
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, 1))
    for causal in (False, True):
        for b in (None, bits):
            a = _run(q, k, v, b, False, causal, -1, -1, 0.1)
            qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
            o = torch.empty_like(qd)
            lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
            md = None if b is None else torch.from_numpy(b.view(np.int32)).cuda()
            af.attn_fwd(qd, kd, vd, o, lse, md, causal=causal, scale=0.1)
            af.attn_check()
            assert np.array_equal(a[0], o.float().cpu().numpy()) and np.array_equal(a[1], lse.cpu().numpy())


VARLEN_CASES = [
    # B, Hq, Hkv, Sq, Sk, d, dtype, causal, wl, wr, mask
    (4, 2, 1, 300, 300, 128, inp.BF16, True, -1, -1, None),
    (4, 8, 2, 120, 640, 128, inp.BF16, True, -1, -1, None),      # head pairs, per-entry lengths
    (4, 4, 2, 257, 520, 64, inp.F16, False, -1, -1, None),
    (3, 2, 2, 384, 700, 128, inp.F16, False, 90, 20, None),
    (4, 2, 1, 260, 400, 64, inp.BF16, True, -1, -1, "shared"),
    (3, 4, 4, 200, 333, 128, inp.BF16, True, 64, -1, "head"),
    (4, 2, 2, 600, 600, 64, inp.F16, True, -1, -1, "sparse"),
]


def _lengths(B, Sq, Sk, seed):
    """Per-entry lengths with the edge cases in the first entries: an entry with no queries,
    one with fewer keys than queries, one at the full padded size; the rest random."""
    g = np.random.default_rng(seed)
    lq = g.integers(1, Sq + 1, size=B).astype(np.int32)
    lk = g.integers(1, Sk + 1, size=B).astype(np.int32)
    lq[0], lk[0] = 0, Sk // 2
    if B > 1:
        lq[1], lk[1] = Sq, max(1, Sq // 3)
    if B > 2:
        lq[2], lk[2] = Sq, Sk
    return lq, lk


@pytest.mark.parametrize("case", VARLEN_CASES, ids=lambda c: "B{}_Hq{}_Sq{}_Sk{}_d{}_c{}_w{}_{}_{}".format(
    c[0], c[1], c[3], c[4], c[5], int(c[7]), c[8], c[9], c[10]))
def test_varlen_parity_and_skip_map(case):
    """Per-entry lengths inside padded buffers: rows below sq_b match the oracle (bottom-right
    alignment per entry), rows at or past it are left untouched, key rows past sk_b do not
    reach the result even when k holds NaN there, and the skip map is exact."""
    B, Hq, Hkv, Sq, Sk, d, dtype, causal, wl, wr, mask = case
    q, k, v = inp.qkv(B, Hq, Hkv, Sk, d, dtype, 7 * Sq + Sk)
    q = q[:, :, :Sq].contiguous()
    lq, lk = _lengths(B, Sq, Sk, Sq + Sk)
    per_head = mask == "head"
    bits = None
    if mask == "shared":
        bits = inp.pack_bits(inp.bernoulli_mask(B, Sk, 5)[:, :Sq])
    elif mask == "head":
        bits = inp.pack_bits(inp.bernoulli_mask(B * Hq, Sk, 6)[:, :Sq]).reshape(B, Hq, Sq, -1)
    elif mask == "sparse":
        bits = inp.pack_bits(inp.block_sparse_mask(B, Sk, 9)[:, :Sq])
    k_nan = k.clone()
    for b in range(B):
        k_nan[b, :, int(lk[b]):] = float("nan")
    dev = "cuda"
    qd, kd, vd = q.to(dev), k_nan.to(dev), v.to(dev)
    md = None if bits is None else torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device=dev)
    vis = torch.zeros((B, Hq, -(-Sq // 128), -(-Sk // 128)), dtype=torch.uint8, device=dev)
    scale = 1.0 / d ** 0.5
    af.attn_fwd_ex(qd, kd, vd, o, lse, md, per_head, causal, wl, wr, scale, vis,
                   seqlens_q=torch.from_numpy(lq).to(dev), seqlens_k=torch.from_numpy(lk).to(dev))
    af.attn_check()
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    o_ref, lse_ref = oracle.attn_rows_ex(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), dtype, None, bits, per_head,
                                         causal, wl, wr, float(np.float32(scale)), seqlens_q=lq, seqlens_k=lk)
    for b in range(B):
        n = int(lq[b])
        assert np.all(np.isnan(o[b, :, n:])) and np.all(np.isnan(lse[b, :, n:])), f"entry {b}: padded rows written"
        if n:
            assert_close(o[b, :, :n], lse[b, :, :n], o_ref[b, :, :n], lse_ref[b, :, :n], f"{case} entry {b}")
    assert np.array_equal(vis.cpu().numpy(), expected_visited(bits, per_head, B, Hq, Sq, Sk, causal, wl, wr,
                                                              seqlens_q=lq, seqlens_k=lk))


def test_varlen_full_lengths_equal_padded():
    """Lengths equal to the padded sizes give bit-identical results to no lengths at all."""
    B, Hq, Hkv, Sq, Sk, d = 2, 2, 2, 200, 450, 64
    q, k, v = inp.qkv(B, Hq, Hkv, Sk, d, inp.F16, 11)
    q = q[:, :, :Sq].contiguous().cuda()
    k, v = k.cuda(), v.cuda()
    outs = []
    for lens in (None, (torch.full((B,), Sq, dtype=torch.int32, device="cuda"),
                        torch.full((B,), Sk, dtype=torch.int32, device="cuda"))):
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
        af.attn_fwd_ex(q, k, v, o, lse, causal=True, seqlens_q=None if lens is None else lens[0],
                       seqlens_k=None if lens is None else lens[1])
        af.attn_check()
        outs.append((o.cpu(), lse.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


PACKED_CASES = [
    # Hq, Hkv, d, dtype, causal, wl, wr, query lengths, key lengths
    (4, 2, 128, inp.BF16, True, -1, -1, [300, 0, 129, 512], [300, 77, 400, 512]),
    (2, 2, 64, inp.F16, False, -1, -1, [1, 256, 333], [700, 256, 333]),
    (4, 1, 64, inp.F16, True, 100, -1, [200, 450, 17, 256, 90], [200, 900, 17, 300, 1]),
    (8, 2, 128, inp.BF16, True, -1, -1, [100, 1, 128, 64, 0, 33], [900, 1, 128, 640, 12, 33]),  # head pairs
]


@pytest.mark.parametrize("case", PACKED_CASES, ids=lambda c: "Hq{}_Hkv{}_d{}_c{}_w{}_{}_n{}".format(
    c[0], c[1], c[2], int(c[4]), c[5], c[6], len(c[7])))
def test_packed_varlen_matches_padded_and_oracle(case):
    """Packed variable-length batches (cu_seqlens): each entry's rows equal the padded
    per-entry-length run bit for bit (same tiles, same order) and the oracle within the
    tolerance; the visited maps agree; rows outside every entry are not written."""
    Hq, Hkv, d, dtype, causal, wl, wr, lq, lk = case
    B = len(lq)
    Sq, Sk = max(lq), max(lk)
    q, k, v = inp.qkv(B, Hq, Hkv, max(Sq, Sk), d, dtype, 31 * Sq + Sk)
    q, k, v = q[:, :, :Sq].contiguous(), k[:, :, :Sk].contiguous(), v[:, :, :Sk].contiguous()
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    # head-major packed buffers with two spare rows after the last entry
    qp = torch.cat([q[b, :, :lq[b]] for b in range(B)] + [torch.zeros(Hq, 2, d, dtype=q.dtype)], dim=1).contiguous()
    kp = torch.cat([k[b, :, :lk[b]] for b in range(B)] + [torch.zeros(Hkv, 2, d, dtype=k.dtype)], dim=1).contiguous()
    vp = torch.cat([v[b, :, :lk[b]] for b in range(B)] + [torch.zeros(Hkv, 2, d, dtype=v.dtype)], dim=1).contiguous()
    dev = "cuda"
    scale = 1.0 / d ** 0.5
    o = torch.full((Hq, qp.shape[1], d), float("nan"), dtype=q.dtype, device=dev)
    lse = torch.full((Hq, qp.shape[1]), float("nan"), dtype=torch.float32, device=dev)
    vis = torch.zeros((B, Hq, -(-Sq // 128), -(-Sk // 128)), dtype=torch.uint8, device=dev)
    af.attn_fwd_packed(qp.to(dev), kp.to(dev), vp.to(dev), o, torch.from_numpy(cq).to(dev),
                       torch.from_numpy(ck).to(dev), Sq, Sk, lse=lse, causal=causal, window_left=wl,
                       window_right=wr, scale=scale, visited=vis)
    af.attn_check()
    # the same batch in padded form with per-entry lengths
    o2 = torch.full((B, Hq, Sq, d), float("nan"), dtype=q.dtype, device=dev)
    lse2 = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device=dev)
    vis2 = torch.zeros_like(vis)
    lqt = torch.tensor(lq, dtype=torch.int32, device=dev)
    lkt = torch.tensor(lk, dtype=torch.int32, device=dev)
    if Sk < Sq:
        pytest.skip("padded form needs Sk >= Sq")
    af.attn_fwd_ex(q.to(dev), k.to(dev), v.to(dev), o2, lse2, None, False, causal, wl, wr, scale, vis2,
                   seqlens_q=lqt, seqlens_k=lkt)
    af.attn_check()
    o, lse, o2, lse2 = o.cpu(), lse.cpu(), o2.cpu(), lse2.cpu()
    assert torch.all(torch.isnan(o[:, cq[-1]:])) and torch.all(torch.isnan(lse[:, cq[-1]:]))
    o_ref, lse_ref = oracle.attn_rows_ex(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), dtype, None, None, False,
                                         causal, wl, wr, float(np.float32(scale)), seqlens_q=np.array(lq),
                                         seqlens_k=np.array(lk))
    for b in range(B):
        rows = slice(int(cq[b]), int(cq[b + 1]))
        n = lq[b]
        assert torch.equal(o[:, rows], o2[b, :, :n]) and torch.equal(lse[:, rows], lse2[b, :, :n]), f"entry {b}"
        if n:
            assert_close(o[:, rows].float().numpy().astype(np.float64), lse[:, rows].numpy().astype(np.float64),
                         o_ref[b, :, :n], lse_ref[b, :, :n], f"{case} entry {b}")
    assert torch.equal(vis.cpu(), vis2.cpu())
