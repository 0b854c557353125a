"""Helpers shared by the GPU tests: run the CUDA path through the C-ABI, compare to the oracle."""
import numpy as np
import torch

import attention_forward_07_gb300 as af
import oracle
from attention_forward_07_gb300 import inputs as inp

O_ATOL, O_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3


def run_cuda(q, k, v, bits, causal, scale, visited=False, dev="cuda:0"):
    """Copy CPU inputs to the device, run attn_fwd (or attn_fwd_visited), return host results."""
    B, Hq, S, d = q.shape
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if bits is None else torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device=dev)
    vis = None
    if visited:
        bm, bn = af.attn_tile_shape(d)
        vis = torch.zeros((B, Hq, -(-S // bm), -(-S // bn)), dtype=torch.uint8, device=dev)
        af.attn_fwd_visited(qd, kd, vd, o, lse, md, causal, scale, vis)
    else:
        af.attn_fwd(qd, kd, vd, o, lse, md, causal=causal, scale=scale)
    af.attn_check()
    out = (o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))
    if visited:
        out = out + (vis.cpu().numpy(),)
    return out


def oracle_full(q, k, v, bits, causal, scale, dtype):
    return oracle.attn_fwd(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), dtype, bits, causal,
                           float(np.float32(scale)))


def oracle_rows(q, k, v, bits, causal, scale, dtype, rows):
    return oracle.attn_rows(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), dtype, rows, bits, causal,
                            float(np.float32(scale)))


def stratified_rows(B, Hq, S, seed):
    """Flat row ids (b*Hq + hq)*S + i for every (b, hq): one seeded random row from every
    32-row warp slice (so every warp of both Q tiles of every 256-row work unit, and every
    unit of every CTA's walk, is represented), plus rows 0, 1, 127, 128 (the Q-tile seam),
    255, 256 (the unit seam), S-256 and S-1."""
    rng = np.random.default_rng(int(seed) + 11)
    nsl = -(-S // 32)
    fixed = np.array(sorted({r for r in (0, 1, 127, 128, 255, 256, S - 256, S - 1) if 0 <= r < S}), np.int64)
    out = []
    for bh in range(B * Hq):
        pick = np.minimum(32 * np.arange(nsl) + rng.integers(0, 32, size=nsl), S - 1)
        out.append(bh * S + np.unique(np.concatenate([pick, fixed])))
    return np.concatenate(out)


def assert_close(o, lse, o_ref, lse_ref, what=""):
    """The parity bar: |O - O_ref| <= 1e-2 + 1e-2*|O_ref| elementwise, |LSE - LSE_ref| <= 1e-3,
    -inf LSE exactly where the oracle has it, and no NaN/Inf anywhere else."""
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    excess = np.abs(o - o_ref) - (O_ATOL + O_RTOL * np.abs(o_ref))
    if excess.max() > 0:
        idx = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"{what}: O out of tolerance at {idx}: got {o[idx]} want {o_ref[idx]} "
                             f"({int((excess > 0).sum())} of {excess.size} elements)")
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg), f"{what}: -inf LSE pattern differs"
    assert np.all(np.isfinite(lse[~neg])), f"{what}: non-finite LSE"
    if (~neg).any():
        err = np.abs(lse[~neg] - lse_ref[~neg]).max()
        assert err <= LSE_ATOL, f"{what}: LSE error {err}"


def expected_visited(bits, per_head, B, Hq, Sq, Sk, causal, window_left=-1, window_right=-1, seqlens_q=None,
                     seqlens_k=None):
    """The visited map the kernel must produce, uint8 [B, Hq, ceil(Sq/128), ceil(Sk/128)].

    Without a custom mask: the oracle's (128-row, 128-key) block map.  With one, the kernel
    first compacts the query rows: the 16-row blocks that hold a kept entry, in ascending
    order, eight to a 128-row tile; a (compacted tile, key tile) block is visited iff one of
    its 16-row blocks holds a kept entry in that key tile -- built here from the oracle's
    (16-row, 128-key) block map."""
    nqt, nkt = -(-Sq // 128), -(-Sk // 128)
    if bits is None:
        ref = oracle.skip_map_ex(None, False, B, Hq, Sq, Sk, causal, window_left, window_right, 128, 128,
                                 seqlens_q=seqlens_q, seqlens_k=seqlens_k)
        return np.repeat(ref.reshape(B, 1, nqt, nkt), Hq, axis=1)
    f16 = oracle.skip_map_ex(bits, per_head, B, Hq, Sq, Sk, causal, window_left, window_right, 16, 128,
                             seqlens_q=seqlens_q, seqlens_k=seqlens_k)
    out = np.zeros((f16.shape[0], nqt, nkt), np.uint8)
    for mb in range(f16.shape[0]):
        blocks = np.nonzero(f16[mb].any(axis=1))[0]
        for ct in range(-(-len(blocks) // 8)):
            out[mb, ct] = f16[mb, blocks[ct * 8:(ct + 1) * 8]].any(axis=0)
    out = out.reshape(B, -1, nqt, nkt)
    return out if out.shape[1] == Hq else np.repeat(out, Hq, axis=1)
