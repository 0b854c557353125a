"""CUDA path vs the fp64 oracle, element by element, through the C-ABI.

Small cases are checked on every output.  The full-size workloads of the pages'
benchmarks are launched exactly as bench.py launches them and checked on a stratified
row sample (every (batch, head) pair: one row from every 32-row warp slice, plus the
tile and unit seams and the last rows); one of them (causal MHA, S = 4096) is checked on
every row.
"""
import numpy as np
import pytest
import torch

from attention_forward_07_gb300 import inputs as inp

from gpu_util import assert_close, expected_visited, oracle_full, oracle_rows, run_cuda, stratified_rows

import oracle

pytestmark = pytest.mark.gpu


def _case(B, Hq, Hkv, S, d, dtype, causal, mask, seed, scale=None):
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, dtype, seed)
    if mask == "bernoulli":
        bits = inp.pack_bits(inp.bernoulli_mask(B, S, seed))
    elif mask == "block90":
        bits = inp.pack_bits(inp.block_sparse_mask(B, S, seed))
    elif mask == "sparse":
        bits = inp.pack_bits(inp.bernoulli_mask(B, S, seed, p_keep=0.02))
    else:
        bits = None
    scale = scale if scale is not None else 1.0 / d ** 0.5
    return q, k, v, bits, causal, scale


SMALL = [
    # B, Hq, Hkv, S, d, dtype, causal, mask
    (1, 2, 2, 128, 64, inp.F16, False, "bernoulli"),     # the tiny masked workload
    (1, 1, 1, 1, 64, inp.F16, False, "none"),            # S = 1
    (1, 1, 1, 1, 128, inp.BF16, True, "none"),
    (2, 2, 2, 33, 128, inp.BF16, False, "none"),         # one ragged tile
    (1, 3, 3, 129, 64, inp.BF16, True, "none"),          # 128 + 1
    (1, 2, 2, 256, 128, inp.BF16, False, "none"),        # exactly one unit
    (1, 2, 2, 257, 128, inp.BF16, True, "none"),         # one unit + one row
    (2, 2, 2, 300, 128, inp.BF16, False, "none"),
    (2, 2, 2, 300, 128, inp.BF16, True, "none"),
    (1, 2, 2, 384, 128, inp.F16, True, "none"),          # fp16, d = 128
    (2, 4, 2, 260, 128, inp.BF16, True, "none"),         # GQA g = 2
    (1, 8, 1, 200, 64, inp.BF16, False, "none"),         # GQA g = 8, d = 64
    (2, 2, 2, 300, 64, inp.F16, False, "bernoulli"),
    (2, 2, 2, 300, 128, inp.BF16, True, "bernoulli"),    # custom AND causal
    (2, 4, 1, 512, 64, inp.F16, False, "block90"),       # tile skipping
    (1, 2, 2, 700, 64, inp.F16, True, "block90"),
    (1, 2, 2, 450, 128, inp.F16, False, "sparse"),       # most rows fully masked in some tiles
    (2, 8, 2, 100, 128, inp.BF16, True, "none"),         # S <= 128, group 4: query-head pairs
    (1, 4, 2, 128, 64, inp.F16, False, "none"),          # S = 128, group 2
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B{}_Hq{}_Hkv{}_S{}_d{}_{}_{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], inp.DTYPE_NAME[c[5]], "causal" if c[6] else "full", c[7]))
def test_small_full_parity(case):
    B, Hq, Hkv, S, d, dtype, causal, mask = case
    q, k, v, bits, causal, scale = _case(B, Hq, Hkv, S, d, dtype, causal, mask, seed=S + 17)
    o, lse = run_cuda(q, k, v, bits, causal, scale)
    o_ref, lse_ref = oracle_full(q, k, v, bits, causal, scale, dtype)
    assert_close(o, lse, o_ref, lse_ref, str(case))


def test_fully_masked_rows_and_tiles():
    B, H, S, d = 1, 2, 300, 64
    q, k, v = inp.qkv(B, H, H, S, d, inp.F16, 5)
    keep = inp.bernoulli_mask(B, S, 5)
    keep[0, 0:128] = False         # a whole query tile with nothing kept
    keep[0, 140] = False           # single rows
    keep[0, 299] = False
    keep[0, :, 128:256] = False    # a whole key tile empty for every row
    bits = inp.pack_bits(keep)
    o, lse = run_cuda(q, k, v, bits, False, 0.125)
    o_ref, lse_ref = oracle_full(q, k, v, bits, False, 0.125, inp.F16)
    assert_close(o, lse, o_ref, lse_ref, "masked rows")
    assert np.all(o[0, :, :128] == 0) and np.all(np.isneginf(lse[0, :, :128]))


def test_causal_equals_lower_triangular_mask():
    B, H, S, d = 2, 2, 333, 128
    q, k, v = inp.qkv(B, H, H, S, d, inp.BF16, 9)
    tri = inp.pack_bits(torch.tril(torch.ones((S, S), dtype=torch.bool)).expand(B, S, S))
    a = run_cuda(q, k, v, None, True, 0.09)
    b = run_cuda(q, k, v, tri, False, 0.09)
    # The causal path walks the key tiles of odd block levels from the diagonal down, the mask
    # path from key 0 up.  The order changes the fp32 sums and the exponent base each row
    # settles on (so P rounds to bf16 differently): absolute differences of order 1e-3, and an
    # output may then round to the neighbouring bf16 value (one step = 2^-7 of its magnitude).
    np.testing.assert_allclose(a[0], b[0], rtol=2.0 ** -7, atol=2e-3)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-4)


@pytest.mark.parametrize("S,causal,mask,d,H,Hkv", [(512, False, "block90", 64, 3, 3), (700, True, "block90", 64, 3, 3),
                                                     (1000, True, "none", 128, 3, 3),
                                                     (384, False, "bernoulli", 128, 3, 3),
                                                     (600, True, "sparse", 64, 3, 3), (100, True, "none", 128, 8, 2)])
def test_skip_map_is_exact(S, causal, mask, d, H, Hkv):
    B = 2
    q, k, v, bits, causal, scale = _case(B, H, Hkv, S, d, inp.F16, causal, mask, seed=S)
    o, lse, vis = run_cuda(q, k, v, bits, causal, scale, visited=True)
    assert np.array_equal(vis, expected_visited(bits, False, B, H, S, S, causal))
    o_ref, lse_ref = oracle_full(q, k, v, bits, causal, scale, inp.F16)
    assert_close(o, lse, o_ref, lse_ref, "visited run")


def test_deterministic():
    q, k, v, bits, causal, scale = _case(2, 4, 2, 777, 128, inp.BF16, True, "none", seed=3)
    a = run_cuda(q, k, v, bits, causal, scale)
    b = run_cuda(q, k, v, bits, causal, scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1], equal_nan=True)


def test_many_units_per_cta_sampled():
    """More work units than SMs: every CTA walks several units of the persistent loop."""
    B, Hq, Hkv, S, d = 4, 8, 2, 2304, 128
    for causal in (False, True):
        q, k, v, bits, causal, scale = _case(B, Hq, Hkv, S, d, inp.BF16, causal, "none", seed=11)
        o, lse = run_cuda(q, k, v, bits, causal, scale)
        rows = inp.sample_rows(B, Hq, S, 24, seed=1)
        o_ref, lse_ref = oracle_rows(q, k, v, bits, causal, scale, inp.BF16, rows)
        assert_close(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, f"causal={causal}")


# ------------------------------------------------------------------------ full-size workloads

SHORT = ["tiny_masked", "short_masked", "short_masked90"]
PREFILL = [n for n in inp.WORKLOADS if n not in SHORT]


@pytest.mark.parametrize("name", SHORT)
def test_short_workloads_full_parity(name):
    w = inp.WORKLOADS[name]
    q, k, v, bits = w.make(w.seed(list(inp.WORKLOADS).index(name)))
    o, lse, vis = run_cuda(q, k, v, bits, w.causal, w.scale, visited=True)
    o_ref, lse_ref = oracle_full(q, k, v, bits, w.causal, w.scale, w.dtype)
    assert_close(o, lse, o_ref, lse_ref, name)
    assert np.array_equal(vis, expected_visited(bits, False, w.B, w.Hq, w.S, w.S, w.causal))


@pytest.mark.parametrize("name", PREFILL)
def test_prefill_workloads_sampled_parity(name):
    w = inp.WORKLOADS[name]
    q, k, v, bits = w.make(w.seed(list(inp.WORKLOADS).index(name)))
    o, lse = run_cuda(q, k, v, bits, w.causal, w.scale)
    rows = stratified_rows(w.B, w.Hq, w.S, seed=w.S)
    o_ref, lse_ref = oracle_rows(q, k, v, bits, w.causal, w.scale, w.dtype, rows)
    assert_close(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, name)
    # properties that hold at any size, checked on every row: finite outputs, |O| <= max|V|
    vmax = float(v.float().abs().max())
    assert np.all(np.isfinite(lse)) and np.abs(o).max() <= vmax * (1 + 1e-2)


def test_prefill_every_row_mha_causal_S4096():
    """Causal MHA, B=8, H=16, S=4096 (one of the pages' prefill configurations) compared
    with the oracle on all 524288 rows, one batch entry at a time."""
    name = "mha_causal_S4096"
    w = inp.WORKLOADS[name]
    q, k, v, bits = w.make(w.seed(list(inp.WORKLOADS).index(name)))
    o, lse = run_cuda(q, k, v, bits, w.causal, w.scale)
    per_b = w.Hq * w.S
    for b in range(w.B):
        rows = np.arange(b * per_b, (b + 1) * per_b, dtype=np.int64)
        o_ref, lse_ref = oracle_rows(q, k, v, bits, w.causal, w.scale, w.dtype, rows)
        assert_close(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, f"{name} b={b}")


def test_packed_workload_sampled_parity():
    """The packed variable-length causal batch of the benchmark's sweep (8 entries of 1k-16k
    rows, GQA 32/8), launched as bench.py launches it, checked entry by entry against the
    oracle on a stratified row sample of every head."""
    import attention_forward_07_gb300 as af
    pw = inp.PACKED_WORKLOADS["packed_causal_gqa8"]
    q, k, v, cu = pw.make(1000 + len(pw.lengths))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((pw.Hq, pw.total), float("nan"), dtype=torch.float32, device="cuda")
    mx = max(pw.lengths)
    af.attn_fwd_packed(qd, kd, vd, o, torch.from_numpy(cu).cuda(), torch.from_numpy(cu).cuda(), mx, mx, lse=lse,
                       causal=True, scale=pw.scale)
    af.attn_check()
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    for b, s in enumerate(pw.lengths):
        lo = int(cu[b])
        qb = q[:, lo:lo + s].unsqueeze(0).contiguous()
        kb = k[:, lo:lo + s].unsqueeze(0).contiguous()
        vb = v[:, lo:lo + s].unsqueeze(0).contiguous()
        rows = stratified_rows(1, pw.Hq, s, seed=s)
        o_ref, lse_ref = oracle_rows(qb, kb, vb, None, True, pw.scale, pw.dtype, rows)
        h, i = rows // s, rows % s
        assert_close(og[h, lo + i], lg[h, lo + i], o_ref, lse_ref, f"packed entry {b} (length {s})")


@pytest.mark.parametrize("name", list(inp.EX_WORKLOADS))
def test_ex_workloads_sampled_parity(name):
    """The attn_fwd_ex cases of the benchmark's sweep, launched as bench.py launches them,
    against the oracle's extended definition on a stratified row sample of every head."""
    import attention_forward_07_gb300 as af
    xw = inp.EX_WORKLOADS[name]
    q, k, v, bits = xw.make(2000 + xw.Sq % 1000)
    dev = "cuda"
    md = None if bits is None else torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).to(dev)
    o = torch.full((xw.B, xw.Hq, xw.Sq, xw.d), float("nan"), dtype=q.dtype, device=dev)
    lse = torch.full((xw.B, xw.Hq, xw.Sq), float("nan"), dtype=torch.float32, device=dev)
    af.attn_fwd_ex(q.to(dev), k.to(dev), v.to(dev), o, lse, md, xw.per_head_mask, xw.causal, xw.window_left, -1,
                   xw.scale)
    af.attn_check()
    rows = stratified_rows(xw.B, xw.Hq, xw.Sq, seed=xw.Sq)
    o_ref, lse_ref = oracle.attn_rows_ex(inp.as_u16(q), inp.as_u16(k), inp.as_u16(v), xw.dtype, rows, bits,
                                         xw.per_head_mask, xw.causal, xw.window_left, -1, xw.scale)
    og = o.float().cpu().numpy().astype(np.float64).reshape(-1, xw.d)
    lg = lse.cpu().numpy().astype(np.float64).reshape(-1)
    assert_close(og[rows], lg[rows], o_ref, lse_ref, name)
