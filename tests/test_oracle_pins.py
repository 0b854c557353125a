"""Pins for the fp64 oracle: it is checked against things other than itself.

* library routines: torch's scaled_dot_product_attention / logsumexp in fp64,
  numpy / torch half and bfloat16 conversions;
* closed forms: zero keys (uniform weights), one kept column per row, two keys,
  one-hot values (O equals the weight matrix);
* invariants: causal == lower-triangular custom mask, GQA == replicated MHA,
  key permutation, a shift added to every key, S = 1, fully masked rows,
  mask bits past column S-1 ignored;
* the tile-emptiness map against a numpy block reduction of the unpacked mask;
* the golden fixtures under tests/golden/.

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, a
sign, a transposed operand, a wrong head mapping, reversed bit order, the
causal triangle the wrong way round) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from attention_forward_07_gb300 import inputs as inp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _u16(t):
    return inp.as_u16(t)


def _f64(t):
    return t.to(torch.float64)


def _library_attention(q, k, v, keep, scale):
    """torch fp64 SDPA with a boolean mask (K/V heads repeated for GQA)."""
    g = q.shape[1] // k.shape[1]
    kk = _f64(k).repeat_interleave(g, dim=1)
    vv = _f64(v).repeat_interleave(g, dim=1)
    qq = _f64(q)
    mask = keep[:, None, :, :]
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    scores = torch.matmul(qq, kk.transpose(-1, -2)) * scale
    scores = scores.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)
    return o.numpy(), lse.numpy()


# ----------------------------------------------------------------------------- widening

def test_widen_f16_all_words_match_numpy():
    words = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = words.view(np.float16).astype(np.float64)
    got = np.array([oracle.widen(int(w), oracle.F16) for w in words])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_widen_bf16_all_words_match_torch():
    words = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(words.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.widen(int(w), oracle.BF16) for w in words])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# ----------------------------------------------------------------------------- library routine

@pytest.mark.parametrize("B,Hq,Hkv,S,d,dtype,causal,maskkind", [
    (2, 2, 2, 37, 8, inp.F16, False, "bernoulli"),
    (1, 4, 2, 45, 16, inp.BF16, True, "none"),
    (2, 4, 1, 33, 8, inp.BF16, True, "bernoulli"),
    (1, 2, 2, 70, 4, inp.F16, False, "none"),
    (2, 6, 3, 64, 8, inp.F16, True, "block90"),
])
def test_matches_torch_sdpa_fp64(B, Hq, Hkv, S, d, dtype, causal, maskkind):
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, dtype, seed=11 + S)
    if maskkind == "bernoulli":
        keep = inp.bernoulli_mask(B, S, seed=3)
    elif maskkind == "block90":
        keep = inp.block_sparse_mask(B, S, seed=4)
    else:
        keep = torch.ones((B, S, S), dtype=torch.bool)
    bits = inp.pack_bits(keep) if maskkind != "none" else None
    if causal:
        keep = keep & torch.tril(torch.ones((S, S), dtype=torch.bool))
    scale = 0.3 if d != 8 else float(np.float32(1 / math.sqrt(d)))
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), dtype, bits, causal, scale)
    o_ref, lse_ref = _library_attention(q, k, v, keep, scale)
    rows_ok = keep.any(dim=-1).numpy()[:, None, :].repeat(Hq, axis=1)
    assert rows_ok.any()
    np.testing.assert_allclose(o[rows_ok], o_ref[rows_ok], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse[rows_ok], lse_ref[rows_ok], rtol=1e-12, atol=1e-12)
    # rows with nothing kept: defined as O = 0, LSE = -inf
    assert np.all(o[~rows_ok] == 0.0)
    assert np.all(np.isneginf(lse[~rows_ok]))


# ----------------------------------------------------------------------------- closed forms

def _exact_tensor(vals, dtype):
    return torch.tensor(vals, dtype=torch.float32).to(inp.TORCH_DTYPE[dtype])


def test_zero_keys_give_uniform_weights():
    """All scores 0: O_i is the mean of the kept V rows and LSE_i = ln(#kept)."""
    B, H, S, d = 1, 1, 40, 4
    q, _, v = inp.qkv(B, H, H, S, d, inp.F16, seed=5)
    k = torch.zeros_like(q)
    keep = inp.bernoulli_mask(B, S, seed=9, p_keep=0.3)
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, inp.pack_bits(keep), False, 0.5)
    vv = _f64(v)[0, 0].numpy()
    for i in range(S):
        kept = keep[0, i].numpy()
        if not kept.any():
            assert np.isneginf(lse[0, 0, i])
            continue
        assert lse[0, 0, i] == pytest.approx(math.log(kept.sum()), abs=1e-14)
        np.testing.assert_allclose(o[0, 0, i], vv[kept].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_one_kept_column_returns_that_row_exactly():
    """One kept column j* per row: O_i = v_{j*} bit for bit, LSE_i = s_{i j*}.
    Small-integer Q, K and a power-of-two scale make s exact in double."""
    B, H, S, d = 1, 2, 24, 8
    rng = np.random.default_rng(1)
    q = _exact_tensor(rng.integers(-4, 5, size=(B, H, S, d)).tolist(), inp.BF16)
    k = _exact_tensor(rng.integers(-4, 5, size=(B, H, S, d)).tolist(), inp.BF16)
    _, _, v = inp.qkv(B, H, H, S, d, inp.BF16, seed=2)
    perm = rng.permutation(S)
    keep = torch.zeros((B, S, S), dtype=torch.bool)
    keep[0, torch.arange(S), torch.from_numpy(perm)] = True
    scale = 0.125
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.BF16, inp.pack_bits(keep), False, scale)
    qn, kn, vn = _f64(q).numpy(), _f64(k).numpy(), _f64(v).numpy()
    for h in range(H):
        for i in range(S):
            j = perm[i]
            assert np.array_equal(o[0, h, i], vn[0, h, j])
            assert lse[0, h, i] == scale * float(np.dot(qn[0, h, i], kn[0, h, j]))


def test_two_keys_closed_form():
    """S = 2, d = 1, no mask: row i weights are a logistic function of s_i0 - s_i1."""
    q = _exact_tensor([[[[1.5], [-2.0]]]], inp.F16)
    k = _exact_tensor([[[[0.75], [-0.5]]]], inp.F16)
    v = _exact_tensor([[[[3.0], [-1.25]]]], inp.F16)
    scale = 0.5
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, None, False, scale)
    for i, qi in enumerate((1.5, -2.0)):
        s0, s1 = scale * qi * 0.75, scale * qi * -0.5
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        assert o[0, 0, i, 0] == pytest.approx(w0 * 3.0 + (1 - w0) * -1.25, rel=1e-14)
        assert lse[0, 0, i] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), rel=1e-14)


def test_one_hot_values_expose_the_weight_matrix():
    """V = identity (d = S): O is the softmax weight matrix itself, so every row sums to 1,
    masked entries are exactly 0, and kept ratios equal exp(s_ij - s_ik)."""
    B, H, S = 1, 1, 32
    q, k, _ = inp.qkv(B, H, H, S, S, inp.F16, seed=8)
    v = torch.eye(S, dtype=torch.float16)[None, None]
    keep = inp.bernoulli_mask(B, S, seed=10, p_keep=0.6)
    keep[0, :, 0] = True  # every row keeps at least column 0
    scale = 0.2
    o, _ = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, inp.pack_bits(keep), False, scale)
    w = o[0, 0]
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(w[~keep[0].numpy()] == 0.0)
    assert np.all(w >= 0.0)
    s = scale * (_f64(q)[0, 0] @ _f64(k)[0, 0].T).numpy()
    for i in range(S):
        kept = np.nonzero(keep[0, i].numpy())[0]
        for j in kept[1:]:
            assert w[i, j] / w[i, 0] == pytest.approx(math.exp(s[i, j] - s[i, 0]), rel=1e-12)


# ----------------------------------------------------------------------------- invariants

def test_causal_equals_lower_triangular_custom_mask():
    B, H, S, d = 2, 2, 50, 16
    q, k, v = inp.qkv(B, H, H, S, d, inp.BF16, seed=21)
    tri = torch.tril(torch.ones((S, S), dtype=torch.bool)).expand(B, S, S)
    a = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.BF16, None, True, 0.25)
    b = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.BF16, inp.pack_bits(tri), False, 0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # and the triangle is the right way round: row 0 sees only key 0
    np.testing.assert_array_equal(a[0][:, :, 0], _f64(v)[:, :, 0].numpy())


def test_gqa_equals_replicated_mha():
    B, Hq, Hkv, S, d = 2, 6, 2, 30, 8
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, inp.F16, seed=31)
    g = Hq // Hkv
    kr, vr = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, seed=1))
    a = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, bits, True, 0.3)
    b = oracle.attn_fwd(_u16(q), _u16(kr), _u16(vr), inp.F16, bits, True, 0.3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_key_permutation_invariance():
    B, H, S, d = 1, 2, 41, 8
    q, k, v = inp.qkv(B, H, H, S, d, inp.BF16, seed=41)
    keep = inp.bernoulli_mask(B, S, seed=2)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(S))
    a = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.BF16, inp.pack_bits(keep), False, 0.35)
    b = oracle.attn_fwd(_u16(q), _u16(k[:, :, perm].contiguous()), _u16(v[:, :, perm].contiguous()),
                        inp.BF16, inp.pack_bits(keep[:, :, perm]), False, 0.35)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13, atol=1e-13)


def test_key_shift_moves_lse_only():
    """Adding u to every key adds scale*<q_i,u> to every score of row i: O is unchanged and
    LSE moves by exactly that amount (small integers keep everything exact)."""
    B, H, S, d = 1, 1, 20, 4
    rng = np.random.default_rng(5)
    qi = rng.integers(-3, 4, size=(B, H, S, d))
    ki = rng.integers(-3, 4, size=(B, H, S, d))
    u = np.array([1, -2, 0, 3])
    q = _exact_tensor(qi.tolist(), inp.F16)
    k0 = _exact_tensor(ki.tolist(), inp.F16)
    k1 = _exact_tensor((ki + u).tolist(), inp.F16)
    _, _, v = inp.qkv(B, H, H, S, d, inp.F16, seed=6)
    scale = 0.25
    o0, l0 = oracle.attn_fwd(_u16(q), _u16(k0), _u16(v), inp.F16, None, True, scale)
    o1, l1 = oracle.attn_fwd(_u16(q), _u16(k1), _u16(v), inp.F16, None, True, scale)
    np.testing.assert_allclose(o1, o0, rtol=1e-13, atol=1e-14)
    shift = scale * (qi[0, 0] @ u)
    np.testing.assert_allclose(l1[0, 0] - l0[0, 0], shift, rtol=0, atol=1e-12)


def test_constant_keys_average_kept_values():
    B, H, S, d = 1, 1, 33, 8
    q, k, v = inp.qkv(B, H, H, S, d, inp.BF16, seed=51)
    k = k[:, :, :1].expand(B, H, S, d).contiguous()
    keep = inp.bernoulli_mask(B, S, seed=52)
    o, _ = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.BF16, inp.pack_bits(keep), False, 0.4)
    vv = _f64(v)[0, 0].numpy()
    for i in range(S):
        kept = keep[0, i].numpy()
        if kept.any():
            np.testing.assert_allclose(o[0, 0, i], vv[kept].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_single_key():
    q, k, v = inp.qkv(1, 3, 3, 1, 8, inp.F16, seed=61)
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, None, True, 0.5)
    assert np.array_equal(o, _f64(v).numpy())
    s = 0.5 * (_f64(q) * _f64(k)).sum(-1).numpy()
    np.testing.assert_allclose(lse, s, rtol=1e-15, atol=0)


def test_fully_masked_rows_are_zero_and_neg_inf():
    B, H, S, d = 1, 2, 40, 8
    q, k, v = inp.qkv(B, H, H, S, d, inp.F16, seed=71)
    keep = inp.bernoulli_mask(B, S, seed=72)
    keep[0, 5] = False
    keep[0, 17] = False
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, inp.pack_bits(keep), False, 0.3)
    for i in (5, 17):
        assert np.all(o[0, :, i] == 0) and np.all(np.isneginf(lse[0, :, i]))
    assert np.all(np.isfinite(lse[0, :, 6]))


def test_bits_past_the_last_column_are_ignored():
    B, H, S, d = 1, 1, 45, 8
    q, k, v = inp.qkv(B, H, H, S, d, inp.F16, seed=81)
    keep = inp.bernoulli_mask(B, S, seed=82)
    bits = inp.pack_bits(keep)
    dirty = bits.copy()
    dirty[:, :, -1] |= np.uint32(0xFFFFFFFF) << np.uint32(S % 32)
    a = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, bits, False, 0.3)
    b = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, dirty, False, 0.3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rows_api_matches_full_evaluation():
    B, Hq, Hkv, S, d = 2, 4, 2, 130, 16
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, inp.BF16, seed=91)
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, seed=92))
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.BF16, bits, True, 0.25)
    rows = inp.sample_rows(B, Hq, S, 5, seed=93)
    o2, l2 = oracle.attn_rows(_u16(q), _u16(k), _u16(v), inp.BF16, rows, bits, True, 0.25)
    assert np.array_equal(o.reshape(-1, d)[rows], o2)
    assert np.array_equal(lse.reshape(-1)[rows], l2)


# ----------------------------------------------------------------------------- skip map

@pytest.mark.parametrize("S,causal,kind", [(128, False, "bernoulli"), (300, True, "none"),
                                           (512, False, "block90"), (700, True, "block90"),
                                           (257, False, "none")])
def test_skip_map_matches_block_reduction(S, causal, kind):
    B, bm, bn = 2, 128, 128
    if kind == "none":
        keep = torch.ones((B, S, S), dtype=torch.bool)
        bits = None
    else:
        keep = inp.bernoulli_mask(B, S, seed=5) if kind == "bernoulli" else inp.block_sparse_mask(B, S, seed=6)
        bits = inp.pack_bits(keep)
    k = keep.numpy().copy()
    if causal:
        k &= np.tril(np.ones((S, S), dtype=bool))
    nqt, nkt = -(-S // bm), -(-S // bn)
    pad = np.zeros((B, nqt * bm, nkt * bn), dtype=bool)
    pad[:, :S, :S] = k
    ref = pad.reshape(B, nqt, bm, nkt, bn).any(axis=(2, 4)).astype(np.uint8)
    got = oracle.skip_map(bits, B, S, causal, bm, bn)
    assert np.array_equal(got, ref)


def test_block90_mask_has_empty_tiles_at_64_rows():
    keep = inp.block_sparse_mask(4, 512, seed=1)
    frac = 1.0 - keep.float().mean().item()
    assert 0.87 < frac < 0.93


# ----------------------------------------------------------------------------- golden fixtures

def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_golden_mask_bit_order():
    """The first page's in-register mask excerpt tests bit (c % 32) of word c / 32."""
    for word_hex, kept in _read_golden("mask_bit_order.txt"):
        word = int(word_hex, 16)
        cols = [] if kept == "-" else [int(c) for c in kept.split(",")]
        words = np.array([[[word]]], dtype=np.uint32)
        assert sorted(np.nonzero(inp.unpack_bits(words, 32)[0, 0])[0].tolist()) == cols
        # the oracle reads the same bits: keys outside `cols` get zero weight
        S = 32
        q = torch.zeros((1, 1, S, 32), dtype=torch.float16)
        k = torch.zeros_like(q)
        v = torch.eye(S, dtype=torch.float16)[None, None]
        mask = np.repeat(words, S, axis=1)
        o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, mask, False, 1.0)
        if cols:
            assert sorted(np.nonzero(o[0, 0, 0])[0].tolist()) == cols
        else:
            assert np.isneginf(lse[0, 0, 0])


def test_golden_tiny_regression():
    """Oracle outputs for a tiny seeded case, written by tests/golden/make_tiny_oracle.py."""
    import json
    with open(os.path.join(GOLDEN, "tiny_oracle.json")) as f:
        data = json.load(f)
    B, Hq, Hkv, S, d = data["shape"]
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, inp.F16, seed=data["seed"])
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, seed=data["seed"]))
    o, lse = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, bits, data["causal"], data["scale"])
    o_ref = np.array([float.fromhex(x) for x in data["o"]]).reshape(o.shape)
    lse_ref = np.array([float.fromhex(x) for x in data["lse"]]).reshape(lse.shape)
    np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-15)
