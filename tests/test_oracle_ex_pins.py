"""Pins for the oracle's extended definition: Sq <= Sk aligned bottom-right, a band of
kept keys (window_left / window_right), per-head custom masks.  Each is tied to the
already-pinned base definition or to a closed form, not to a re-typed formula."""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_07_gb300 import inputs as inp


def _u16(t):
    return inp.as_u16(t)


def _f64(t):
    return t.to(torch.float64)


def test_reduces_to_base_definition():
    B, Hq, Hkv, S, d = 2, 4, 2, 77, 16
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, inp.BF16, 3)
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, 3))
    for causal in (False, True):
        a = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.BF16, bits, causal, 0.2)
        b = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.BF16, None, bits, False, causal, -1, -1, 0.2)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bottom_right_alignment_is_the_tail_of_the_square_problem():
    """Queries Sk-Sq .. Sk-1 of a square causal problem are exactly the Sq < Sk problem
    (prefill of the last Sq tokens against a cache of Sk keys)."""
    B, Hq, Hkv, Sk, Sq, d = 2, 2, 1, 90, 33, 8
    q_full, k, v = inp.qkv(B, Hq, Hkv, Sk, d, inp.F16, 5)
    q = q_full[:, :, Sk - Sq:].contiguous()
    full = oracle.attn_fwd(_u16(q_full), _u16(k), _u16(v), inp.F16, None, True, 0.3)
    part = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.F16, None, None, False, True, -1, -1, 0.3)
    assert np.array_equal(part[0], full[0][:, :, Sk - Sq:]) and np.array_equal(part[1], full[1][:, :, Sk - Sq:])


def test_zero_width_band_keeps_the_aligned_diagonal_exactly():
    """window_left = window_right = 0: row i keeps only key i + Sk - Sq, so O is that V row
    bit for bit and LSE is its score (small integers keep the score exact)."""
    B, H, Sq, Sk, d = 1, 2, 10, 25, 4
    rng = np.random.default_rng(4)
    q = torch.tensor(rng.integers(-3, 4, (B, H, Sq, d)), dtype=torch.float32).to(torch.float16)
    k = torch.tensor(rng.integers(-3, 4, (B, H, Sk, d)), dtype=torch.float32).to(torch.float16)
    _, _, v = inp.qkv(B, H, H, Sk, d, inp.F16, 6)
    o, lse = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.F16, None, None, False, False, 0, 0, 0.5)
    for i in range(Sq):
        j = i + Sk - Sq
        assert np.array_equal(o[0, :, i], _f64(v)[0, :, j].numpy())
        assert np.array_equal(lse[0, :, i], 0.5 * (_f64(q)[0, :, i] * _f64(k)[0, :, j]).sum(-1).numpy())


def test_band_equals_the_same_band_as_custom_words():
    B, Hq, S, d = 2, 2, 70, 8
    q, k, v = inp.qkv(B, Hq, Hq, S, d, inp.F16, 7)
    wl, wr = 9, 3
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    band = np.broadcast_to((j >= i - wl) & (j <= i + wr), (B, S, S))
    bits = inp.pack_bits(band)
    a = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.F16, None, None, False, False, wl, wr, 0.25)
    b = oracle.attn_fwd(_u16(q), _u16(k), _u16(v), inp.F16, bits, False, 0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # and the skip maps agree
    m1 = oracle.skip_map_ex(None, False, B, Hq, S, S, False, wl, wr, 16, 16)
    m2 = oracle.skip_map(bits, B, S, False, 16, 16)
    assert np.array_equal(m1, m2)


def test_wide_band_is_no_band_and_causal_is_right_band_zero():
    B, H, Sq, Sk, d = 1, 2, 40, 64, 8
    q, k, v = inp.qkv(B, H, H, Sk, d, inp.BF16, 8)
    q = q[:, :, :Sq].contiguous()
    a = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.BF16, None, None, False, True, -1, -1, 0.2)
    b = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.BF16, None, None, False, False, 10 ** 6, 0, 0.2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_per_head_masks():
    B, Hq, Hkv, S, d = 2, 4, 2, 50, 8
    q, k, v = inp.qkv(B, Hq, Hkv, S, d, inp.F16, 9)
    shared = inp.pack_bits(inp.bernoulli_mask(B, S, 9))
    per_head = np.repeat(shared[:, None], Hq, axis=1)
    a = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.F16, None, shared, False, True, -1, -1, 0.3)
    b = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.F16, None, per_head, True, True, -1, -1, 0.3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # distinct heads: head h keeps only column (i + 7h) mod S -> that V row exactly
    keep = torch.zeros((B, Hq, S, S), dtype=torch.bool)
    for h in range(Hq):
        keep[:, h, torch.arange(S), (torch.arange(S) + 7 * h) % S] = True
    bits = inp.pack_bits(keep.reshape(B * Hq, S, S)).reshape(B, Hq, S, -1)
    o, _ = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.F16, None, bits, True, False, -1, -1, 0.3)
    vv = _f64(v).repeat_interleave(Hq // Hkv, dim=1).numpy()
    for h in range(Hq):
        cols = (np.arange(S) + 7 * h) % S
        assert np.array_equal(o[:, h], vv[:, h, cols])


def test_extended_matches_torch_sdpa():
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 37, 61, 16
    q, k, v = inp.qkv(B, Hq, Hkv, Sk, d, inp.BF16, 10)
    q = q[:, :, :Sq].contiguous()
    keep = inp.bernoulli_mask(B * Hq, Sk, 10)[:, :Sq, :].reshape(B, Hq, Sq, Sk)
    bits = inp.pack_bits(keep.reshape(B * Hq, Sq, Sk)).reshape(B, Hq, Sq, -1)
    wl, wr = 20, 5
    pos = np.arange(Sq)[:, None] + Sk - Sq
    j = np.arange(Sk)[None, :]
    band = torch.from_numpy((j >= pos - wl) & (j <= pos + wr) & (j <= pos))
    allowed = keep & band
    o, lse = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.BF16, None, bits, True, True, wl, wr, 0.3)
    g = Hq // Hkv
    kk, vv = _f64(k).repeat_interleave(g, 1), _f64(v).repeat_interleave(g, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(_f64(q), kk, vv, attn_mask=allowed, scale=0.3).numpy()
    sc = (torch.matmul(_f64(q), kk.transpose(-1, -2)) * 0.3).masked_fill(~allowed, float("-inf"))
    lref = torch.logsumexp(sc, -1).numpy()
    ok = allowed.any(-1).numpy()
    np.testing.assert_allclose(o[ok], ref[ok], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse[ok], lref[ok], rtol=1e-12, atol=1e-12)
    assert np.all(o[~ok] == 0) and np.all(np.isneginf(lse[~ok]))


def test_varlen_entries_equal_separate_problems():
    """Each batch entry with its own lengths equals the same entry run alone at those lengths
    (which the pins above tie to the base definition); padded rows have no value."""
    B, Hq, Hkv, Sq, Sk, d = 3, 2, 1, 40, 70, 8
    q, k, v = inp.qkv(B, Hq, Hkv, Sk, d, inp.BF16, 12)
    q = q[:, :, :Sq].contiguous()
    lq = np.array([40, 17, 0], np.int32)
    lk = np.array([70, 25, 9], np.int32)
    keep = inp.bernoulli_mask(B, Sk, 12)[:, :Sq]
    bits = inp.pack_bits(keep)
    for causal, wl, wr, mb in ((True, -1, -1, None), (False, 6, 2, bits), (True, 11, -1, bits)):
        o, lse = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.BF16, None, mb, False, causal, wl, wr, 0.3,
                                     seqlens_q=lq, seqlens_k=lk)
        for b in range(B):
            sq, sk = int(lq[b]), int(lk[b])
            assert np.all(np.isnan(lse[b, :, sq:])) and np.all(np.isnan(o[b, :, sq:]))
            if sq == 0:
                continue
            qb = q[b:b + 1, :, :sq].contiguous()
            kb, vb = k[b:b + 1, :, :sk].contiguous(), v[b:b + 1, :, :sk].contiguous()
            mbb = None if mb is None else inp.pack_bits(keep[b:b + 1, :sq, :sk])
            if sk >= sq:
                ref = oracle.attn_rows_ex(_u16(qb), _u16(kb), _u16(vb), inp.BF16, None, mbb, False, causal, wl, wr, 0.3)
                assert np.array_equal(o[b:b + 1, :, :sq], ref[0]) and np.array_equal(lse[b:b + 1, :, :sq], ref[1])
        # the skip map agrees with the rows that have a kept entry
        m = oracle.skip_map_ex(mb, False, B, Hq, Sq, Sk, causal, wl, wr, 16, 16, seqlens_q=lq, seqlens_k=lk)
        assert m.shape == (B, 3, 5)
        assert not m[2].any()  # entry 2 has no query rows


def test_varlen_short_keys_make_early_rows_empty_under_causal():
    """sk_b < sq_b: query i sits at key position i + sk_b - sq_b < 0 for the first rows, so
    under causal they keep nothing (O = 0, LSE = -inf); later rows match the tail problem."""
    B, H, Sq, Sk, d = 1, 1, 12, 12, 4
    q, k, v = inp.qkv(B, H, H, Sk, d, inp.F16, 13)
    o, lse = oracle.attn_rows_ex(_u16(q), _u16(k), _u16(v), inp.F16, None, None, False, True, -1, -1, 0.5,
                                 seqlens_q=np.array([10], np.int32), seqlens_k=np.array([6], np.int32))
    assert np.all(np.isneginf(lse[0, 0, :4])) and np.all(o[0, 0, :4] == 0)
    tail = oracle.attn_rows_ex(_u16(q[:, :, 4:10].contiguous()), _u16(k[:, :, :6].contiguous()),
                               _u16(v[:, :, :6].contiguous()), inp.F16, None, None, False, True, -1, -1, 0.5)
    assert np.array_equal(o[:, :, 4:10], tail[0]) and np.array_equal(lse[:, :, 4:10], tail[1])


def test_expected_visited_compaction_helper():
    """The helper that states the kernel's visited map under custom masks: with no empty
    16-row block it is the plain (128, 128) block map; with empty blocks it is built over
    the compacted rows (live blocks in ascending order, eight per tile)."""
    from gpu_util import expected_visited
    B, Hq, S = 2, 3, 300
    bits = inp.pack_bits(inp.bernoulli_mask(B, S, 5))
    got = expected_visited(bits, False, B, Hq, S, S, True)
    ref = oracle.skip_map(bits, B, S, True, 128, 128)
    assert np.array_equal(got, np.repeat(ref[:, None], Hq, axis=1))
    keep = np.zeros((1, S, S), bool)
    keep[0, 2 * 16 + 3, 10] = True     # block 2 -> key tile 0
    keep[0, 5 * 16 + 9, 200] = True    # block 5 -> key tile 1
    keep[0, 17 * 16 + 1, 290] = True   # block 17 -> key tile 2
    bits = inp.pack_bits(keep)
    got = expected_visited(bits, False, 1, 1, S, S, False)
    want = np.zeros((1, 1, 3, 3), np.uint8)
    want[0, 0, 0] = 1                  # all three live blocks land in compacted tile 0
    assert np.array_equal(got, want)
    plain = oracle.skip_map(bits, 1, S, False, 128, 128)
    assert plain[0, 0].tolist() == [1, 1, 0] and plain[0, 2].tolist() == [0, 0, 1]
