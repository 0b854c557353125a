"""Pins for the oracle's block-emptiness map under the extended rule (oracle.skip_map_ex).

The map says, for every (mask row block, query tile, key tile), whether the block holds a
kept entry: the tile-skip rule of the page "Opus 4.6 + AutoResearch驱动25轮迭代..." (first
code excerpt, the warp ballot over a tile's mask words) applied to the kept set of
ordinary attention (page "NVIDIA让AI狂肝7天自己写算子", FlashAttention-lineage section) with
this library's extensions: Sq <= Sk aligned at the bottom right, a key band, per-head
masks and per-entry lengths inside padded buffers.

Each expected map here is built independently of the oracle: the kept matrix is written
out in numpy from the definition (query i of entry b sits at key position
i + sk_b - sq_b; rows >= sq_b and keys >= sk_b do not exist), the mask words are unpacked
with inputs.unpack_bits, and the matrix is reduced over (bm, bn) blocks.  The cases are
chosen so that a slip in any index of the oracle's loop -- the alignment offset, the row
or key bound, the mask row of a per-head mask -- changes at least one block.
"""
import numpy as np
import pytest

import oracle
from attention_forward_07_gb300 import inputs as inp


def kept_matrix(bits, per_head, B, Hq, Sq, Sk, causal, wl, wr, lens_q, lens_k):
    """bool [B*Hm, Sq, Sk]: the kept entries, straight from the definition."""
    Hm = Hq if (bits is not None and per_head) else 1
    out = np.zeros((B * Hm, Sq, Sk), bool)
    if bits is not None:
        words = np.asarray(bits, dtype=np.uint32).reshape(B * Hm, Sq, -1)
        mask = inp.unpack_bits(words, Sk)
    for mb in range(B * Hm):
        b = mb // Hm
        sq = Sq if lens_q is None else int(lens_q[b])
        sk = Sk if lens_k is None else int(lens_k[b])
        i = np.arange(Sq)[:, None]
        j = np.arange(Sk)[None, :]
        pos = i + (sk - sq)
        keep = (i < sq) & (j < sk)
        if causal:
            keep &= j <= pos
        if wl >= 0:
            keep &= j >= pos - wl
        if wr >= 0:
            keep &= j <= pos + wr
        if bits is not None:
            keep &= mask[mb]
        out[mb] = keep
    return out


def block_reduce(keep, bm, bn):
    n, Sq, Sk = keep.shape
    nqt, nkt = -(-Sq // bm), -(-Sk // bn)
    pad = np.zeros((n, nqt * bm, nkt * bn), bool)
    pad[:, :Sq, :Sk] = keep
    return pad.reshape(n, nqt, bm, nkt, bn).any(axis=(2, 4)).astype(np.uint8)


def expected(bits, per_head, B, Hq, Sq, Sk, causal, wl, wr, bm, bn, lens_q=None, lens_k=None):
    return block_reduce(kept_matrix(bits, per_head, B, Hq, Sq, Sk, causal, wl, wr, lens_q, lens_k), bm, bn)


def _mask(n, Sq, Sk, seed, p_keep):
    """Random kept bits [n, Sq, ceil(Sk/32)] (a rectangular Bernoulli mask)."""
    rng = np.random.default_rng(seed)
    return inp.pack_bits(rng.random((n, Sq, Sk)) < p_keep)


CASES = [
    # B, Hq, Sq, Sk, causal, wl, wr, mask ("none" | "shared" | "head"), p_keep, lens, bm, bn
    (2, 1, 40, 100, True, -1, -1, "none", 0, None, 8, 16),                # Sq < Sk, causal
    (2, 1, 37, 90, False, 5, 2, "none", 0, None, 8, 8),                   # band, ragged tiles
    (1, 1, 20, 64, True, 3, -1, "none", 0, None, 4, 4),                   # causal window
    (2, 3, 33, 70, False, -1, -1, "head", 0.03, None, 8, 16),             # per-head masks
    (2, 3, 33, 70, True, 12, -1, "head", 0.2, None, 16, 8),               # per-head + causal window
    (3, 1, 40, 70, True, -1, -1, "none", 0, ([40, 17, 0], [70, 25, 9]), 8, 8),      # sq_b = 0
    (3, 1, 24, 40, True, -1, -1, "none", 0, ([20, 24, 9], [6, 40, 3]), 4, 8),       # sk_b < sq_b
    (3, 2, 48, 80, True, 6, -1, "head", 0.1, ([48, 30, 5], [33, 80, 12]), 8, 16),   # lengths + heads
    (2, 1, 50, 50, False, 4, 4, "shared", 0.05, ([50, 21], [50, 44]), 16, 16),      # Sq = Sk, lens
    (2, 2, 64, 96, False, -1, 0, "shared", 0.1, ([64, 31], [96, 40]), 16, 32),      # right band 0
    (2, 1, 30, 96, False, -1, -1, "none", 0, ([30, 12], [96, 40]), 8, 16),          # key bound alone
    (2, 2, 30, 96, False, 20, -1, "shared", 0.9, ([30, 12], [96, 40]), 8, 16),      # bits past sk_b
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Sq{}_Sk{}_c{}_w{}_{}_{}_lens{}_{}x{}".format(
    c[0], c[1], c[2], c[3], int(c[4]), c[5], c[6], c[7], int(c[9] is not None), c[10], c[11]))
def test_skip_map_ex_against_the_kept_matrix(case):
    B, Hq, Sq, Sk, causal, wl, wr, mk, p_keep, lens, bm, bn = case
    per_head = mk == "head"
    bits = None
    if mk == "shared":
        bits = _mask(B, Sq, Sk, Sq * Sk, p_keep)
    elif mk == "head":
        bits = _mask(B * Hq, Sq, Sk, Sq + Sk, p_keep).reshape(B, Hq, Sq, -1)
    lq = lk = None
    if lens is not None:
        lq, lk = np.array(lens[0], np.int32), np.array(lens[1], np.int32)
    got = oracle.skip_map_ex(bits, per_head, B, Hq, Sq, Sk, causal, wl, wr, bm, bn, seqlens_q=lq, seqlens_k=lk)
    want = expected(bits, per_head, B, Hq, Sq, Sk, causal, wl, wr, bm, bn, lq, lk)
    assert got.shape == want.shape
    assert np.array_equal(got, want)
    # the case is informative: some blocks are kept and some are empty
    assert 0 < int(want.sum()) < want.size


def test_per_entry_alignment_is_each_entrys_own():
    """Entry 1 has sq_b = 8, sk_b = 8 inside Sq = 8, Sk = 64: its last query sits at key 7,
    not at key 63, so under causal only key tile 0 is kept; entry 0 (full lengths) reaches
    key tile 7.  An offset taken from the padded shape (Sk - Sq) would keep entry 1's
    tile 7."""
    got = oracle.skip_map_ex(None, False, 2, 1, 8, 64, True, 0, 0, 8, 8,
                             seqlens_q=np.array([8, 8], np.int32), seqlens_k=np.array([64, 8], np.int32))
    assert got.shape == (2, 1, 8)
    assert got[0, 0].tolist() == [0, 0, 0, 0, 0, 0, 0, 1]
    assert got[1, 0].tolist() == [1, 0, 0, 0, 0, 0, 0, 0]


def test_rows_past_the_entry_length_keep_nothing():
    """sq_b = 5 in a padded Sq = 16: query tiles past row 4 are empty for every key tile
    even without a mask (a row bound taken from Sq would keep them)."""
    got = oracle.skip_map_ex(None, False, 1, 1, 16, 16, False, -1, -1, 4, 4,
                             seqlens_q=np.array([5], np.int32), seqlens_k=np.array([16], np.int32))
    assert got[0, :, :].tolist() == [[1, 1, 1, 1], [1, 1, 1, 1], [0, 0, 0, 0], [0, 0, 0, 0]]


def test_per_head_mask_rows_are_the_heads_own():
    """Head h of entry b keeps only key column 8*h + 4*b (one bit per row), so block
    (b*Hq + h, qt, kt) is kept iff kt == 2*h + b (bn = 4): the mask row of a per-head mask is
    (b*Hq + h), not b or h alone."""
    B, Hq, Sq, Sk, bn = 2, 3, 8, 32, 4
    keep = np.zeros((B, Hq, Sq, Sk), bool)
    for b in range(B):
        for h in range(Hq):
            keep[b, h, :, 8 * h + 4 * b] = True
    bits = inp.pack_bits(keep.reshape(B * Hq, Sq, Sk)).reshape(B, Hq, Sq, -1)
    got = oracle.skip_map_ex(bits, True, B, Hq, Sq, Sk, False, -1, -1, 4, bn)
    for b in range(B):
        for h in range(Hq):
            row = [1 if kt == 2 * h + b else 0 for kt in range(Sk // bn)]
            assert got[b * Hq + h, 0].tolist() == row and got[b * Hq + h, 1].tolist() == row
