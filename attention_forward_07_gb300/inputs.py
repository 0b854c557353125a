"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and packs them into the library's input
formats; it holds none of the attention arithmetic.  Both the CUDA path and the
fp64 oracle consume what it produces.

Recipe (the workloads of the pages' benchmarks, all synthetic):

* Q, K, V ~ N(0, 1) in float32 from ``torch.Generator('cpu').manual_seed(seed)``,
  rounded to fp16 / bf16, laid out ``[B, H, S, d]``;
* custom masks are drawn from a second generator seeded ``seed + 1``;
  ``bernoulli_mask`` keeps each (b, row, col) with probability ``p_keep``;
  ``block_sparse_mask`` zeroes whole 16-row blocks with probability 0.8 and
  fills the others Bernoulli(0.5), for an expected masked fraction of 0.9;
* masks are packed least-significant bit first into uint32 words
  ``[B, S, ceil(S/32)]``, one word per 32 columns, 1 = attend, shared by every
  head of a batch entry.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

F16, BF16 = 0, 1
TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}
DTYPE_NAME = {F16: "f16", BF16: "bf16"}


def qkv(B, Hq, Hkv, S, d, dtype, seed):
    """Q [B,Hq,S,d], K and V [B,Hkv,S,d], N(0,1) rounded to fp16/bf16, on the CPU."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    dt = TORCH_DTYPE[dtype]
    q = torch.randn((B, Hq, S, d), generator=g, dtype=torch.float32).to(dt)
    k = torch.randn((B, Hkv, S, d), generator=g, dtype=torch.float32).to(dt)
    v = torch.randn((B, Hkv, S, d), generator=g, dtype=torch.float32).to(dt)
    return q, k, v


def bernoulli_mask(B, S, seed, p_keep=0.5):
    """bool [B, S, S]: each entry kept with probability p_keep."""
    g = torch.Generator(device="cpu").manual_seed(int(seed) + 1)
    return torch.rand((B, S, S), generator=g) < p_keep


def block_sparse_mask(B, S, seed, block=16, p_zero=0.8, p_keep=0.5):
    """bool [B, S, S]: each block of `block` rows is all-zero with probability p_zero,
    otherwise Bernoulli(p_keep) per entry (expected masked fraction 0.9)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed) + 1)
    nblk = (S + block - 1) // block
    zero = torch.rand((B, nblk), generator=g) < p_zero
    m = torch.rand((B, S, S), generator=g) < p_keep
    rows_zero = zero.repeat_interleave(block, dim=1)[:, :S]
    m[rows_zero] = False
    return m


def pack_bits(mask):
    """bool [B, S, S] -> uint32 [B, S, ceil(S/32)], bit (c % 32) of word c // 32 = mask[.., c]."""
    m = np.asarray(mask.numpy() if isinstance(mask, torch.Tensor) else mask, dtype=bool)
    B, R, C = m.shape
    W = (C + 31) // 32
    padded = np.zeros((B, R, W * 32), dtype=bool)
    padded[:, :, :C] = m
    by = np.packbits(padded, axis=-1, bitorder="little")
    return np.ascontiguousarray(by).view("<u4").reshape(B, R, W).astype(np.uint32)


def unpack_bits(words, S):
    """Inverse of pack_bits: uint32 [B, R, W] -> bool [B, R, S]."""
    w = np.ascontiguousarray(np.asarray(words, dtype="<u4"))
    by = w.view(np.uint8)
    bits = np.unpackbits(by, axis=-1, bitorder="little")
    return bits[:, :, :S].astype(bool)


def as_u16(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit words of a CPU fp16/bf16 tensor as a uint16 numpy array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(B, Hq, S, n_random, seed, fixed=(0, 1, 127, 128)):
    """Flat row ids (b*Hq + hq)*S + i: for every (b, hq) the rows in `fixed` that exist,
    row S-1, and n_random rows drawn from a seeded generator."""
    rng = np.random.default_rng(int(seed) + 7)
    ids = []
    for bh in range(B * Hq):
        rows = {r for r in fixed if r < S} | {S - 1}
        if n_random > 0:
            rows |= set(int(x) for x in rng.integers(0, S, size=n_random))
        ids.extend(bh * S + r for r in sorted(rows))
    return np.asarray(ids, dtype=np.int64)


@dataclass(frozen=True)
class Workload:
    """One benchmark configuration of the pages (shapes, dtype, mask kind)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    d: int
    dtype: int
    causal: bool
    mask: str  # "none" | "bernoulli" | "block90"

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d)))

    def flops(self) -> float:
        """4*B*Hq*S^2*d, halved for causal (the dense count, also for custom masks)."""
        f = 4.0 * self.B * self.Hq * self.S * self.S * self.d
        return f / 2 if self.causal else f

    def seed(self, index: int) -> int:
        return index * 1000 + self.S

    def make(self, seed):
        q, k, v = qkv(self.B, self.Hq, self.Hkv, self.S, self.d, self.dtype, seed)
        if self.mask == "bernoulli":
            bits = pack_bits(bernoulli_mask(self.B, self.S, seed))
        elif self.mask == "block90":
            bits = pack_bits(block_sparse_mask(self.B, self.S, seed))
        else:
            bits = None
        return q, k, v, bits


@dataclass(frozen=True)
class PackedWorkload:
    """A packed variable-length batch (this library's extension of the pages' prefill set):
    entries of the given lengths laid out head-major, q / o [Hq, total, d], k / v
    [Hkv, total, d], entry b at rows cu[b] .. cu[b+1]-1, queries and keys of equal length."""
    name: str
    lengths: tuple
    Hq: int
    Hkv: int
    d: int
    dtype: int
    causal: bool

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def total(self) -> int:
        return int(sum(self.lengths))

    def flops(self) -> float:
        """Sum over entries of 4*Hq*s^2*d, halved for causal (the prefill formula per entry)."""
        f = sum(4.0 * self.Hq * s * s * self.d for s in self.lengths)
        return f / 2 if self.causal else f

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    def make(self, seed):
        """q [Hq, total, d], k and v [Hkv, total, d] (N(0,1), rounded), cu_seqlens int32 [B+1]."""
        q, k, v = qkv(1, self.Hq, self.Hkv, self.total, self.d, self.dtype, seed)
        return q[0].contiguous(), k[0].contiguous(), v[0].contiguous(), self.cu_seqlens()


def _prefill(name, S, Hq, Hkv, causal):
    return Workload(name, 32768 // S, Hq, Hkv, S, 128, BF16, causal, "none")


WORKLOADS = {
    "tiny_masked": Workload("tiny_masked", 1, 2, 2, 128, 64, F16, False, "bernoulli"),
    "short_masked": Workload("short_masked", 16, 16, 16, 512, 64, F16, False, "bernoulli"),
    "short_masked90": Workload("short_masked90", 16, 16, 16, 512, 64, F16, False, "block90"),
}
for _S in (4096, 8192, 16384, 32768):
    WORKLOADS[f"mha_causal_S{_S}"] = _prefill(f"mha_causal_S{_S}", _S, 16, 16, True)
    WORKLOADS[f"mha_S{_S}"] = _prefill(f"mha_S{_S}", _S, 16, 16, False)
    for _hkv in (4, 8):
        WORKLOADS[f"gqa{_hkv}_causal_S{_S}"] = _prefill(f"gqa{_hkv}_causal_S{_S}", _S, 32, _hkv, True)
        WORKLOADS[f"gqa{_hkv}_S{_S}"] = _prefill(f"gqa{_hkv}_S{_S}", _S, 32, _hkv, False)

# Packed variable-length causal prefill, 8 entries of 1k-16k rows (53248 in all), GQA 32/8.
PACKED_WORKLOADS = {
    "packed_causal_gqa8": PackedWorkload("packed_causal_gqa8", (16384, 1024, 8192, 2048, 12288, 4096, 3072, 6144),
                                         32, 8, 128, BF16, True),
}


@dataclass(frozen=True)
class ExWorkload:
    """A generalised-mode case of this library's extensions (attn_fwd_ex): Sq queries against
    Sk keys aligned at the bottom right, an optional left window, optional per-head Bernoulli
    masks; bf16, d = 128."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    causal: bool
    window_left: int
    per_head_mask: bool
    d: int = 128
    dtype: int = BF16

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d)))

    def kept_pairs(self) -> int:
        """(row, key) pairs the band keeps (custom bits counted dense), per (batch, head)."""
        i = np.arange(self.Sq)[:, None] + (self.Sk - self.Sq)
        j = np.arange(self.Sk)[None, :]
        keep = np.ones((self.Sq, self.Sk), bool)
        if self.causal:
            keep &= j <= i
        if self.window_left >= 0:
            keep &= j >= i - self.window_left
        return int(keep.sum())

    def flops(self) -> float:
        """4*d per kept (row, key) pair: the two contractions over the band."""
        return 4.0 * self.d * self.B * self.Hq * self.kept_pairs()

    def make(self, seed):
        """q [B,Hq,Sq,d], k and v [B,Hkv,Sk,d]; per-head mask bits [B,Hq,Sq,ceil(Sk/32)] or None."""
        q, k, v = qkv(self.B, self.Hq, self.Hkv, self.Sk, self.d, self.dtype, seed)
        q = q[:, :, self.Sk - self.Sq:].contiguous()
        bits = None
        if self.per_head_mask:
            bits = pack_bits(bernoulli_mask(self.B * self.Hq, self.Sk, seed)[:, :self.Sq]).reshape(
                self.B, self.Hq, self.Sq, -1)
        return q, k, v, bits


# Generalised-mode cases: a chunk of new queries against a long cache (GQA query-head pairs),
# a causal sliding window over a long sequence, per-head custom masks.
EX_WORKLOADS = {
    "ex_sq128_sk32768_gqa8": ExWorkload("ex_sq128_sk32768_gqa8", 8, 32, 8, 128, 32768, True, -1, False),
    "ex_window1024_S32768_gqa8": ExWorkload("ex_window1024_S32768_gqa8", 1, 32, 8, 32768, 32768, True, 1024, False),
    "ex_perhead_mask_S4096_mha": ExWorkload("ex_perhead_mask_S4096_mha", 2, 16, 16, 4096, 4096, False, -1, True),
}
