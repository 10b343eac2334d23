"""Seeded synthetic inputs for MLA split-KV decode.

This module only draws and lays out data: Gaussian queries and latents, paged
cache pools, shuffled block tables and per-request context lengths. It holds
none of the attention arithmetic, so both the CUDA path and the f64 oracle can
be fed from it without sharing any of the method's code.

Conventions (shared by every consumer):

* 16-bit tensors are stored as ``numpy.uint16`` bit patterns together with a
  dtype tag ``"f16"`` (IEEE binary16) or ``"bf16"`` (bfloat16). f64 draws are
  rounded once, to nearest-even, into the tagged type.
* dtype ``"e4m3"``: the caches are ``numpy.uint8`` 8-bit E4M3 patterns drawn
  directly as bits (random sign, exponent field, mantissa; no NaN pattern),
  read with a scalar ``cache_scale``; the queries are fp16.
* ``ckv``  : ``[num_blocks, block_size, 512]`` -- compressed latent, one row per
  cached token (the key *and* the value of absorbed attention).
* ``kpe``  : ``[num_blocks, block_size, 64]`` -- rotary key part.
* ``q_abs``: ``[B, q_len, H, 512]`` absorbed query, ``q_pe``: ``[B, q_len, H, 64]``.
* ``block_table``: ``[B, max_blocks]`` int32 physical page ids; entries past a
  request's last page are filled with -1 and never used.
* ``context_lens``: ``[B]`` int32 tokens per request.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

KV_LORA_RANK = 512  # r: width of the compressed latent ckv
ROPE_DIM = 64  # d_r: width of the rotary key kpe


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round f64/f32 values to IEEE half (nearest-even) and return the bits."""
    return np.asarray(x).astype(np.float16).view(np.uint16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round values to bfloat16 and return the bits.

    The value is rounded to f32 (nearest-even), then the f32 bit pattern is
    rounded to its top 16 bits (nearest-even on the dropped half-word).
    """
    bits = np.asarray(x).astype(np.float32).view(np.uint32).astype(np.uint64)
    bits = bits + 0x7FFF + ((bits >> 16) & 1)
    return (bits >> 16).astype(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return to_f16_bits(x)
    if dtype == "bf16":
        return to_bf16_bits(x)
    raise ValueError(f"unknown dtype tag {dtype!r}")


@dataclasses.dataclass
class DecodeCase:
    """One batch of absorbed-MLA decode inputs over a paged latent cache."""

    dtype: str
    num_heads: int
    q_len: int
    block_size: int
    scale: float
    causal: bool
    q_abs: np.ndarray  # uint16 [B, q_len, H, 512]
    q_pe: np.ndarray  # uint16 [B, q_len, H, 64]
    ckv: np.ndarray  # uint16 [num_blocks, bs, 512]
    kpe: np.ndarray  # uint16 [num_blocks, bs, 64]
    block_table: np.ndarray  # int32 [B, max_blocks]
    context_lens: np.ndarray  # int32 [B]
    cache_scale: float = 1.0  # e4m3 caches: the value of pattern x is e4m3(x) * cache_scale

    @property
    def num_requests(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.ckv.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def latent_bytes(self) -> int:
        """Bytes of ckv+kpe a single pass over every request's context touches."""
        per = 1 if self.dtype == "e4m3" else 2
        return int(self.context_lens.astype(np.int64).sum()) * (KV_LORA_RANK + ROPE_DIM) * per


def pages_for(n_tokens: int, block_size: int) -> int:
    return (int(n_tokens) + block_size - 1) // block_size


def e4m3_bits(rng: np.random.Generator, shape) -> np.ndarray:
    """Random 8-bit E4M3 patterns: random sign and mantissa, exponent field 4..9 (values 0.125 to 7.5 in
    magnitude) for 15 of 16 entries, and field 0 (zero and subnormals) for the rest; never the NaN pattern."""
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8) << 7
    exp = rng.integers(4, 10, size=shape, dtype=np.uint8)
    exp = np.where(rng.integers(0, 16, size=shape) == 0, 0, exp).astype(np.uint8)
    mant = rng.integers(0, 8, size=shape, dtype=np.uint8)
    return (sign | (exp << 3) | mant).astype(np.uint8)


def _latent_pool(rng: np.random.Generator, num_blocks: int, block_size: int,
                 dtype: str, std: float):
    if dtype == "e4m3":
        return (e4m3_bits(rng, (num_blocks, block_size, KV_LORA_RANK)),
                e4m3_bits(rng, (num_blocks, block_size, ROPE_DIM)))
    ckv = to_bits(rng.standard_normal((num_blocks, block_size, KV_LORA_RANK)) * std, dtype)
    kpe = to_bits(rng.standard_normal((num_blocks, block_size, ROPE_DIM)) * std, dtype)
    return ckv, kpe


def _queries(rng: np.random.Generator, B: int, q_len: int, H: int, dtype: str):
    q_abs = to_bits(rng.standard_normal((B, q_len, H, KV_LORA_RANK)), dtype)
    q_pe = to_bits(rng.standard_normal((B, q_len, H, ROPE_DIM)), dtype)
    return q_abs, q_pe


def _tables_from_pages(page_lists: Sequence[Sequence[int]]) -> np.ndarray:
    width = max(1, max(len(p) for p in page_lists))
    bt = np.full((len(page_lists), width), -1, dtype=np.int32)
    for b, pages in enumerate(page_lists):
        bt[b, : len(pages)] = np.asarray(pages, dtype=np.int32)
    return bt


def make_decode_case(seed: int, context_lens: Sequence[int], num_heads: int = 16,
                     q_len: int = 1, block_size: int = 32, dtype: str = "f16",
                     scale: Optional[float] = None, latent_std: float = 1.0,
                     pool_blocks: Optional[int] = None, causal: bool = False,
                     shuffle: bool = True, cache_scale: float = 0.25) -> DecodeCase:
    """A batch whose requests own disjoint pages of one shared, shuffled pool.

    The pool holds ``pool_blocks`` pages (default: twice the pages needed, so
    the table really is a scatter). One permutation of the pool is drawn and
    split, in request order, into each request's pages.
    """
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in context_lens]
    need = [pages_for(L, block_size) for L in lens]
    total = sum(need)
    nb = pool_blocks if pool_blocks is not None else max(1, 2 * total)
    if nb < total:
        raise ValueError("pool smaller than the pages the batch needs")
    perm = rng.permutation(nb) if shuffle else np.arange(nb)
    pages, off = [], 0
    for n in need:
        pages.append(perm[off: off + n].tolist())
        off += n
    q_abs, q_pe = _queries(rng, len(lens), q_len, num_heads, "f16" if dtype == "e4m3" else dtype)
    ckv, kpe = _latent_pool(rng, nb, block_size, dtype, latent_std)
    return DecodeCase(dtype=dtype, num_heads=num_heads, q_len=q_len, block_size=block_size,
                      scale=scale if scale is not None else 1.0 / math.sqrt(192.0),
                      causal=causal, q_abs=q_abs, q_pe=q_pe, ckv=ckv, kpe=kpe,
                      block_table=_tables_from_pages(pages),
                      context_lens=np.asarray(lens, dtype=np.int32),
                      cache_scale=cache_scale if dtype == "e4m3" else 1.0)


@dataclasses.dataclass
class SegmentedCase:
    """A verify window over a prefix stored as non-contiguous segments.

    ``segments[k]`` is a :class:`DecodeCase` view that shares ``ckv``/``kpe``
    and the queries with every other segment but has its own block table and
    lengths. The last segment holds the window's own ``q_len`` tokens and is
    causal; the prefix segments are not (every window row sees all of them).
    """

    segments: List[DecodeCase]

    @property
    def base(self) -> DecodeCase:
        return self.segments[0]


def make_segmented_case(seed: int, B: int, q_len: int,
                        segment_tokens: Sequence[int] = (40960, 28672, 12288),
                        num_heads: int = 16, block_size: int = 32, dtype: str = "f16",
                        scale: Optional[float] = None, latent_std: float = 1.0,
                        pool_blocks: Optional[int] = None) -> SegmentedCase:
    """Multi-row verify windows whose prefix lives in several page regions.

    Every request has the same segment lengths (``segment_tokens``) followed by
    a tail segment of ``q_len`` tokens (the window itself). Each segment's
    pages are drawn from its own disjoint, shuffled region of one pool.
    """
    rng = np.random.default_rng(seed)
    seg_lens = [int(s) for s in segment_tokens] + [int(q_len)]
    per_req = [pages_for(s, block_size) for s in seg_lens]
    total = B * sum(per_req)
    nb = pool_blocks if pool_blocks is not None else max(1, total + total // 4)
    if nb < total:
        raise ValueError("pool smaller than the pages the batch needs")
    perm = rng.permutation(nb)
    # region k of the permutation serves segment k of every request
    tables, off = [], 0
    for k, npg in enumerate(per_req):
        reg = perm[off: off + B * npg]
        off += B * npg
        tables.append(_tables_from_pages([reg[b * npg:(b + 1) * npg].tolist() for b in range(B)]))
    q_abs, q_pe = _queries(rng, B, q_len, num_heads, dtype)
    ckv, kpe = _latent_pool(rng, nb, block_size, dtype, latent_std)
    sc = scale if scale is not None else 1.0 / math.sqrt(192.0)
    segs = []
    for k, L in enumerate(seg_lens):
        segs.append(DecodeCase(dtype=dtype, num_heads=num_heads, q_len=q_len,
                               block_size=block_size, scale=sc,
                               causal=(k == len(seg_lens) - 1), q_abs=q_abs, q_pe=q_pe,
                               ckv=ckv, kpe=kpe, block_table=tables[k],
                               context_lens=np.full((B,), L, dtype=np.int32)))
    return SegmentedCase(segments=segs)


def window_view(case: SegmentedCase, q_len: int) -> SegmentedCase:
    """The same prefix with a shorter verify window: the first ``q_len`` query rows
    and the first ``q_len`` tokens of the window segment (its pages and cache are
    shared with ``case``, nothing is copied but the queries)."""
    segs = case.segments
    if not 1 <= q_len <= segs[0].q_len:
        raise ValueError("q_len must be in [1, the case's window]")
    q_abs = np.ascontiguousarray(segs[0].q_abs[:, :q_len])
    q_pe = np.ascontiguousarray(segs[0].q_pe[:, :q_len])
    out = []
    for k, s in enumerate(segs):
        lens = s.context_lens if k < len(segs) - 1 else np.full_like(s.context_lens, q_len)
        out.append(dataclasses.replace(s, q_len=q_len, q_abs=q_abs, q_pe=q_pe, context_lens=lens))
    return SegmentedCase(segments=out)


def concat_segments(case: SegmentedCase) -> DecodeCase:
    """The same tokens as one logical sequence per request (prefix, then window).

    Segments are block-aligned except the last, so the logical block table is
    the concatenation of the segments' tables.
    """
    segs = case.segments
    B = segs[0].num_requests
    rows = []
    for b in range(B):
        pages = []
        for s in segs:
            n = pages_for(int(s.context_lens[b]), s.block_size)
            pages.extend(s.block_table[b, :n].tolist())
        rows.append(pages)
    lens = sum(s.context_lens.astype(np.int64) for s in segs).astype(np.int32)
    base = segs[0]
    return dataclasses.replace(base, causal=True, block_table=_tables_from_pages(rows),
                               context_lens=lens)


def uniform_lengths(seed: int, B: int, lo: int, hi: int) -> List[int]:
    """Integer context lengths drawn uniformly from [lo, hi] (inclusive)."""
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=B)]


def permute_pool(case: DecodeCase, seed: int) -> DecodeCase:
    """Same logical content under a different physical page placement.

    Pages are moved to new slots of the pool and the block table is rewritten to
    follow them, so every request still reads the same token rows.
    """
    rng = np.random.default_rng(seed)
    nb = case.num_blocks
    perm = rng.permutation(nb)  # old page i -> new slot perm[i]
    ckv = np.empty_like(case.ckv)
    kpe = np.empty_like(case.kpe)
    ckv[perm] = case.ckv
    kpe[perm] = case.kpe
    bt = case.block_table.copy()
    used = bt >= 0
    bt[used] = perm[bt[used]]
    return dataclasses.replace(case, ckv=ckv, kpe=kpe, block_table=bt)
