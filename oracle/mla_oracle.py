"""f64 CPU oracle for matrix-absorbed MLA split-KV decode.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or runs
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code with the CUDA library.

Every quantity is computed in float64 from the exact values of the 16-bit
inputs. The functions restate, step by step, what the source pages define:

* "feat(core): matrix-absorbed MLA decode over a compressed-latent KV cache"
  (mlxcel PR #995), section *What changed*, ``mla/decode.rs``: absorbed decode
  is softmax attention ``SDPA(q_absorbed, ckv, ckv, scale, mask)`` whose mask
  slot carries the rope score ``scale * q_pe @ kpe^T`` (plus the causal mask).
  The latent is both key and value.
* Same page, ``mla/split_kv.rs``: a plan cuts the latent (token) range into
  chunks; each chunk yields a *normalized* partial and its *log2* LSE; the
  chunks are merged by ``paged_attention_merge_states`` (section *How #898's
  merge kernel is reused*: LSE must be base 2).
* Same page, ``mla/absorb.rs``: the fold of ``kv_b_proj`` into ``W_UK
  [H, qk_nope, r]`` (query side) and ``W_UV^T [H, r, v_head]`` (output side);
  section *Verified vs unverified*: a host f64 reference performing the
  pre-absorption computation.
* "Wire MLA split-KV decode" (vllm-metal PR #601), section *What changed*: the
  slices are combined with each slice's LSE so the result equals ordinary
  attention.
* MTPLX PR #639, commit log (segmented KV cache, per-segment attention with an
  LSE merge): rows with no visible key carry ``lse = -inf``, get weight 0 and
  merge to zeros; the causal window rule ``gp <= row_limit``.

Readings taken where the pages are silent: LSE is log2 of the sum of exp of the *scaled* score; a partial is divided
by its own chunk's sum; chunk ``p`` of ``P`` covers tokens
``[p*C, min((p+1)*C, L))`` with ``C = ceil(ceil(L/P)/bs)*bs``; window row ``i``
of ``q_len`` sees absolute positions ``t <= L - q_len + i``.

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
(closed forms, library cross-checks, brute force, invariants and the memory
figures printed on the mlxcel page).
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

LN2 = math.log(2.0)

# ---------------------------------------------------------------------------
# exact decoding of the 16-bit inputs
# ---------------------------------------------------------------------------


def decode16(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact f64 value of IEEE-half or bfloat16 bit patterns (uint16)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def decode_e4m3(bits: np.ndarray) -> np.ndarray:
    """Exact f64 value of 8-bit E4M3 floating-point patterns (uint8).

    The pages leave caches other than 16-bit out ("Paged-backed and non-FP16
    latent caches, both declined", mlxcel PR #995, *Left out*); the format is
    taken as the OCP 8-bit E4M3 one: sign bit, 4 exponent bits with bias 7, 3
    mantissa bits; exponent field 0 is subnormal (mantissa x 2^-9); the one
    pattern S.1111.111 is NaN; there are no infinities (largest finite 448).
    """
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((b & 0x7) == 7), np.nan, val)


def decode_cache(bits: np.ndarray, case) -> np.ndarray:
    """Exact f64 value of cache entries: 16-bit patterns, or E4M3 patterns times the case's cache scale
    (a scalar folded into the dequantized value, as mlxcel PR #995, *What changed*, folds a global scale:
    ``(x @ W^T) * s == x @ (W * s)^T``)."""
    if case.dtype == "e4m3":
        return decode_e4m3(bits) * float(case.cache_scale)
    return decode16(bits, case.dtype)


def query_dtype(case) -> str:
    """The queries' 16-bit type: the case's dtype, fp16 beside an E4M3 cache."""
    return "f16" if case.dtype == "e4m3" else case.dtype


# ---------------------------------------------------------------------------
# paged cache addressing
# ---------------------------------------------------------------------------


def physical_rows(block_table_row: np.ndarray, n_tokens: int, block_size: int) -> np.ndarray:
    """Physical cache row of logical tokens 0..n-1 of one request.

    Token ``t`` lives in page ``block_table[t // bs]`` at slot ``t % bs``
    (the paged MLA cache of "Wire MLA split-KV decode", *What changed*).
    Returns flat row indices into ``cache.reshape(num_blocks*bs, width)``.
    """
    t = np.arange(n_tokens, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[t // block_size]
    if n_tokens and pages.min() < 0:
        raise ValueError("block table entry < 0 inside the context")
    return pages * block_size + (t % block_size)


def visible(n_tokens: int, q_len: int, i: int, causal: bool) -> np.ndarray:
    """Boolean mask of the tokens row ``i`` of a ``q_len`` window attends to.

    Without a causal mask every cached token is visible. With it, the window's
    rows are the last ``q_len`` tokens of the request and row ``i`` sees
    positions ``t <= L - q_len + i`` (MTPLX PR #639, the ``gp <= row_limit``
    mask of the flash kernels; mlxcel PR #995, additive causal mask).
    """
    t = np.arange(n_tokens)
    if not causal:
        return np.ones(n_tokens, dtype=bool)
    return t <= (n_tokens - q_len + i)


# ---------------------------------------------------------------------------
# absorbed attention for one query row
# ---------------------------------------------------------------------------


def scores(q_abs: np.ndarray, q_pe: np.ndarray, ckv_rows: np.ndarray,
           kpe_rows: np.ndarray, scale: float) -> np.ndarray:
    """Scaled scores of one query row against a set of cached tokens.

    ``s_t = scale * (q_abs . ckv_t) + scale * (q_pe . kpe_t)``: the latent
    half is the SDPA query-key product, the rope half is the additive term in
    SDPA's mask slot, both under the same scale (mlxcel PR #995, ``mla/decode.rs``).
    Shapes: q_abs [r], q_pe [d_r], ckv_rows [n, r], kpe_rows [n, d_r] -> [n].
    """
    latent = ckv_rows @ q_abs
    rope = kpe_rows @ q_pe
    return scale * latent + scale * rope


def attend(s: np.ndarray, values: np.ndarray) -> Tuple[np.ndarray, float]:
    """Softmax-weighted average of ``values`` and the log2 LSE of ``s``.

    Plain softmax definition with the maximum subtracted for range:
    ``m = max s``, ``w_t = exp(s_t - m)``, ``l = sum w``, ``o = sum w_t v_t / l``,
    ``lse2 = (m + ln l) / ln 2``. An empty set gives ``o = 0`` and
    ``lse2 = -inf`` (MTPLX PR #639: rows with no visible key).
    """
    if s.size == 0:
        return np.zeros(values.shape[1], dtype=np.float64), -math.inf
    m = float(np.max(s))
    w = np.exp(s - m)
    l = float(np.sum(w))
    o = (w @ values) / l
    lse2 = (m + math.log(l)) / LN2
    return o, lse2


def _request_rows(case, b: int):
    """f64 latent rows of request b (logical token order) and its queries."""
    L = int(case.context_lens[b])
    bs = case.block_size
    rows = physical_rows(case.block_table[b], L, bs)
    ckv = case.ckv.reshape(-1, case.ckv.shape[-1])
    kpe = case.kpe.reshape(-1, case.kpe.shape[-1])
    ckv_rows = decode_cache(ckv[rows], case)
    kpe_rows = decode_cache(kpe[rows], case)
    qa = decode16(case.q_abs[b], query_dtype(case))  # [q_len, H, r]
    qp = decode16(case.q_pe[b], query_dtype(case))  # [q_len, H, d_r]
    return L, ckv_rows, kpe_rows, qa, qp


def unsplit(case, heads: Sequence[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Unsplit absorbed decode ("Stage 1" of mlxcel PR #995).

    Returns ``out [B, q_len, H, r]`` and ``lse2 [B, q_len, H]``. ``heads``
    restricts the computation to some heads (the others are left NaN), for
    sampled checks at full size.
    """
    B, q_len, H = case.num_requests, case.q_len, case.num_heads
    r = case.ckv.shape[-1]
    out = np.full((B, q_len, H, r), np.nan)
    lse = np.full((B, q_len, H), np.nan)
    hs = range(H) if heads is None else heads
    for b in range(B):
        L, ckv_rows, kpe_rows, qa, qp = _request_rows(case, b)
        for i in range(q_len):
            vis = visible(L, q_len, i, case.causal)
            cv, kv = ckv_rows[vis], kpe_rows[vis]
            for h in hs:
                s = scores(qa[i, h], qp[i, h], cv, kv, case.scale)
                out[b, i, h], lse[b, i, h] = attend(s, cv)
    return out, lse


# ---------------------------------------------------------------------------
# split into chunks, partials, merge
# ---------------------------------------------------------------------------


def chunk_bounds(n_tokens: int, n_parts: int, block_size: int) -> List[Tuple[int, int]]:
    """Contiguous, block-aligned token ranges of a split into ``n_parts``.

    Chunk length ``C = ceil(ceil(L / P) / bs) * bs``; chunk ``p`` is
    ``[min(p*C, L), min((p+1)*C, L))`` and may be empty when L is small.
    (mlxcel PR #995, ``MlaSplitPlan`` "cuts the latent range".)
    """
    if n_parts < 1:
        raise ValueError("n_parts >= 1")
    per = -(-n_tokens // n_parts)
    C = -(-per // block_size) * block_size
    C = max(C, block_size)
    return [(min(p * C, n_tokens), min((p + 1) * C, n_tokens)) for p in range(n_parts)]


def partials(case, chunks: Sequence[Tuple[int, int, int]], heads: Sequence[int] = None):
    """Normalized partial and log2 LSE of every chunk.

    ``chunks[n] = (b, t0, t1)``: request ``b``, logical tokens ``[t0, t1)``.
    Each partial is the attention of the row over the visible tokens of the
    chunk alone, divided by the chunk's own sum (mlxcel PR #995,
    ``mla/split_kv.rs``). Returns ``[N, q_len, H, r]`` and ``[N, q_len, H]``.
    """
    N = len(chunks)
    q_len, H = case.q_len, case.num_heads
    r = case.ckv.shape[-1]
    part = np.full((N, q_len, H, r), np.nan)
    lse = np.full((N, q_len, H), np.nan)
    hs = range(H) if heads is None else heads
    cache = {}
    for n, (b, t0, t1) in enumerate(chunks):
        if b not in cache:
            cache = {b: _request_rows(case, b)}
        L, ckv_rows, kpe_rows, qa, qp = cache[b]
        in_chunk = np.zeros(L, dtype=bool)
        in_chunk[t0:t1] = True
        for i in range(q_len):
            vis = visible(L, q_len, i, case.causal) & in_chunk
            cv, kv = ckv_rows[vis], kpe_rows[vis]
            for h in hs:
                s = scores(qa[i, h], qp[i, h], cv, kv, case.scale)
                part[n, i, h], lse[n, i, h] = attend(s, cv)
    return part, lse


def merge(part: np.ndarray, lse2: np.ndarray, o_indptr: Sequence[int]):
    """LSE-weighted merge of request-major partials (base-2 LSE).

    For request ``b`` its partials are ``o_indptr[b] .. o_indptr[b+1]-1``. Per
    row: ``M = max_p lse_p``; if ``M = -inf`` the result is 0 with LSE -inf;
    otherwise ``w_p = 2^(lse_p - M)``, ``out = sum w_p o_p / sum w_p`` and
    ``lse = M + log2 sum w_p`` (mlxcel PR #995, merge contract of
    ``paged_attention_merge_states``; vllm-metal PR #601, reduce by LSE).
    """
    B = len(o_indptr) - 1
    shp = part.shape[1:]
    out = np.zeros((B,) + shp)
    out_lse = np.full((B,) + shp[:-1], -math.inf)
    for b in range(B):
        lo, hi = int(o_indptr[b]), int(o_indptr[b + 1])
        if hi <= lo:
            continue
        ls = lse2[lo:hi]  # [P, ...rows]
        M = np.max(ls, axis=0)
        finite = np.isfinite(M)
        Msafe = np.where(finite, M, 0.0)
        w = np.where(np.isfinite(ls), np.exp2(ls - Msafe[None]), 0.0)
        wsum = np.sum(w, axis=0)
        num = np.einsum("p...,p...d->...d", w, np.nan_to_num(part[lo:hi]))
        den = np.where(finite, wsum, 1.0)
        out[b] = np.where(finite[..., None], num / den[..., None], 0.0)
        out_lse[b] = np.where(finite, Msafe + np.log2(den), -math.inf)
    return out, out_lse


def merge_natural_log(part: np.ndarray, lse2: np.ndarray, o_indptr: Sequence[int]):
    """Negative control: the same merge with natural-log LSE fed in.

    mlxcel PR #995 (*How #898's merge kernel is reused*): a natural-log LSE
    still merges and returns a plausible, wrong weighted average. This feeds
    ``lse_ln = lse2 * ln 2`` into the base-2 merge.
    """
    return merge(part, lse2 * LN2, o_indptr)


def plan_chunks(context_lens: Sequence[int], parts: Sequence[int], block_size: int):
    """Request-major chunk list and ``o_indptr`` for per-request part counts."""
    chunks, indptr = [], [0]
    for b, (L, P) in enumerate(zip(context_lens, parts)):
        for t0, t1 in chunk_bounds(int(L), int(P), block_size):
            chunks.append((b, t0, t1))
        indptr.append(len(chunks))
    return chunks, indptr


# ---------------------------------------------------------------------------
# the pre-absorption (decompressed) computation and the fold
# ---------------------------------------------------------------------------


def absorb_query(q_nope: np.ndarray, W_UK: np.ndarray) -> np.ndarray:
    """``q_abs[h] = q_nope[h] @ W_UK[h]`` with ``W_UK [H, qk_nope, r]``.

    The query-side fold of ``kv_b_proj`` (mlxcel PR #995, ``mla/absorb.rs``).
    """
    return np.einsum("hn,hnr->hr", q_nope, W_UK)


def unembed(o_latent: np.ndarray, W_UV_T: np.ndarray) -> np.ndarray:
    """``o_v[h] = o_latent[h] @ W_UV^T[h]`` with ``W_UV^T [H, r, v_head]``."""
    return np.einsum("hr,hrv->hv", o_latent, W_UV_T)


def decompressed_decode(q_nope, q_pe, W_UK, W_UV_T, ckv_rows, kpe_rows, scale):
    """Decode with per-head K/V up-projected from the latent (no absorption).

    ``k_nope[t,h] = W_UK[h] @ ckv_t`` (qk_nope wide), ``v[t,h] = ckv_t @ W_UV^T[h]``
    (v_head wide), ``s = scale*(q_nope.k_nope + q_pe.kpe)``, output
    ``softmax(s) @ v``: the computation the fold replaces (mlxcel PR #995,
    *Verified vs unverified*). Shapes: q_nope [H, n], q_pe [H, d_r],
    W_UK [H, n, r], W_UV_T [H, r, v], ckv_rows [T, r], kpe_rows [T, d_r].
    """
    H = q_nope.shape[0]
    out = []
    for h in range(H):
        k_nope = ckv_rows @ W_UK[h].T  # [T, n]
        v = ckv_rows @ W_UV_T[h]  # [T, v]
        s = scale * (k_nope @ q_nope[h] + kpe_rows @ q_pe[h])
        o, _ = attend(s, v)
        out.append(o)
    return np.stack(out)


# ---------------------------------------------------------------------------
# the steps either side of attention: the cache write and the unembed
# ---------------------------------------------------------------------------


def cache_append(ckv, kpe, block_table, context_lens, ckv_new, kpe_new, block_size):
    """The paged cache after writing each request's newest tokens.

    Token ``i`` of the ``q_len`` new tokens of request ``b`` is logical
    position ``t = L_b - q_len + i`` (``context_lens`` already counts the new
    tokens, the convention of the causal window: the window's rows are the
    last ``q_len`` tokens of the request), stored at the physical row of ``t``
    ("Wire MLA split-KV decode", *Bench*: the wrapper writes the new token's
    latent into the paged cache before attention). Positions below 0 are not
    written. Works on the bit patterns; returns new arrays.
    """
    ckv = np.array(ckv, copy=True)
    kpe = np.array(kpe, copy=True)
    flat_c = ckv.reshape(-1, ckv.shape[-1])
    flat_k = kpe.reshape(-1, kpe.shape[-1])
    B, q_len = ckv_new.shape[0], ckv_new.shape[1]
    for b in range(B):
        L = int(context_lens[b])
        for i in range(q_len):
            t = L - q_len + i
            if t < 0:
                continue
            row = int(block_table[b][t // block_size]) * block_size + t % block_size
            flat_c[row] = ckv_new[b, i]
            flat_k[row] = kpe_new[b, i]
    return ckv, kpe


def merge_unembed(part, lse2, o_indptr, W_UV_T):
    """Merged latent output taken to the value space: ``merge`` then, per
    request and row, ``unembed`` (mlxcel PR #995, *What changed*: the output
    side of the fold, ``W_UV^T [H, r, v_head]``). Returns ``[B, q_len, H, v]``
    and the merged log2 LSE."""
    out, out_lse = merge(part, lse2, o_indptr)
    B, q_len = out.shape[0], out.shape[1]
    ov = np.stack([np.stack([unembed(out[b, i], W_UV_T) for i in range(q_len)]) for b in range(B)])
    return ov, out_lse


# ---------------------------------------------------------------------------
# KV-memory accounting (mlxcel PR #995, performance-validation commit)
# ---------------------------------------------------------------------------


def latent_elems_per_token(kv_lora_rank: int, rope_dim: int) -> int:
    """Elements cached per token per layer by the absorbed path: ckv + kpe."""
    return kv_lora_rank + rope_dim


def decompressed_elems_per_token(num_heads: int, qk_head_dim: int, v_head_dim: int) -> int:
    """Elements per token per layer when per-head K and V are cached."""
    return num_heads * (qk_head_dim + v_head_dim)


def max_context_tokens(budget_bytes: int, elems_per_token: int, elem_bytes: int,
                       num_layers: int) -> int:
    """Tokens that fit a KV budget: ``floor(budget / (elems * bytes * layers))``."""
    return budget_bytes // (elems_per_token * elem_bytes * num_layers)
