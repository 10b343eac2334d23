"""The closed form that `mla_selfcheck` relies on, checked by the f64 oracle.

`mla_selfcheck` (include/mla_split_kv.h) decodes a built-in case and expects,
without any reference computation: for 15 "needle" heads the latent row of the
needle token and a base-2 LSE of 64 log2 e; for the head with zero queries the
mean latent row and LSE log2 L. This test builds the same case in numpy,
runs the oracle on it and confirms those expectations, so the library's own
check stands on the pages' definition of the partial and its LSE (mlxcel PR
#995, *What changed*) and not only on its author's arithmetic. The case
construction below restates the one in the library's `selfcheck.cu`.
"""
import math

import numpy as np
import pytest

from mla_split_kv_gb300.inputs import DecodeCase
from oracle import mla_oracle as orc

LENS = (6000, 700)
H, BS, POOL, RANK, ROPE = 16, 32, 256, 512, 64
SCALE, NEEDLE, UNUSED = 4.0, 16.0, 1000.0


def rope_col(h):
    return 5 + 8 * h


def latent_col(h):
    return 37 + 61 * (h - 8)


def needle_token(b, h):
    if h == 14:
        return LENS[b] - 1
    return h * 397 + 123 if b == 0 else h * 43 + 5


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    return (x.view(np.uint32) >> 16).astype(np.uint16)  # every value here is exact in bf16


def build(dtype: str) -> DecodeCase:
    max_blocks = -(-LENS[0] // BS)
    table = np.full((2, max_blocks), -1, dtype=np.int32)
    nxt = 0
    for b, L in enumerate(LENS):
        for i in range(-(-L // BS)):
            table[b, i] = (nxt * 37 + 11) % POOL
            nxt += 1
    ckv = np.full((POOL * BS, RANK), UNUSED, dtype=np.float32)
    kpe = np.zeros((POOL * BS, ROPE), dtype=np.float32)
    d = np.arange(RANK)
    for b, L in enumerate(LENS):
        for t in range(L):
            r = table[b, t // BS] * BS + t % BS
            ckv[r] = ((13 * t + 7 * d) % 64 - 32) * 0.125
    q_abs = np.zeros((2, 1, H, RANK), dtype=np.float32)
    q_pe = np.zeros((2, 1, H, ROPE), dtype=np.float32)
    for b in range(2):
        for h in range(8):
            q_pe[b, 0, h, rope_col(h)] = 1.0
            t = needle_token(b, h)
            kpe[table[b, t // BS] * BS + t % BS, rope_col(h)] = NEEDLE
        for h in range(8, 15):
            q_abs[b, 0, h, latent_col(h)] = 1.0
            t = needle_token(b, h)
            ckv[table[b, t // BS] * BS + t % BS, latent_col(h)] = NEEDLE
    return DecodeCase(dtype=dtype, num_heads=H, q_len=1, block_size=BS, scale=SCALE, causal=False,
                      q_abs=to_bits(q_abs, dtype), q_pe=to_bits(q_pe, dtype),
                      ckv=to_bits(ckv, dtype).reshape(POOL, BS, RANK), kpe=to_bits(kpe, dtype).reshape(POOL, BS, ROPE),
                      block_table=table, context_lens=np.array(LENS, dtype=np.int32))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_selfcheck_case_has_the_closed_form_answer(dtype):
    case = build(dtype)
    out, lse = orc.unsplit(case)
    ckv = orc.decode16(case.ckv, dtype).reshape(POOL * BS, RANK)
    for b, L in enumerate(LENS):
        rows = orc.physical_rows(case.block_table[b], L, BS)
        assert len(set(rows.tolist())) == L and np.all(ckv[rows] != UNUSED)  # pages disjoint, all owned
        for h in range(15):
            t = needle_token(b, h)
            np.testing.assert_allclose(out[b, 0, h], ckv[rows[t]], rtol=0, atol=1e-12)
            assert abs(lse[b, 0, h] - SCALE * NEEDLE / math.log(2)) < 1e-9
        np.testing.assert_allclose(out[b, 0, 15], ckv[rows].mean(axis=0), rtol=0, atol=1e-12)
        assert abs(lse[b, 0, 15] - math.log2(L)) < 1e-12


def test_selfcheck_case_columns_and_needles_cover_both_halves():
    # the pair kernel splits latent columns 0..255 / 256..511 and rope columns 0..31 / 32..63
    assert {rope_col(h) // 32 for h in range(8)} == {0, 1}
    assert {latent_col(h) // 256 for h in range(8, 15)} == {0, 1}
    for b, L in enumerate(LENS):
        ts = [needle_token(b, h) for h in range(15)]
        assert max(ts) == L - 1 and min(ts) >= 0 and L % BS != 0
