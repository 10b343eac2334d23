"""The seeded input generators keep the recipe they state.

Same seed, same bits; requests own disjoint pages of the pool; the draws have
the stated spread; the 16-bit roundings agree with independent conversions
(numpy for fp16, torch for bf16); re-placing the pool or concatenating
segments keeps every request's logical token rows.
"""
import numpy as np
import pytest
import torch

from mla_split_kv_gb300 import inputs as gen


def logical_rows(case, b, arr):
    L = int(case.context_lens[b])
    t = np.arange(L)
    pages = case.block_table[b, t // case.block_size]
    return arr.reshape(-1, arr.shape[-1])[pages * case.block_size + t % case.block_size]


def test_same_seed_same_bits_other_seed_other_bits():
    a = gen.make_decode_case(3, [700, 90], num_heads=16, block_size=32)
    b = gen.make_decode_case(3, [700, 90], num_heads=16, block_size=32)
    c = gen.make_decode_case(4, [700, 90], num_heads=16, block_size=32)
    for f in ("q_abs", "q_pe", "ckv", "kpe", "block_table", "context_lens"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert not np.array_equal(a.ckv, c.ckv) and not np.array_equal(a.block_table, c.block_table)


def test_requests_own_disjoint_pages_of_the_pool():
    lens = [1000, 33, 0, 4096]
    case = gen.make_decode_case(5, lens, block_size=16)
    seen = set()
    for b, L in enumerate(lens):
        n = gen.pages_for(L, 16)
        row = case.block_table[b]
        assert np.all(row[n:] == -1)
        ids = row[:n].tolist()
        assert all(0 <= i < case.num_blocks for i in ids)
        assert not seen.intersection(ids)
        seen.update(ids)
    assert case.num_blocks == 2 * sum(gen.pages_for(L, 16) for L in lens)


@pytest.mark.parametrize("std", [1.0, 0.5])
def test_draws_have_the_stated_spread(std):
    case = gen.make_decode_case(6, [4096], block_size=32, latent_std=std, dtype="f16")
    ckv = gen_decode(case.ckv, "f16")
    q = gen_decode(case.q_abs, "f16")
    assert abs(ckv.mean()) < 0.01 * std and abs(ckv.std() - std) < 0.01 * std
    assert abs(q.std() - 1.0) < 0.05


def gen_decode(bits, dtype):
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_sixteen_bit_roundings_match_independent_conversions():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 3, [0.0, -0.0, 1e-8, 65504.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]])
    assert np.array_equal(gen.to_f16_bits(x), x.astype(np.float16).view(np.uint16))
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gen.to_bf16_bits(x.astype(np.float32)), want)


def test_repacking_the_pool_keeps_every_request_logical_rows():
    case = gen.make_decode_case(7, [777, 64], block_size=32)
    moved = gen.permute_pool(case, 11)
    assert not np.array_equal(moved.block_table, case.block_table)
    for b in range(2):
        assert np.array_equal(logical_rows(case, b, case.ckv), logical_rows(moved, b, moved.ckv))
        assert np.array_equal(logical_rows(case, b, case.kpe), logical_rows(moved, b, moved.kpe))


def test_concatenated_segments_are_the_segments_in_order():
    seg = gen.make_segmented_case(8, B=2, q_len=4, segment_tokens=(64, 96), block_size=32)
    whole = gen.concat_segments(seg)
    for b in range(2):
        parts = [logical_rows(s, b, s.ckv) for s in seg.segments]
        assert np.array_equal(logical_rows(whole, b, whole.ckv), np.concatenate(parts))
        assert int(whole.context_lens[b]) == 64 + 96 + 4
    # the segments' pages come from disjoint regions of the pool
    used = [set(s.block_table[s.block_table >= 0].tolist()) for s in seg.segments]
    for i in range(len(used)):
        for j in range(i + 1, len(used)):
            assert not used[i] & used[j]


def test_e4m3_cache_bits_and_case():
    """E4M3 caches are uint8 patterns with no NaN, magnitudes 0.125 .. 7.5 or zero/subnormal, fp16 queries and a
    power-of-two cache scale; the byte count of a pass is half the 16-bit one."""
    c = gen.make_decode_case(3, [500, 77], num_heads=16, block_size=32, dtype="e4m3", cache_scale=0.25)
    assert c.ckv.dtype == np.uint8 and c.kpe.dtype == np.uint8 and c.q_abs.dtype == np.uint16
    for x in (c.ckv, c.kpe):
        assert not np.any((x & 0x7F) == 0x7F)  # no NaN pattern
        e = (x >> 3) & 0xF
        assert set(np.unique(e).tolist()) <= {0, 4, 5, 6, 7, 8, 9}
        assert 0.04 < np.mean(e == 0) < 0.09  # about one entry in 16 is zero or subnormal
    assert c.cache_scale == 0.25
    f = gen.make_decode_case(3, [500, 77], num_heads=16, block_size=32, dtype="f16")
    assert 2 * c.latent_bytes() == f.latent_bytes()
