"""Plant plausible slips in the oracle (on the CPU) and check a pin catches each.

Each mutation monkeypatches one oracle function with a version carrying a
typical mistake; the listed pin tests must then fail. This guards the pins
themselves: a pin that cannot see a dropped term is not a pin.
"""
import math

import numpy as np
import pytest

from oracle import mla_oracle as orc
import tests.test_oracle_pins as pins
import tests.test_selfcheck_case_cpu as selfcase


def _drop_rope(q_abs, q_pe, ckv_rows, kpe_rows, scale):
    return scale * (ckv_rows @ q_abs)


def _scale_latent_only(q_abs, q_pe, ckv_rows, kpe_rows, scale):
    return scale * (ckv_rows @ q_abs) + (kpe_rows @ q_pe)


def _natural_log_lse(s, values):
    if s.size == 0:
        return np.zeros(values.shape[1]), -math.inf
    m = float(np.max(s))
    w = np.exp(s - m)
    l = float(np.sum(w))
    return (w @ values) / l, m + math.log(l)


def _causal_off_by_one(n_tokens, q_len, i, causal):
    t = np.arange(n_tokens)
    if not causal:
        return np.ones(n_tokens, dtype=bool)
    return t < (n_tokens - q_len + i)


def _page_slip(block_table_row, n_tokens, block_size):
    t = np.arange(n_tokens, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[t // block_size]
    return pages * block_size + (t % block_size) + (t // block_size) % 2  # shifts odd pages by one row


def _merge_natural(part, lse2, o_indptr):
    B = len(o_indptr) - 1
    out = np.zeros((B,) + part.shape[1:])
    out_lse = np.full((B,) + part.shape[1:-1], -math.inf)
    for b in range(B):
        lo, hi = o_indptr[b], o_indptr[b + 1]
        ls = lse2[lo:hi]
        M = ls.max(axis=0)
        w = np.exp(ls - M)  # e-base weights on log2 values
        out[b] = np.einsum("p...,p...d->...d", w, part[lo:hi]) / w.sum(axis=0)[..., None]
        out_lse[b] = M + np.log2(w.sum(axis=0))
    return out, out_lse


def _chunks_unaligned(n_tokens, n_parts, block_size):
    C = -(-n_tokens // n_parts)  # forgets to round the chunk length up to whole pages
    return [(min(p * C, n_tokens), min((p + 1) * C, n_tokens)) for p in range(n_parts)]


def _indptr_slip(context_lens, parts, block_size):
    chunks, indptr = [], [0]
    for b, (L, P) in enumerate(zip(context_lens, parts)):
        indptr.append(len(chunks))  # records the start instead of the end of request b
        for t0, t1 in orc.chunk_bounds(int(L), int(P), block_size):
            chunks.append((b, t0, t1))
    return chunks, indptr


def _append_one_late(ckv, kpe, block_table, context_lens, ckv_new, kpe_new, block_size):
    # writes token i at position L - q_len + i + 1 (one past the window's own slot)
    ckv = np.array(ckv, copy=True)
    kpe = np.array(kpe, copy=True)
    fc, fk = ckv.reshape(-1, ckv.shape[-1]), kpe.reshape(-1, kpe.shape[-1])
    for b in range(ckv_new.shape[0]):
        for i in range(ckv_new.shape[1]):
            t = int(context_lens[b]) - ckv_new.shape[1] + i + 1
            if 0 <= t < len(block_table[b]) * block_size and block_table[b][t // block_size] >= 0:
                row = int(block_table[b][t // block_size]) * block_size + t % block_size
                fc[row], fk[row] = ckv_new[b, i], kpe_new[b, i]
    return ckv, kpe


def _e4m3_bias_eight(bits):
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    e, m = (b >> 3) & 0xF, (b & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -10, (1 + m / 8) * np.exp2(e - 8.0))  # exponent bias 8 instead of 7
    return np.where(b & 0x80, -val, val)


def _cache_scale_dropped(bits, case):
    return orc.decode_e4m3(bits) if case.dtype == "e4m3" else orc.decode16(bits, case.dtype)


def _unembed_other_side(o_latent, W_UV_T):
    return np.einsum("hr,hrv->hv", o_latent, W_UV_T[::-1])  # heads' projections swapped


MUTATIONS = [
    ("scores", _drop_rope, [pins.test_rope_score_is_additive,
                            lambda: pins.test_matches_torch_sdpa_on_concatenated_keys("f16", 1, False)]),
    ("scores", _scale_latent_only, [lambda: pins.test_matches_torch_sdpa_on_concatenated_keys("f16", 1, False)]),
    ("attend", _natural_log_lse, [pins.test_zero_query_gives_uniform_mean_and_log2_count,
                                  lambda: selfcase.test_selfcheck_case_has_the_closed_form_answer("f16")]),
    ("visible", _causal_off_by_one, [pins.test_visible_rule_small_window,
                                     pins.test_brute_force_pure_python_tiny]),
    ("physical_rows", _page_slip, [pins.test_physical_rows_hand_table,
                                   lambda: pins.test_matches_torch_sdpa_on_concatenated_keys("f16", 1, False)]),
    ("merge", _merge_natural, [pins.test_merge_weights_are_base_two]),
    ("chunk_bounds", _chunks_unaligned, [pins.test_chunk_bounds_examples_and_invariants,
                                         pins.test_plan_chunks_covers_every_token_once_request_major]),
    ("plan_chunks", _indptr_slip, [pins.test_plan_chunks_covers_every_token_once_request_major]),
    ("cache_append", _append_one_late, [pins.test_cache_append_hand_table,
                                        pins.test_cache_append_of_the_cached_tail_is_the_identity_and_shifted_rows_are_not]),
    ("decode_e4m3", _e4m3_bias_eight, [pins.test_decode_e4m3_known_bit_patterns,
                                       pins.test_decode_e4m3_matches_torch_float8_on_every_pattern]),
    ("decode_cache", _cache_scale_dropped, [pins.test_e4m3_cache_matches_torch_sdpa_with_its_scale]),
    ("unembed", _unembed_other_side, [pins.test_absorbed_equals_decompressed_and_transposed_fold_does_not,
                                      pins.test_merge_unembed_is_the_decompressed_decode_of_a_split]),
]


@pytest.mark.parametrize("name,fn,tests", MUTATIONS, ids=[m[1].__name__ for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, fn, tests):
    monkeypatch.setattr(orc, name, fn)
    for t in tests:
        with pytest.raises((AssertionError, ValueError, IndexError)):
            t()
