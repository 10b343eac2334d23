"""Pins for the f64 oracle, checked against things other than itself.

Each test fixes the oracle to a closed form, a library routine, brute force on
tiny inputs, an invariant the pages state, or a number printed on a page. The
tests are chosen so that a plausible slip (a dropped rope term, a scale on one
half only, a natural log for log2, a wrong page index, a swapped operand of the
fold, an off-by-one in the causal rule) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from mla_split_kv_gb300 import inputs as gen
from oracle import mla_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_case(seed=0, lens=(37,), H=2, q_len=1, bs=8, dtype="f16", causal=False, std=1.0):
    return gen.make_decode_case(seed, lens, num_heads=H, q_len=q_len, block_size=bs,
                                dtype=dtype, causal=causal, latent_std=std)


# --- exact decoding -----------------------------------------------------------

def test_decode16_known_bit_patterns():
    f16 = np.array([0x3C00, 0xC000, 0x7BFF, 0x0001, 0x3555], dtype=np.uint16)
    want = [1.0, -2.0, 65504.0, 2.0 ** -24, 0.333251953125]
    assert orc.decode16(f16, "f16").tolist() == want
    bf = np.array([0x3F80, 0x4049, 0xBF00, 0x0080], dtype=np.uint16)
    assert orc.decode16(bf, "bf16").tolist() == [1.0, 3.140625, -0.5, 2.0 ** -126]


def test_decode_e4m3_known_bit_patterns():
    """E4M3 patterns against the format's table (bias 7, subnormals at exponent field 0, 448 the largest)."""
    bits = np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3F, 0x40, 0x7E, 0xB8, 0xFE, 0x5A], dtype=np.uint8)
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.875, 2.0, 448.0, -1.0, -448.0, 20.0]
    assert orc.decode_e4m3(bits).tolist() == want
    neg_zero = orc.decode_e4m3(np.array([0x80], dtype=np.uint8))[0]
    assert neg_zero == 0.0 and math.copysign(1.0, neg_zero) == -1.0
    assert np.isnan(orc.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_decode_e4m3_matches_torch_float8_on_every_pattern():
    """All 256 patterns against torch's own float8_e4m3fn type (a library decode)."""
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.decode_e4m3(bits)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]) and np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_cache_matches_torch_sdpa_with_its_scale():
    """An E4M3 cache read as torch float8 values times the cache scale, fp16 queries: textbook SDPA."""
    case = gen.make_decode_case(8, [40, 11], num_heads=3, block_size=8, dtype="e4m3", cache_scale=0.125)
    out, lse = orc.unsplit(case)
    f8 = lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e4m3fn).to(torch.float64) * 0.125
    for b in range(2):
        L = int(case.context_lens[b])
        K, V = [], []
        for t in range(L):
            page = int(case.block_table[b][t // case.block_size])
            slot = t % case.block_size
            ck, kp = f8(case.ckv[page, slot]), f8(case.kpe[page, slot])
            K.append(torch.cat([ck, kp]))
            V.append(ck)
        K, V = torch.stack(K), torch.stack(V)
        Q = torch.tensor(np.concatenate([orc.decode16(case.q_abs[b], "f16"), orc.decode16(case.q_pe[b], "f16")],
                                        axis=-1)).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K.expand(3, L, 576), V.expand(3, L, 512),
                                                               scale=case.scale)
        np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        lse_ref = torch.logsumexp(case.scale * (Q @ K.T), dim=-1) / math.log(2)
        np.testing.assert_allclose(lse[b], lse_ref.permute(1, 0).numpy(), rtol=0, atol=1e-12)


# --- paged addressing and causal rule -----------------------------------------

def test_physical_rows_hand_table():
    bt = np.array([5, 2, 7], dtype=np.int32)
    rows = orc.physical_rows(bt, 9, 4)
    assert rows.tolist() == [20, 21, 22, 23, 8, 9, 10, 11, 28]


def test_visible_rule_small_window():
    # L = 5 tokens, window of 3 rows: row 0 is token 2, row 2 is token 4.
    assert orc.visible(5, 3, 0, True).tolist() == [True, True, True, False, False]
    assert orc.visible(5, 3, 2, True).tolist() == [True] * 5
    # q_len = 1 makes the causal mask vacuous
    assert orc.visible(5, 1, 0, True).all()
    assert orc.visible(5, 3, 0, False).all()


# --- closed forms ---------------------------------------------------------------

def test_zero_query_gives_uniform_mean_and_log2_count():
    case = small_case(seed=1, lens=(29,), H=3)
    case.q_abs[:] = 0
    case.q_pe[:] = 0
    out, lse = orc.unsplit(case)
    rows = orc.physical_rows(case.block_table[0], 29, case.block_size)
    ckv = orc.decode16(case.ckv.reshape(-1, 512)[rows], "f16")
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(ckv.mean(axis=0), (3, 512)), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], math.log2(29), rtol=0, atol=1e-13)


def test_single_token_returns_its_latent_row():
    case = small_case(seed=2, lens=(1,), H=2)
    out, lse = orc.unsplit(case)
    row = orc.physical_rows(case.block_table[0], 1, case.block_size)[0]
    ckv = orc.decode16(case.ckv.reshape(-1, 512)[row], "f16")
    kpe = orc.decode16(case.kpe.reshape(-1, 64)[row], "f16")
    for h in range(2):
        qa = orc.decode16(case.q_abs[0, 0, h], "f16")
        qp = orc.decode16(case.q_pe[0, 0, h], "f16")
        s = sum(float(a) * float(b) for a, b in zip(qa, ckv)) * case.scale \
            + sum(float(a) * float(b) for a, b in zip(qp, kpe)) * case.scale
        np.testing.assert_array_equal(out[0, 0, h], ckv)
        assert abs(lse[0, 0, h] - s / math.log(2)) < 1e-12


def test_two_tokens_logistic_form():
    case = small_case(seed=3, lens=(2,), H=2)
    out, lse = orc.unsplit(case)
    rows = orc.physical_rows(case.block_table[0], 2, case.block_size)
    ckv = orc.decode16(case.ckv.reshape(-1, 512)[rows], "f16")
    kpe = orc.decode16(case.kpe.reshape(-1, 64)[rows], "f16")
    for h in range(2):
        qa = orc.decode16(case.q_abs[0, 0, h], "f16")
        qp = orc.decode16(case.q_pe[0, 0, h], "f16")
        s = [case.scale * (float(np.dot(qa, ckv[t])) + float(np.dot(qp, kpe[t]))) for t in range(2)]
        sig = 1.0 / (1.0 + math.exp(-(s[0] - s[1])))
        want = sig * ckv[0] + (1.0 - sig) * ckv[1]
        np.testing.assert_allclose(out[0, 0, h], want, rtol=0, atol=1e-12)
        # log2(e^s0 + e^s1) via log1p form
        hi, lo = max(s), min(s)
        want_lse = (hi + math.log1p(math.exp(lo - hi))) / math.log(2)
        assert abs(lse[0, 0, h] - want_lse) < 1e-12


def test_dominant_token_wins():
    case = small_case(seed=4, lens=(16,), H=1, std=0.1)
    L = 16
    rows = orc.physical_rows(case.block_table[0], L, case.block_size)
    # make token 5's latent parallel to a large query so its score dominates by >> 60
    qa = np.zeros(512)
    qa[:8] = 1.0
    case.q_abs[0, 0, 0] = gen.to_f16_bits(qa)
    case.q_pe[0, 0, 0] = 0
    big = np.zeros(512)
    big[:8] = 64.0
    case.ckv.reshape(-1, 512)[rows[5]] = gen.to_f16_bits(big)
    out, _ = orc.unsplit(case)
    np.testing.assert_allclose(out[0, 0, 0], big, rtol=0, atol=1e-12)


# --- rope additivity and the textbook routine -----------------------------------

def test_rope_score_is_additive():
    rng = np.random.default_rng(5)
    qa, qp = rng.standard_normal(512), rng.standard_normal(64)
    cv, kv = rng.standard_normal((11, 512)), rng.standard_normal((11, 64))
    sc = 0.0721
    full = orc.scores(qa, qp, cv, kv, sc)
    only_latent = orc.scores(qa, np.zeros(64), cv, kv, sc)
    only_rope = orc.scores(np.zeros(512), qp, cv, kv, sc)
    np.testing.assert_allclose(full, only_latent + only_rope, rtol=0, atol=1e-12)
    # the rope half really contributes (a dropped term would make it vanish)
    assert np.abs(only_rope).max() > 0.1


@pytest.mark.parametrize("dtype,q_len,causal", [("f16", 1, False), ("bf16", 1, False), ("f16", 4, True)])
def test_matches_torch_sdpa_on_concatenated_keys(dtype, q_len, causal):
    """[q_abs|q_pe] . [ckv|kpe]^T with V = ckv is textbook SDPA with d_qk=576, d_v=512."""
    case = small_case(seed=6, lens=(45, 13), H=3, q_len=q_len, dtype=dtype, causal=causal)
    out, lse = orc.unsplit(case)
    for b in range(2):
        L = int(case.context_lens[b])
        # gather by walking the pages with explicit loops (independent of physical_rows)
        K, V = [], []
        for t in range(L):
            page = int(case.block_table[b][t // case.block_size])
            slot = t % case.block_size
            ck = orc.decode16(case.ckv[page, slot], dtype)
            kp = orc.decode16(case.kpe[page, slot], dtype)
            K.append(np.concatenate([ck, kp]))
            V.append(ck)
        K = torch.tensor(np.array(K))
        V = torch.tensor(np.array(V))
        Q = torch.tensor(np.concatenate([orc.decode16(case.q_abs[b], dtype),
                                         orc.decode16(case.q_pe[b], dtype)], axis=-1))  # [q_len,H,576]
        Q = Q.permute(1, 0, 2)  # [H, q_len, 576]
        mask = None
        if causal:
            ii = torch.arange(q_len)[:, None]
            tt = torch.arange(L)[None, :]
            mask = tt <= (L - q_len + ii)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K.expand(3, L, 576), V.expand(3, L, 512), attn_mask=mask, scale=case.scale)
        np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        s = case.scale * (Q @ K.T)  # [H, q_len, L]
        if causal:
            s = s.masked_fill(~mask, -math.inf)
        lse_ref = torch.logsumexp(s, dim=-1) / math.log(2)
        np.testing.assert_allclose(lse[b], lse_ref.permute(1, 0).numpy(), rtol=0, atol=1e-12)


def test_brute_force_pure_python_tiny():
    case = small_case(seed=7, lens=(6,), H=2, q_len=2, bs=4, causal=True)
    out, lse = orc.unsplit(case)
    L, q_len = 6, 2
    for h in range(2):
        for i in range(q_len):
            qa = [float(x) for x in orc.decode16(case.q_abs[0, i, h], "f16")]
            qp = [float(x) for x in orc.decode16(case.q_pe[0, i, h], "f16")]
            ss, vs = [], []
            for t in range(L - q_len + i + 1):
                page = int(case.block_table[0][t // 4])
                ck = [float(x) for x in orc.decode16(case.ckv[page, t % 4], "f16")]
                kp = [float(x) for x in orc.decode16(case.kpe[page, t % 4], "f16")]
                dot = 0.0
                for a, c in zip(qa, ck):
                    dot += a * c
                for a, c in zip(qp, kp):
                    dot += a * c
                ss.append(case.scale * dot)
                vs.append(ck)
            z = sum(math.exp(x) for x in ss)
            want = [sum(math.exp(ss[t]) * vs[t][d] for t in range(len(ss))) / z for d in range(512)]
            np.testing.assert_allclose(out[0, i, h], want, rtol=0, atol=1e-12)
            assert abs(lse[0, i, h] - math.log(z) / math.log(2)) < 1e-12


# --- chunking ----------------------------------------------------------------------

def test_chunk_bounds_examples_and_invariants():
    assert orc.chunk_bounds(100, 3, 32) == [(0, 64), (64, 100), (100, 100)]
    assert orc.chunk_bounds(4096, 4, 32) == [(0, 1024), (1024, 2048), (2048, 3072), (3072, 4096)]
    assert orc.chunk_bounds(20000, 3, 32) == [(0, 6688), (6688, 13376), (13376, 20000)]
    for L in (1, 31, 32, 33, 1000, 32768, 20000, 131071):
        for P in (1, 2, 3, 5, 8):
            for bs in (16, 32, 64):
                ch = orc.chunk_bounds(L, P, bs)
                assert len(ch) == P
                assert ch[0][0] == 0 and ch[-1][1] == L
                for (a0, a1), (b0, b1) in zip(ch, ch[1:]):
                    assert a1 == b0
                for t0, t1 in ch:
                    assert t0 <= t1 and (t0 % bs == 0 or t0 == L)


def test_plan_chunks_covers_every_token_once_request_major():
    # brute force over tiny batches: each (request, token) lies in exactly one chunk of that
    # request, the chunks of request b are o_indptr[b]..o_indptr[b+1]-1, P_b of them, and
    # every chunk starts on a page boundary (or at the end of an exhausted request)
    lens, parts, bs = [0, 5, 33, 64, 100], [1, 2, 3, 2, 4], 16
    chunks, indptr = orc.plan_chunks(lens, parts, bs)
    assert indptr[0] == 0 and indptr[-1] == len(chunks) == sum(parts)
    for b, (L, P) in enumerate(zip(lens, parts)):
        mine = chunks[indptr[b]:indptr[b + 1]]
        assert len(mine) == P and all(c[0] == b for c in mine)
        hits = np.zeros(L, dtype=int)
        for _, t0, t1 in mine:
            assert t0 % bs == 0 or t0 == L
            hits[t0:t1] += 1
        assert np.all(hits == 1)
        starts = [t0 for _, t0, _ in mine]
        assert starts == sorted(starts)


# --- split + merge -----------------------------------------------------------------

@pytest.mark.parametrize("chunk_len", [1, 7, 8, 29, 90])
def test_split_merge_equals_unsplit_every_chunk_length(chunk_len):
    """mlxcel PR #995: split_kv matches the reference at every chunk length."""
    case = small_case(seed=8, lens=(90, 41), H=2, q_len=3, causal=True)
    ref, ref_lse = orc.unsplit(case)
    chunks, indptr = [], [0]
    for b, L in enumerate(case.context_lens):
        t = 0
        while t < L:
            chunks.append((b, t, min(t + chunk_len, int(L))))
            t += chunk_len
        indptr.append(len(chunks))
    part, lse = orc.partials(case, chunks)
    out, out_lse = orc.merge(part, lse, indptr)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out_lse, ref_lse, rtol=0, atol=1e-12)


def test_merge_weights_are_base_two():
    """Two partials whose LSEs differ by exactly 1 merge with weights 2:1."""
    a = np.full((1, 1, 1, 4), 3.0)
    b = np.full((1, 1, 1, 4), -6.0)
    part = np.concatenate([a, b])
    lse = np.array([[[5.0]], [[4.0]]])
    out, out_lse = orc.merge(part, lse, [0, 2])
    np.testing.assert_allclose(out[0, 0, 0], (2 * 3.0 + 1 * -6.0) / 3.0, atol=1e-15)
    assert abs(out_lse[0, 0, 0] - (5.0 + math.log2(1.5))) < 1e-15


def test_merge_is_associative_across_regroupings():
    case = small_case(seed=9, lens=(120,), H=2)
    chunks = [(0, 0, 33), (0, 33, 70), (0, 70, 120)]
    part, lse = orc.partials(case, chunks)
    all3, all3_lse = orc.merge(part, lse, [0, 3])
    ab, ab_lse = orc.merge(part[:2], lse[:2], [0, 2])
    left, left_lse = orc.merge(np.concatenate([ab, part[2:]]), np.concatenate([ab_lse, lse[2:]]), [0, 2])
    bc, bc_lse = orc.merge(part[1:], lse[1:], [0, 2])
    right, right_lse = orc.merge(np.concatenate([part[:1], bc]), np.concatenate([lse[:1], bc_lse]), [0, 2])
    for x, y in ((left, all3), (right, all3), (left_lse, all3_lse), (right_lse, all3_lse)):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


def test_natural_log_lse_merge_is_wrong_by_a_wide_margin():
    """Negative control (mlxcel PR #995, merge_rejects_natural_log_lse_units)."""
    case = small_case(seed=10, lens=(64,), H=2)
    # shift chunk 0's scores up: unequal LSEs so the wrong units cannot pass by symmetry
    chunks = [(0, 0, 32), (0, 32, 64)]
    part, lse = orc.partials(case, chunks)
    lse = lse.copy()
    lse[0] += 3.0 / math.log(2)
    good, _ = orc.merge(part, lse, [0, 2])
    bad, _ = orc.merge_natural_log(part, lse, [0, 2])
    # weights differ: w0/w1 = 2^d (log2) vs 2^(d ln2) (natural log fed as log2)
    err = np.abs(good - bad).max()
    assert err > 10 * 2e-3
    # and the correct merge is unaffected by adding the same constant to every LSE
    good2, _ = orc.merge(part, lse + 7.25, [0, 2])
    np.testing.assert_allclose(good2, good, atol=1e-13)


def test_empty_chunks_and_all_empty_rows():
    case = small_case(seed=11, lens=(20,), H=2)
    part, lse = orc.partials(case, [(0, 0, 20), (0, 20, 20)])
    assert np.all(lse[1] == -math.inf) and np.all(part[1] == 0)
    out, out_lse = orc.merge(part, lse, [0, 2])
    ref, ref_lse = orc.unsplit(case)
    np.testing.assert_allclose(out[0], ref[0], atol=1e-13)
    out0, lse0 = orc.merge(part[1:], lse[1:], [0, 1])
    assert np.all(out0 == 0) and np.all(lse0 == -math.inf)


def test_causal_mask_positive_control():
    """mlxcel PR #995: the masked test must not pass on a no-op mask."""
    case = small_case(seed=12, lens=(40,), H=2, q_len=8, causal=True)
    masked, _ = orc.unsplit(case)
    case.causal = False
    unmasked, _ = orc.unsplit(case)
    assert np.abs(masked - unmasked).max() > 0.05
    # the last row sees every token either way
    np.testing.assert_allclose(masked[0, -1], unmasked[0, -1], atol=1e-13)


def test_paging_invariance():
    case = small_case(seed=13, lens=(77, 5), H=2, q_len=2, causal=True)
    a, la = orc.unsplit(case)
    b, lb = orc.unsplit(gen.permute_pool(case, seed=99))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_segments_merge_to_the_concatenated_sequence():
    seg = gen.make_segmented_case(14, B=2, q_len=3, segment_tokens=(40, 24, 16), num_heads=2,
                                  block_size=8)
    whole = gen.concat_segments(seg)
    ref, ref_lse = orc.unsplit(whole)
    parts, lses = [], []
    for s in seg.segments:
        p, l = orc.partials(s, [(b, 0, int(s.context_lens[b])) for b in range(2)])
        parts.append(p)
        lses.append(l)
    # regroup request-major: request b's partials are the segments in order
    P = np.stack(parts, axis=1).reshape((-1,) + parts[0].shape[1:])
    Ls = np.stack(lses, axis=1).reshape((-1,) + lses[0].shape[1:])
    out, out_lse = orc.merge(P, Ls, [0, 4, 8])
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(out_lse, ref_lse, atol=1e-12)


# --- the fold (pre-absorption reference) ------------------------------------------

def test_absorbed_equals_decompressed_and_transposed_fold_does_not():
    rng = np.random.default_rng(15)
    H, n, r, v, dr, T = 3, 128, 512, 128, 64, 23
    q_nope = rng.standard_normal((H, n))
    q_pe = rng.standard_normal((H, dr))
    W_UK = rng.standard_normal((H, n, r)) / math.sqrt(r)
    W_UV_T = rng.standard_normal((H, r, v)) / math.sqrt(r)
    ckv = rng.standard_normal((T, r))
    kpe = rng.standard_normal((T, dr))
    sc = 1 / math.sqrt(192)
    ref = orc.decompressed_decode(q_nope, q_pe, W_UK, W_UV_T, ckv, kpe, sc)
    q_abs = orc.absorb_query(q_nope, W_UK)
    lat = np.stack([orc.attend(orc.scores(q_abs[h], q_pe[h], ckv, kpe, sc), ckv)[0] for h in range(H)])
    got = orc.unembed(lat, W_UV_T)
    assert np.abs(got - ref).max() / np.abs(ref).max() < 1e-10
    # A shape-valid slip: folding the wrong matrices (W_UV^T on the query side and
    # W_UK^T on the output side; qk_nope == v_head makes both shapes fit).
    q_abs_wrong = orc.absorb_query(q_nope, np.transpose(W_UV_T, (0, 2, 1)))
    lat_w = np.stack([orc.attend(orc.scores(q_abs_wrong[h], q_pe[h], ckv, kpe, sc), ckv)[0]
                      for h in range(H)])
    bad = orc.unembed(lat_w, np.transpose(W_UK, (0, 2, 1)))
    assert np.abs(bad - ref).max() / np.abs(ref).max() > 1e-2


# --- memory figures printed on the mlxcel page -------------------------------------

def test_kv_memory_table_matches_printed_figures():
    g = json.load(open(os.path.join(GOLDEN, "kv_memory_mlxcel995.json")))
    geo = g["geometry_read_for_the_pin"]
    st = g["geometry_stated_on_page"]
    lat = orc.latent_elems_per_token(st["kv_lora_rank"], st["qk_rope_head_dim"])
    dec = orc.decompressed_elems_per_token(geo["num_heads"], geo["qk_head_dim"], geo["v_head_dim"])
    assert lat == g["printed"]["latent_elems_per_token_per_layer"]
    assert f"{dec / lat:.2f}x" == g["printed"]["kv_bytes_ratio"]
    assert orc.max_context_tokens(geo["budget_bytes"], dec, geo["elem_bytes"], st["num_layers"]) \
        == g["printed"]["max_context_tokens_under_16GiB_decompressed"]
    assert orc.max_context_tokens(geo["budget_bytes"], lat, geo["elem_bytes"], st["num_layers"]) \
        == g["printed"]["max_context_tokens_under_16GiB_latent"]


# --- the steps either side of attention ----------------------------------------------

def test_cache_append_hand_table():
    """Two requests, pages of 4 tokens: each new token lands at the hand-computed physical row, nothing else
    moves, and a position before the start of the context is not written."""
    ckv = np.zeros((6, 4, 2), dtype=np.uint16)
    kpe = np.zeros((6, 4, 1), dtype=np.uint16)
    bt = np.array([[5, 2, -1], [0, 3, 1]], dtype=np.int32)
    lens = np.array([6, 1], dtype=np.int32)  # request 0: tokens 4, 5 are new; request 1: only token 0 exists
    new_c = np.array([[[11, 12], [13, 14]], [[21, 22], [23, 24]]], dtype=np.uint16)
    new_k = np.array([[[1], [2]], [[3], [4]]], dtype=np.uint16)
    c2, k2 = orc.cache_append(ckv, kpe, bt, lens, new_c, new_k, 4)
    want_c = ckv.copy()
    want_k = kpe.copy()
    want_c[2, 0] = [11, 12]  # b=0, t=4: page 2 (block_table[0][1]), slot 0
    want_c[2, 1] = [13, 14]  # b=0, t=5: page 2, slot 1
    want_k[2, 0] = [1]
    want_k[2, 1] = [2]
    want_c[0, 0] = [23, 24]  # b=1, i=1 -> t=0: page 0 slot 0; i=0 -> t=-1 is not written
    want_k[0, 0] = [4]
    assert np.array_equal(c2, want_c) and np.array_equal(k2, want_k)
    assert np.array_equal(ckv, np.zeros_like(ckv))  # the inputs are not modified


def test_cache_append_of_the_cached_tail_is_the_identity_and_shifted_rows_are_not():
    case = gen.make_decode_case(17, [77, 130, 31], num_heads=16, q_len=3, block_size=16, dtype="f16")
    q = 3
    tail_c = np.stack([case.ckv.reshape(-1, 512)[orc.physical_rows(case.block_table[b], int(L), 16)[-q:]]
                       for b, L in enumerate(case.context_lens)])
    tail_k = np.stack([case.kpe.reshape(-1, 64)[orc.physical_rows(case.block_table[b], int(L), 16)[-q:]]
                       for b, L in enumerate(case.context_lens)])
    c2, k2 = orc.cache_append(case.ckv, case.kpe, case.block_table, case.context_lens, tail_c, tail_k, 16)
    assert np.array_equal(c2, case.ckv) and np.array_equal(k2, case.kpe)
    # the rows one position earlier are different data: writing them there changes the cache
    prev_c = np.stack([case.ckv.reshape(-1, 512)[orc.physical_rows(case.block_table[b], int(L), 16)[-q - 1:-1]]
                       for b, L in enumerate(case.context_lens)])
    c3, _ = orc.cache_append(case.ckv, case.kpe, case.block_table, case.context_lens, prev_c, tail_k, 16)
    assert not np.array_equal(c3, case.ckv)


def test_merge_unembed_is_the_decompressed_decode_of_a_split():
    """Split the context, merge with the unembed: the decompressed (pre-absorption) decode of the whole
    context, to 1e-10."""
    rng = np.random.default_rng(18)
    H, n, r, v, dr, T = 2, 128, 512, 128, 64, 37
    q_nope = rng.standard_normal((H, n))
    q_pe = rng.standard_normal((H, dr))
    W_UK = rng.standard_normal((H, n, r)) / math.sqrt(r)
    W_UV_T = rng.standard_normal((H, r, v)) / math.sqrt(r)
    ckv = rng.standard_normal((T, r))
    kpe = rng.standard_normal((T, dr))
    sc = 1 / math.sqrt(192)
    ref = orc.decompressed_decode(q_nope, q_pe, W_UK, W_UV_T, ckv, kpe, sc)
    q_abs = orc.absorb_query(q_nope, W_UK)
    parts, lses = [], []
    for t0, t1 in [(0, 16), (16, 32), (32, T)]:
        row = [orc.attend(orc.scores(q_abs[h], q_pe[h], ckv[t0:t1], kpe[t0:t1], sc), ckv[t0:t1]) for h in range(H)]
        parts.append(np.stack([o for o, _ in row])[None])
        lses.append(np.array([l for _, l in row])[None])
    P = np.stack(parts)   # [3, 1, H, r]
    L = np.stack(lses)    # [3, 1, H]
    ov, _ = orc.merge_unembed(P, L, [0, 3], W_UV_T)
    assert np.abs(ov[0, 0] - ref).max() / np.abs(ref).max() < 1e-10
    # the transposed projection (a shape-valid slip when r == v would not apply; here use the wrong head)
    bad, _ = orc.merge_unembed(P, L, [0, 3], W_UV_T[::-1])
    assert np.abs(bad[0, 0] - ref).max() / np.abs(ref).max() > 1e-2
