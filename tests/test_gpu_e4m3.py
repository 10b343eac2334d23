"""GPU parity for 8-bit E4M3 latent caches on the paired 16-row kernel.

The oracle reads each cache byte as its exact E4M3 value times the cache
scale. The kernel loads the bytes, widens them to fp16 in shared memory
(exact: every E4M3 value is an fp16 value) and folds the scale into the score
scale and the output. From the widening on, the arithmetic is the fp16 path's
(plus one rounding of each folded product), so the tolerance is the one stated
for 16-bit inputs with fp32 accumulation: max-abs 2e-3 and rel-L2 1e-3 on fp32
results, max-abs 2e-3 on every finite log2 LSE. And since scaling by a power
of two commutes with every rounding, for such a scale the same bytes widened
on the host into an fp16 cache holding value * scale must give the fp16 path's
results bit for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

from mla_split_kv_gb300 import binding as nb
from mla_split_kv_gb300 import build as nbuild
from mla_split_kv_gb300 import inputs as gen
from mla_split_kv_gb300 import runtime as rt
from oracle import mla_oracle as orc

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    nbuild.build()
    nb.load()
    yield
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_OK, f"device error word {code:#x}"


def assert_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref).max() if got.size else 0.0
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nrm if nrm > 0 else np.linalg.norm(got - ref)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rel:.3e}"


def assert_lse_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf), f"{what}: -inf pattern differs"
    if (~inf).any():
        err = np.abs(got[~inf] - ref[~inf]).max()
        assert err <= MAX_ABS, f"{what}: lse max-abs {err:.3e}"


def widened_f16(case):
    """The same cache as fp16 patterns of value * scale (exact for the scales used here), same queries."""
    ckv = gen.to_bits(orc.decode_cache(case.ckv, case), "f16")
    kpe = gen.to_bits(orc.decode_cache(case.kpe, case), "f16")
    assert np.array_equal(orc.decode16(ckv, "f16"), orc.decode_cache(case.ckv, case))  # exact
    return dataclasses.replace(case, dtype="f16", ckv=ckv, kpe=kpe, cache_scale=1.0)


def uniform(case, P, C, dc=None, subs=1, exchange=0):
    dc = dc or rt.upload(case)
    B, q, H = case.num_requests, case.q_len, case.num_heads
    part, lse = rt.alloc_partials(B * P, q, H)
    part.fill_(float("nan"))
    ws = rt.alloc_workspace(B * P, subs, C, q, H) if subs > 1 else None
    rt.decode_partial(dc, part, lse, num_partitions=P, kernel=nb.MLA_KERNEL_TC, cluster=C, subs=subs, workspace=ws,
                      score_exchange=exchange)
    ind = rt.uniform_indptr(B, P)
    out = rt.merge_states(part, lse, ind, B, q, H, "f32")
    return part, lse, out


@pytest.mark.parametrize("lens,bs,P,C,cs", [
    ([4096], 32, 2, 2, 0.25),
    ([1, 127, 128, 129, 1000], 16, 1, 2, 0.25),   # one token, a tile less one, a tile, a ragged tail
    ([5000, 300, 0], 64, 3, 4, 2.0 ** -6),        # an empty request
    ([20000], 32, 4, 8, 0.125),
    ([777, 4133], 16, 2, 16, 0.25),
    ([3000, 129], 32, 2, 2, 0.3),                 # a scale that is not a power of two
])
def test_e4m3_partials_and_merge_against_the_oracle(lens, bs, P, C, cs):
    case = gen.make_decode_case(61, lens, num_heads=16, block_size=bs, dtype="e4m3", cache_scale=cs)
    nb.mla_reset_counters()
    part, lse, out = uniform(case, P, C)
    assert nb.mla_get_counters()[nb.CTR_PARTIAL_TC] == 1
    chunks, _ = orc.plan_chunks(case.context_lens, [P] * case.num_requests, bs)
    ref_part, ref_lse = orc.partials(case, chunks)
    assert_close(part.cpu().numpy(), ref_part, f"e4m3 partials {lens} bs={bs} C={C}")
    assert_lse_close(lse.cpu().numpy(), ref_lse, "e4m3 lse")
    ref, _ = orc.unsplit(case)
    live = case.context_lens > 0
    assert_close(out.cpu().numpy()[live], ref[live], "e4m3 merged")


@pytest.mark.parametrize("lens,bs,P,C,subs,cs", [
    ([9000, 129], 32, 2, 2, 1, 0.25),
    ([4133], 16, 3, 4, 1, 16.0),
    ([20017, 3000], 64, 2, 2, 3, 2.0 ** -5),     # partitions spread over clusters (workspace merge)
    ([1000, 1, 0], 32, 1, 8, 1, 1.0),
])
def test_e4m3_equals_the_fp16_path_on_the_widened_cache(lens, bs, P, C, subs, cs):
    """The same bits as the fp16 kernel given value * scale as an fp16 cache: the widening is exact and the
    scale, a power of two, commutes with every rounding."""
    case = gen.make_decode_case(62, lens, num_heads=16, block_size=bs, dtype="e4m3", cache_scale=cs)
    got = uniform(case, P, C, subs=subs)
    want = uniform(widened_f16(case), P, C, subs=subs)
    for g, w in zip(got, want):
        assert torch.equal(g, w)


def test_e4m3_bitwise_repeatable_and_prefix_ready():
    """One plan, repeated: the same bits; loading the first tiles before the dependency wait (tables_ready,
    prefix_ready) changes nothing."""
    lens = [30000, 1500]
    case = gen.make_decode_case(63, lens, num_heads=16, block_size=32, dtype="e4m3")
    dc = rt.upload(case)
    plan = nb.mla_plan(lens, 16, 1, 32, nb.mla_device_query(), dtype="e4m3")
    assert plan.cluster_ctas >= 2
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    outs = []
    for ready in (False, False, True):
        part, lse = rt.alloc_partials(plan.num_chunks, 1, 16)
        out = torch.empty((2, 1, 16, 512), device="cuda")
        ws = rt.alloc_decode_workspace(2, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, 16)
        rt.decode(dc, part, lse, ind, out, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas, chunks_dev=chunks,
                  subs=plan.clusters_per_chunk, workspace=ws, tables_ready=ready, prefix_ready=ready)
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    heads = [0, 9, 15]
    ref, _ = orc.unsplit(case, heads=heads)
    assert_close(outs[0].cpu().numpy()[:, :, heads], ref[:, :, heads], "e4m3 decode")


@pytest.mark.parametrize("way", [nb.MLA_DECODE_MERGE_ENTRIES, nb.MLA_DECODE_MERGE_TICKETS])
@pytest.mark.parametrize("L", [32768, 131072])
def test_e4m3_decode_ways_on_the_planner_plan(way, L):
    """mla_decode on the planner's plan for one long request, both ways: the oracle on sampled heads, and the
    fp16 path's bits on the widened cache."""
    case = gen.make_decode_case(64, [L], num_heads=16, block_size=32, dtype="e4m3")
    plan = nb.mla_plan([L], 16, 1, 32, nb.mla_device_query(), dtype="e4m3")
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    outs = []
    for c in (case, widened_f16(case)):
        dc = rt.upload(c)
        part, lse = rt.alloc_partials(plan.num_chunks, 1, 16)
        out = torch.empty((1, 1, 16, 512), device="cuda")
        out_lse = torch.empty((1, 1, 16), device="cuda")
        ws = rt.alloc_decode_workspace(1, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, 16)
        rt.decode(dc, part, lse, ind, out, out_lse, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas,
                  chunks_dev=chunks, subs=plan.clusters_per_chunk, workspace=ws, tables_ready=True, decode_merge=way)
        outs.append((out, out_lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    heads = [0, 5, 15]
    ref, ref_lse = orc.unsplit(case, heads=heads)
    assert_close(outs[0][0].cpu().numpy()[:, :, heads], ref[:, :, heads], f"e4m3 L={L} way={way}")
    assert_lse_close(outs[0][1].cpu().numpy()[:, :, heads], ref_lse[:, :, heads], "e4m3 out lse")


def test_e4m3_out_of_range_page_reads_zeros_and_is_flagged():
    case = gen.make_decode_case(65, [300, 200], num_heads=16, block_size=32, dtype="e4m3")
    case.block_table[0, 2] = case.num_blocks + 3  # tokens 64-95 of request 0
    nb.mla_check_device_errors(None)
    part, lse, out = uniform(case, 1, 2)
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_ERR_DEVICE_CHECK and code & 2
    # the oracle over the same request with that page's rows as zeros
    fixed = dataclasses.replace(case, ckv=case.ckv.copy(), kpe=case.kpe.copy(), block_table=case.block_table.copy())
    spare = min(set(range(case.num_blocks)) - set(case.block_table[case.block_table >= 0].tolist()))
    fixed.ckv[spare] = 0
    fixed.kpe[spare] = 0
    fixed.block_table[0, 2] = spare
    ref, _ = orc.unsplit(fixed)
    assert_close(out.cpu().numpy(), ref, "e4m3 bad page")


@pytest.mark.parametrize("H,q_len,bs,lens,cs,exchange,heads", [
    (128, 1, 64, [9000, 2500, 130], 0.25, 0, [0, 45, 90, 127]),   # the many-head shape on E4M3 caches
    (64, 1, 32, [5000, 777], 2.0 ** -4, 0, None),                  # a 64-row group
    (16, 4, 32, [4000, 2000], 0.25, 0, None),                      # a verify window: 64 rows, causal
    (16, 16, 16, [3000, 1000], 0.5, 0, [0, 8, 15]),                # 256 rows: two 128-row groups, causal
    (128, 1, 64, [6000, 1000], 0.25, 1, [3, 64, 126]),             # with the fp16 score exchange
])
def test_e4m3_many_rows_against_the_oracle_and_the_fp16_path(H, q_len, bs, lens, cs, exchange, heads):
    """More than 16 rows: the 128-row kernel's pairs widen the tiles in place as the 16-row kernel does. Against
    the oracle, and (power-of-two scales) the fp16 path's bits on the host-widened cache."""
    case = gen.make_decode_case(66, lens, num_heads=H, q_len=q_len, block_size=bs, dtype="e4m3", cache_scale=cs,
                                causal=q_len > 1)
    nb.mla_reset_counters()
    got = uniform(case, 2, 2, exchange=exchange)
    assert nb.mla_get_counters()[nb.CTR_PARTIAL_TC] == 1
    hs = heads if heads is not None else list(range(H))
    chunks, _ = orc.plan_chunks(case.context_lens, [2] * case.num_requests, bs)
    if heads is None:
        ref_part, ref_lse = orc.partials(case, chunks)
        assert_close(got[0].cpu().numpy(), ref_part, f"e4m3 many-row partials H={H} q_len={q_len}")
        assert_lse_close(got[1].cpu().numpy(), ref_lse, "e4m3 many-row lse")
    ref, _ = orc.unsplit(case, heads=hs)
    assert_close(got[2].cpu().numpy()[:, :, hs], ref[:, :, hs], f"e4m3 many-row merged H={H} q_len={q_len}")
    # the fp16 path on the same exchange (the default sends E4M3 caches' partial scores as fp32)
    want = uniform(widened_f16(case), 2, 2,
                   exchange=nb.MLA_SCORE_EXCHANGE_F32 if exchange == nb.MLA_SCORE_EXCHANGE_EXACT else exchange)
    for g, w in zip(got, want):
        assert torch.equal(g, w)
