"""The steps either side of attention on the GPU: the paged cache write and the merge with the unembed.

mla_cache_append must leave the device caches bit-identical to the oracle's
cache_append on the same bits. mla_merge_unembed must match the oracle's
merge_unembed (f64) within the stated tolerance (max-abs 2e-3, rel-L2 1e-3 on
fp32 results), reproduce the fp32 product of mla_merge_states' own output to
fp32 rounding, give the merged LSE bit for bit, and round a 16-bit output once.
"""
import dataclasses
import math

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
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rel:.3e}"


def new_tokens(seed, B, q_len, dtype):
    rng = np.random.default_rng(seed)
    return (gen.to_bits(rng.standard_normal((B, q_len, 512)), dtype),
            gen.to_bits(rng.standard_normal((B, q_len, 64)), dtype))


def append_on_device(case, dc, ckv_new, kpe_new, q_len):
    cn = rt.to_device_16(ckv_new, case.dtype, "cuda")
    kn = rt.to_device_16(kpe_new, case.dtype, "cuda")
    nb.mla_cache_append(cn.data_ptr(), kn.data_ptr(), dc.block_table.data_ptr(), dc.context_lens.data_ptr(),
                        case.num_requests, q_len, case.block_size, case.num_blocks, case.max_blocks,
                        dc.ckv.data_ptr(), dc.kpe.data_ptr(), None)


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("bs,q_len,dtype", [(16, 1, "f16"), (32, 4, "f16"), (64, 3, "bf16"), (32, 32, "f16")])
def test_cache_append_matches_the_oracle_bit_for_bit(bs, q_len, dtype):
    lens = [0, 2, 31, 33, 1000, 4133]  # a context shorter than the window: its early positions are skipped
    case = gen.make_decode_case(41, lens, num_heads=16, q_len=q_len, block_size=bs, dtype=dtype)
    dc = rt.upload(case)
    ckv_new, kpe_new = new_tokens(42, len(lens), q_len, dtype)
    nb.mla_reset_counters()
    append_on_device(case, dc, ckv_new, kpe_new, q_len)
    assert nb.mla_get_counters()[nb.CTR_WRAP] == 1
    want_c, want_k = orc.cache_append(case.ckv, case.kpe, case.block_table, case.context_lens, ckv_new, kpe_new, bs)
    assert np.array_equal(bits(dc.ckv), want_c)
    assert np.array_equal(bits(dc.kpe), want_k)
    assert not np.array_equal(want_c, case.ckv)  # the check sees the writes


def test_cache_append_out_of_range_page_is_flagged_and_not_written():
    case = gen.make_decode_case(43, [100, 64], num_heads=16, block_size=32, dtype="f16")
    case.block_table[0, 3] = case.num_blocks + 7  # the page of request 0's last token
    dc = rt.upload(case)
    ckv_new, kpe_new = new_tokens(44, 2, 1, "f16")
    nb.mla_check_device_errors(None)
    append_on_device(case, dc, ckv_new, kpe_new, 1)
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_ERR_DEVICE_CHECK and code & 2
    # request 1's token was written; nothing else changed
    fixed = case.block_table.copy()
    fixed[0, 3] = -1
    want_c, _ = orc.cache_append(case.ckv, case.kpe, fixed, np.array([0, 64], np.int32), ckv_new[1:2].repeat(2, 0),
                                 kpe_new[1:2].repeat(2, 0), 32)
    assert np.array_equal(bits(dc.ckv), want_c)


def unembed_weights(seed, H, v_head, dtype):
    rng = np.random.default_rng(seed)
    return gen.to_bits(rng.standard_normal((H, 512, v_head)) / math.sqrt(512.0), dtype)


@pytest.mark.parametrize("H,q_len,dtype,v_head", [(16, 1, "f16", 128), (16, 4, "bf16", 64), (128, 1, "bf16", 128),
                                                  (64, 2, "f16", 256)])
def test_merge_unembed_against_the_oracle_and_the_merge(H, q_len, dtype, v_head):
    case = gen.make_decode_case(45, [3000, 1200, 17], num_heads=H, q_len=q_len, block_size=32, dtype=dtype,
                                latent_std=0.5, causal=q_len > 1)
    dc = rt.upload(case)
    B, P = case.num_requests, 3
    part, lse = rt.alloc_partials(B * P, q_len, H)
    rt.decode_partial(dc, part, lse, num_partitions=P, kernel=nb.MLA_KERNEL_TC, cluster=2)
    ind = rt.uniform_indptr(B, P)
    w_bits = unembed_weights(46, H, v_head, dtype)
    w = rt.to_device_16(w_bits, dtype, "cuda")
    out = torch.empty((B, q_len, H, v_head), dtype=torch.float32, device="cuda")
    out_lse = torch.empty((B, q_len, H), dtype=torch.float32, device="cuda")
    nb.mla_merge_unembed(part.data_ptr(), lse.data_ptr(), ind.data_ptr(), B, q_len, H, w.data_ptr(),
                         nb.DTYPE_CODES[dtype], v_head, out.data_ptr(), nb.MLA_F32, out_lse.data_ptr(), None)
    # 1. the oracle: merge of the exact partials, then the unembed, all in f64
    chunks, indptr = orc.plan_chunks(case.context_lens, [P] * B, case.block_size)
    ref_part, ref_lse = orc.partials(case, chunks)
    W = orc.decode16(w_bits, dtype)
    ref, ref_out_lse = orc.merge_unembed(ref_part, ref_lse, indptr, W)
    assert_close(out.cpu().numpy(), ref, f"merge+unembed H={H} q={q_len} {dtype}")
    # 2. the merge kernel's own fp32 output times W (f64 on the host): the same up to fp32 rounding
    lat_lse = torch.empty_like(out_lse)
    lat = rt.merge_states(part, lse, ind, B, q_len, H, "f32", out_lse=lat_lse).cpu().double().numpy()
    prod = np.einsum("biHr,Hrv->biHv", lat, W)
    assert np.abs(out.cpu().double().numpy() - prod).max() <= 1e-5 * max(1.0, np.abs(prod).max())
    assert torch.equal(out_lse, lat_lse)  # the merged LSE, bit for bit
    # 3. a 16-bit output is the fp32 output rounded once
    out16 = torch.empty((B, q_len, H, v_head), dtype=rt.TORCH_DTYPE[dtype], device="cuda")
    nb.mla_merge_unembed(part.data_ptr(), lse.data_ptr(), ind.data_ptr(), B, q_len, H, w.data_ptr(),
                         nb.DTYPE_CODES[dtype], v_head, out16.data_ptr(), nb.DTYPE_CODES[dtype], None, None)
    assert torch.equal(out16, out.to(out16.dtype))


def test_layer_call_append_decode_unembed():
    """A whole decode layer call on the device: write the new token into its page, the partial decode over the
    cache that now holds it, then the merge with the unembed; against the oracle doing the same steps."""
    lens = [20000, 7777]
    case = gen.make_decode_case(47, lens, num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    ckv_new, kpe_new = new_tokens(48, 2, 1, "f16")
    append_on_device(case, dc, ckv_new, kpe_new, 1)
    c2, k2 = orc.cache_append(case.ckv, case.kpe, case.block_table, case.context_lens, ckv_new, kpe_new, 32)
    after = dataclasses.replace(case, ckv=c2, kpe=k2)
    plan = nb.mla_plan(lens, 16, 1, 32, nb.mla_device_query())
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    part, lse = rt.alloc_partials(plan.num_chunks, 1, 16)
    ws = rt.alloc_workspace(plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, 16)
    rt.decode_partial(dc, part, lse, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas, chunks_dev=chunks,
                      subs=plan.clusters_per_chunk, workspace=ws)
    w_bits = unembed_weights(49, 16, 128, "f16")
    w = rt.to_device_16(w_bits, "f16", "cuda")
    ov = torch.empty((2, 1, 16, 128), dtype=torch.float32, device="cuda")
    nb.mla_merge_unembed(part.data_ptr(), lse.data_ptr(), ind.data_ptr(), 2, 1, 16, w.data_ptr(), nb.MLA_F16, 128,
                         ov.data_ptr(), nb.MLA_F32, None, None)
    heads = [0, 11]
    lat, _ = orc.unsplit(after, heads=heads)
    W = orc.decode16(w_bits, "f16")
    ref = np.stack([np.stack([orc.unembed(lat[b, 0][heads], W[heads])]) for b in range(2)])
    assert_close(ov.cpu().numpy()[:, :, heads], ref, "layer call")


@pytest.mark.parametrize("counts,q_len,H", [
    ([300, 0, 129, 1], 1, 16),   # more partials than one piece of weights, an empty request, a single partial
    ([5, 140, 0, 64, 2] * 4, 2, 64),  # 40 rows of a head: two full row groups and a ragged one
])
def test_merge_unembed_many_partials(counts, q_len, H):
    """Partials written straight into the buffers (no attention call): some requests with more than 128
    partials, requests with none, and rows whose every partial is empty (LSE -inf)."""
    rng = np.random.default_rng(50)
    B, S = len(counts), sum(counts)
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    part_np = rng.standard_normal((S, q_len, H, 512)).astype(np.float32)
    lse_np = (rng.standard_normal((S, q_len, H)) * 4.0).astype(np.float32)
    lse_np[rng.random((S, q_len, H)) < 0.2] = -np.inf  # empty partials
    lse_np[int(indptr[3]):int(indptr[4]), :, 1] = -np.inf  # request 3, head 1: every partial empty
    part_np[np.isinf(lse_np)] = 0.0
    part = torch.from_numpy(part_np).cuda()
    lse = torch.from_numpy(lse_np).cuda()
    ind = torch.from_numpy(indptr).cuda()
    w_bits = unembed_weights(51, H, 64, "bf16")
    w = rt.to_device_16(w_bits, "bf16", "cuda")
    out = torch.empty((B, q_len, H, 64), dtype=torch.float32, device="cuda")
    out_lse = torch.empty((B, q_len, H), dtype=torch.float32, device="cuda")
    nb.mla_merge_unembed(part.data_ptr(), lse.data_ptr(), ind.data_ptr(), B, q_len, H, w.data_ptr(), nb.MLA_BF16,
                         64, out.data_ptr(), nb.MLA_F32, out_lse.data_ptr(), None)
    W = orc.decode16(w_bits, "bf16")
    ref, ref_lse = orc.merge_unembed(part_np.astype(np.float64), lse_np.astype(np.float64), indptr, W)
    assert_close(out.cpu().numpy(), ref, f"many partials B={B} q={q_len} H={H}")
    got_lse = out_lse.cpu().numpy()
    assert np.array_equal(np.isinf(got_lse), np.isinf(ref_lse))
    fin = np.isfinite(ref_lse)
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= 1e-5 * max(1.0, np.abs(ref_lse[fin]).max())
    # the merge kernel's own latent times W, and its LSE bit for bit
    lat_lse = torch.empty_like(out_lse)
    lat = rt.merge_states(part, lse, ind, B, q_len, H, "f32", out_lse=lat_lse).cpu().double().numpy()
    prod = np.einsum("biHr,Hrv->biHv", lat, W)
    assert np.abs(out.cpu().double().numpy() - prod).max() <= 1e-5 * max(1.0, np.abs(prod).max())
    assert torch.equal(out_lse, lat_lse)
    empty = [b for b in range(B) if counts[b] == 0]
    assert empty and not out[empty].any() and not out[3, :, 1].any()  # no partials, or only empty ones: zero


TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.mark.parametrize("lens,H,dtype,v_head,P,C,k", [
    ([32768], 16, "f16", 128, None, None, None),      # the planner's plan on the paired kernel (pair entries)
    ([131072], 16, "bf16", 64, None, None, None),
    ([700, 0, 5000, 64], 16, "f16", 256, 2, 2, 2),    # several requests, an empty one, spread partitions
    ([200000], 16, "f16", 32, 16, 2, 9),              # 144 entries: more than one piece of weights
    ([3000, 1200], 128, "bf16", 128, None, None, None),  # the 128-row kernel: chunk partials, then the merge
    ([2000, 900], 64, "f16", 512, None, None, None),   # the largest v_head (16 blocks of 32 columns)
    ([300 + 97 * b for b in range(20)], 16, "f16", 96, None, None, None),  # 20 rows a head: two row groups
])
def test_decode_unembed_against_the_oracle_and_mla_decode(lens, H, dtype, v_head, P, C, k):
    """mla_decode_unembed: the oracle's unembed of the exact attention on sampled heads; mla_decode's own fp32
    latent times W to fp32 rounding, its LSE bit for bit; a 16-bit output that is the fp32 one rounded once."""
    case = gen.make_decode_case(52, lens, num_heads=H, block_size=32, dtype=dtype, latent_std=0.5)
    dc = rt.upload(case)
    B = len(lens)
    if P is None:
        plan = nb.mla_plan(lens, H, 1, 32, nb.mla_device_query(), dtype=dtype)
        N, C, k = plan.num_chunks, plan.cluster_ctas, plan.clusters_per_chunk
        kw = dict(chunks_dev=rt.chunks_to_device(plan.chunks), cluster=C, subs=k)
        ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
        nparts = 1
    else:
        N, nparts = B * P, P
        kw = dict(cluster=C, subs=k)
        ind = rt.uniform_indptr(B, P)
    ws = rt.alloc_decode_workspace(B, N, k, C, 1, H)
    kw.update(kernel=nb.MLA_KERNEL_TC, workspace=ws, tables_ready=True)
    w_bits = unembed_weights(53, H, v_head, dtype)
    w = rt.to_device_16(w_bits, dtype, "cuda")
    W = orc.decode16(w_bits, dtype)
    res = {}
    for dt in ("f32", dtype):
        part, lse = rt.alloc_partials(N, 1, H)
        out_v = torch.full((B, 1, H, v_head), float("nan"), dtype=TDT[dt], device="cuda")
        out_lse = torch.full((B, 1, H), float("nan"), device="cuda")
        nb.mla_reset_counters()
        rt.decode_unembed(dc, part, lse, ind, w, out_v, out_lse, num_partitions=nparts, **kw)
        ctr = nb.mla_get_counters()
        assert ctr[nb.CTR_PARTIAL_TC] == 1 and ctr[nb.CTR_WRAP] == 1 and ctr[nb.CTR_MERGE] == 0
        res[dt] = (out_v, out_lse)
    out_v, out_lse = res["f32"]
    assert torch.equal(res[dtype][0], out_v.to(TDT[dtype])) and torch.equal(res[dtype][1], out_lse)
    # mla_decode's fp32 latent on the same plan, times W
    part, lse = rt.alloc_partials(N, 1, H)
    lat = torch.empty((B, 1, H, 512), dtype=torch.float32, device="cuda")
    lat_lse = torch.empty((B, 1, H), dtype=torch.float32, device="cuda")
    rt.decode(dc, part, lse, ind, lat, lat_lse, num_partitions=nparts, **kw)
    prod = np.einsum("biHr,Hrv->biHv", lat.cpu().double().numpy(), W)
    assert np.abs(out_v.cpu().double().numpy() - prod).max() <= 1e-5 * max(1.0, np.abs(prod).max())
    assert torch.equal(out_lse, lat_lse)
    # the oracle on sampled heads
    heads = [0, H // 2 - 1, H - 1]
    ref_lat, ref_lse = orc.unsplit(case, heads=heads)
    ref = np.stack([np.stack([orc.unembed(ref_lat[b, 0][heads], W[heads])]) for b in range(B)])
    got = out_v.cpu().numpy()[:, :, heads]
    live = [b for b, L in enumerate(lens) if L > 0]
    assert_close(got[live], ref[live], f"decode+unembed {lens} H={H} {dtype}")
    got_lse = out_lse.cpu().numpy()[:, :, heads]
    assert np.abs(got_lse[live] - ref_lse[:, :, heads][live]).max() <= MAX_ABS
    for b, L in enumerate(lens):
        if L == 0:
            assert not out_v[b].any() and torch.all(torch.isneginf(out_lse[b]))
