"""mla_decode's ways on the paired 16-row kernel against the two ABI calls and the oracle.

The default: every CTA pair writes its unnormalized part and the entries merge
kernel combines them; against the f64 oracle within the stated tolerance
(max-abs 2e-3, rel-L2 1e-3 on fp32 results), the same bits on a repeat, and
with prefix_ready the same bits as without it. The single launch
(decode_merge = MLA_DECODE_MERGE_TICKETS): the merge runs inside the partial
kernel with the merge kernel's arithmetic in its order, so the chunk partials,
the LSE and the merged output must be the same bits as mla_decode_partial +
mla_merge_states give.
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
TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


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
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rel:.3e}"


def both_paths(case, dc, chunks_dev, ind, N, kernel, C, k, out_dtype="f16", tables_ready=False, num_partitions=1,
               ws_fused=None, with_lse=True):
    """(partials, lse, out, out_lse) of mla_decode, then of mla_decode_partial + mla_merge_states."""
    B, q, H = case.num_requests, case.q_len, case.num_heads
    res = []
    for fused in (True, False):
        part, lse = rt.alloc_partials(N, q, H)
        part.fill_(float("nan"))
        out = torch.full((B, q, H, 512), float("nan"), dtype=TDT[out_dtype], device="cuda")
        out_lse = torch.full((B, q, H), float("nan"), device="cuda") if with_lse else None
        if fused:
            ws = ws_fused if ws_fused is not None else rt.alloc_decode_workspace(B, N, k, C, q, H)
            desc = rt.make_desc(dc, chunks_dev, kernel, C, None, k, ws, tables_ready, decode_merge=nb.MLA_DECODE_MERGE_TICKETS)
            rt.decode(dc, part, lse, ind, out, out_lse, num_partitions=num_partitions, desc=desc)
        else:
            ws = rt.alloc_workspace(N, k, C, q, H)
            desc = rt.make_desc(dc, chunks_dev, kernel, C, None, k, ws, tables_ready)
            rt.decode_partial(dc, part, lse, num_partitions=num_partitions, desc=desc)
            rt.merge_states(part, lse, ind, B, q, H, out_dtype, out=out, out_lse=out_lse)
        res.append((part, lse, out, out_lse))
    return res


def assert_same_bits(a, b):
    for x, y in zip(a, b):
        if x is not None:
            assert torch.equal(x, y)


@pytest.mark.parametrize("L", [32768, 49152, 65536, 81920, 98304, 131072])
def test_single_launch_equals_two_launches_at_every_bench_context(L):
    """The bench's workload and launch configuration (planner plan, tables read before the dependency wait):
    one launch, the same bits as the two launches, and the oracle on sampled heads."""
    case = gen.make_decode_case(2, [L], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    plan = nb.mla_plan([L], 16, 1, 32, nb.mla_device_query())
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    nb.mla_reset_counters()
    fused, plain = both_paths(case, dc, chunks, ind, plan.num_chunks, nb.MLA_KERNEL_TC, plan.cluster_ctas,
                              plan.clusters_per_chunk, "f16", tables_ready=True)
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_DECODE_FUSED] == 1 and ctr[nb.CTR_PARTIAL_TC] == 2 and ctr[nb.CTR_MERGE] == 1
    assert_same_bits(fused, plain)
    # fp32 output of the fused path against the oracle
    out32 = torch.empty((1, 1, 16, 512), device="cuda")
    part, lse = rt.alloc_partials(plan.num_chunks, 1, 16)
    ws = rt.alloc_decode_workspace(1, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, 16)
    rt.decode(dc, part, lse, ind, out32, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas, chunks_dev=chunks,
              subs=plan.clusters_per_chunk, workspace=ws, tables_ready=True, decode_merge=nb.MLA_DECODE_MERGE_TICKETS)
    heads = [0, 7, 15]
    ref, _ = orc.unsplit(case, heads=heads)
    assert_close(out32.cpu().numpy()[:, :, heads], ref[:, :, heads], f"fused L={L}")
    assert torch.equal(out32.to(torch.float16), fused[2])


@pytest.mark.parametrize("C,bs,out_dtype,dtype", [(2, 16, "f32", "f16"), (4, 32, "f16", "f16"), (8, 64, "bf16", "f16"),
                                                  (16, 32, "f32", "f16"), (2, 32, "f32", "bf16"), (4, 64, "bf16", "bf16")])
def test_single_launch_ragged_batch_with_empty_requests(C, bs, out_dtype, dtype):
    """A batch of ragged requests (empty, one token, partial pages, several tiles) on the uniform split: the
    same bits as the two launches, the oracle on every head, an empty request merges to zeros."""
    lens = [0, 1, 31, 33, 127, 129, 1000, 4133]
    case = gen.make_decode_case(31, lens, num_heads=16, block_size=bs, dtype=dtype,
                                latent_std=0.5 if dtype == "bf16" else 1.0)
    dc = rt.upload(case)
    P, B = 3, len(lens)
    ind = rt.uniform_indptr(B, P)
    fused, plain = both_paths(case, dc, None, ind, B * P, nb.MLA_KERNEL_TC, C, 1, out_dtype, num_partitions=P)
    assert_same_bits(fused, plain)
    ref, ref_lse = orc.unsplit(case)
    out = fused[2].float().cpu().numpy()
    assert np.all(out[0] == 0) and np.all(np.isneginf(fused[3].cpu().numpy()[0]))
    if out_dtype == "f32":
        assert_close(out[1:], ref[1:], f"ragged C={C} bs={bs}")
        got_lse = fused[3].cpu().numpy()[1:]
        assert np.abs(got_lse - ref_lse[1:]).max() <= MAX_ABS


@pytest.mark.parametrize("L,P,C,k,bs", [(20017, 3, 2, 5, 16), (65536, 6, 4, 6, 32), (9000, 2, 16, 2, 32)])
def test_single_launch_with_partitions_spread_over_clusters(L, P, C, k, bs):
    """Partitions spread over k clusters (the workspace merge of each chunk, then the request merge, all in
    one launch), two requests so both request tickets are exercised."""
    case = gen.make_decode_case(32, [L, L // 3], num_heads=16, block_size=bs, dtype="f16")
    dc = rt.upload(case)
    ind = rt.uniform_indptr(2, P)
    fused, plain = both_paths(case, dc, None, ind, 2 * P, nb.MLA_KERNEL_TC, C, k, "f32", num_partitions=P)
    assert_same_bits(fused, plain)
    ref, _ = orc.unsplit(case)
    assert_close(fused[2].cpu().numpy(), ref, f"spread L={L} P={P} C={C} k={k}")


def test_single_launch_bitwise_reproducible_and_workspace_reused():
    case = gen.make_decode_case(33, [131072], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    plan = nb.mla_plan([131072], 16, 1, 32, nb.mla_device_query())
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    ws = rt.alloc_decode_workspace(1, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, 16)
    outs = []
    for _ in range(3):
        part, lse = rt.alloc_partials(plan.num_chunks, 1, 16)
        out = torch.empty((1, 1, 16, 512), dtype=torch.float16, device="cuda")
        rt.decode(dc, part, lse, ind, out, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas, chunks_dev=chunks,
                  subs=plan.clusters_per_chunk, workspace=ws, tables_ready=True, decode_merge=nb.MLA_DECODE_MERGE_TICKETS)
        outs.append((part, lse, out))
    for other in outs[1:]:
        assert_same_bits(outs[0], other)
    torch.cuda.synchronize()
    assert int(ws.view(torch.int32)[: 16].abs().sum()) == 0  # request tickets back at zero


@pytest.mark.parametrize("H,dtype,kernel", [(128, "bf16", nb.MLA_KERNEL_TC), (16, "f16", nb.MLA_KERNEL_SIMT),
                                            (64, "f16", nb.MLA_KERNEL_TC)])
def test_decode_without_the_fused_merge_is_the_two_launches(H, dtype, kernel):
    """Kernels without the fused merge: mla_decode enqueues the partial kernel and the merge kernel."""
    case = gen.make_decode_case(34, [3000, 700], num_heads=H, block_size=64 if dtype == "bf16" else 32, dtype=dtype,
                                latent_std=0.5)
    dc = rt.upload(case)
    ind = rt.uniform_indptr(2, 2)
    nb.mla_reset_counters()
    fused, plain = both_paths(case, dc, None, ind, 4, kernel, 2, 1, "f32", num_partitions=2)
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_DECODE_FUSED] == 0 and ctr[nb.CTR_MERGE] == 2
    assert_same_bits(fused, plain)


def default_decode(case, dc, plan, chunks, ind, out_dtype="f32", ws=None, mode=nb.MLA_DECODE_MERGE_ENTRIES):
    B = case.num_requests
    part, lse = rt.alloc_partials(plan.num_chunks, 1, 16)
    out = torch.empty((B, 1, 16, 512), dtype=TDT[out_dtype], device="cuda")
    out_lse = torch.empty((B, 1, 16), device="cuda")
    if ws is None:
        ws = rt.alloc_decode_workspace(B, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, 16)
    rt.decode(dc, part, lse, ind, out, out_lse, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas, chunks_dev=chunks,
              subs=plan.clusters_per_chunk, workspace=ws, tables_ready=True, decode_merge=mode)
    return out, out_lse


@pytest.mark.parametrize("L", [32768, 49152, 65536, 81920, 98304, 131072])
def test_default_decode_on_the_paired_kernel_every_bench_context(L):
    """mla_decode's default on the paired kernel: every CTA pair writes its unnormalized part and the entries
    merge kernel (a dependent launch) combines them; against the oracle on sampled heads, and the same bits on
    a second call."""
    case = gen.make_decode_case(2, [L], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    plan = nb.mla_plan([L], 16, 1, 32, nb.mla_device_query())
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    nb.mla_reset_counters()
    out, out_lse = default_decode(case, dc, plan, chunks, ind)
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_PARTIAL_TC] == 1 and ctr[nb.CTR_MERGE] == 1 and ctr[nb.CTR_DECODE_FUSED] == 0
    heads = [0, 7, 15]
    ref, ref_lse = orc.unsplit(case, heads=heads)
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], f"default L={L}")
    assert np.abs(out_lse.cpu().numpy()[:, :, heads] - ref_lse[:, :, heads]).max() <= MAX_ABS
    out2, lse2 = default_decode(case, dc, plan, chunks, ind)
    assert torch.equal(out, out2) and torch.equal(out_lse, lse2)


@pytest.mark.parametrize("lens,P,C,k", [([700, 333, 5000], 2, 2, 2), ([1, 64, 65, 9000], 3, 4, 1),
                                        ([20000] * 2, 3, 16, 1), ([0, 3000], 2, 2, 3), ([100000], 9, 2, 11)])
def test_default_decode_several_requests_and_many_entries(lens, P, C, k):
    """Several requests in one call (an empty request merges to zeros), and one request of 99 pair entries
    (more than one round of the merge's loads): the oracle on every row, and a 16-bit output that is the fp32
    output rounded once."""
    case = gen.make_decode_case(35, lens, num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    B = len(lens)
    ind = rt.uniform_indptr(B, P)
    ws = rt.alloc_decode_workspace(B, B * P, k, C, 1, 16)
    res = {}
    for dt in ("f32", "f16"):
        part, lse = rt.alloc_partials(B * P, 1, 16)
        out = torch.full((B, 1, 16, 512), float("nan"), dtype=TDT[dt], device="cuda")
        out_lse = torch.full((B, 1, 16), float("nan"), device="cuda")
        rt.decode(dc, part, lse, ind, out, out_lse, num_partitions=P, kernel=nb.MLA_KERNEL_TC, cluster=C, subs=k,
                  workspace=ws)
        res[dt] = (out, out_lse)
    out, out_lse = res["f32"]
    assert torch.equal(res["f16"][0], out.to(torch.float16)) and torch.equal(res["f16"][1], out_lse)
    ref, ref_lse = orc.unsplit(case) if B > 1 else orc.unsplit(case, heads=[0, 5, 15])
    got = out.cpu().numpy()
    if B == 1:
        got = got[:, :, [0, 5, 15]]
        ref, ref_lse = ref[:, :, [0, 5, 15]], ref_lse[:, :, [0, 5, 15]]
    lse_got = out_lse.cpu().numpy() if B > 1 else out_lse.cpu().numpy()[:, :, [0, 5, 15]]
    live = [i for i, L in enumerate(lens) if L > 0]
    for i, L in enumerate(lens):
        if L == 0:
            assert np.all(got[i] == 0) and np.all(np.isneginf(lse_got[i]))
    assert_close(got[live], ref[live], f"default decode {lens}")
    assert np.abs(lse_got[live] - ref_lse[live]).max() <= MAX_ABS


@pytest.mark.parametrize("C,k,bs,out_dtype", [(2, 1, 16, "f32"), (4, 3, 32, "f16"), (16, 1, 64, "bf16"),
                                              (8, 2, 32, "f32")])
def test_default_decode_ragged_batch_with_empty_requests(C, k, bs, out_dtype):
    """Ragged requests on the uniform split (empty, one token, partial pages, several tiles; with and without
    partitions spread over clusters): the oracle on every head, an empty request merges to zeros, and a
    16-bit output is the fp32 output rounded once."""
    lens = [0, 1, 31, 33, 127, 129, 1000, 4133]
    case = gen.make_decode_case(36, lens, num_heads=16, block_size=bs, dtype="f16")
    dc = rt.upload(case)
    P, B = 3, len(lens)
    ind = rt.uniform_indptr(B, P)
    res = {}
    for dt in ("f32", out_dtype):
        part, lse = rt.alloc_partials(B * P, 1, 16)
        out = torch.empty((B, 1, 16, 512), dtype=TDT[dt], device="cuda")
        out_lse = torch.empty((B, 1, 16), device="cuda")
        ws = rt.alloc_decode_workspace(B, B * P, k, C, 1, 16)
        rt.decode(dc, part, lse, ind, out, out_lse, num_partitions=P, kernel=nb.MLA_KERNEL_TC, cluster=C, subs=k,
                  workspace=ws)
        res[dt] = (out, out_lse)
    out, out_lse = res["f32"]
    ref, ref_lse = orc.unsplit(case)
    got = out.cpu().numpy()
    assert np.all(got[0] == 0) and np.all(np.isneginf(out_lse.cpu().numpy()[0]))
    assert_close(got[1:], ref[1:], f"default ragged C={C} k={k} bs={bs}")
    assert np.abs(out_lse.cpu().numpy()[1:] - ref_lse[1:]).max() <= MAX_ABS
    assert torch.equal(res[out_dtype][0], out.to(TDT[out_dtype]))


@pytest.mark.parametrize("H,dtype", [(16, "f16"), (64, "f16"), (128, "bf16")])
def test_batch_of_32_requests_through_mla_decode(H, dtype):
    """The largest batch of the heads x batch grid: 32 requests of 8192 tokens through mla_decode with the
    planner's plan (16 heads: the paired kernel and the entries merge; 64 and 128 heads: the 128-row kernel and
    the merge kernel), sampled requests and heads against the oracle."""
    B, L = 32, 8192
    bs = 64 if dtype == "bf16" else 32
    case = gen.make_decode_case(37, [L] * B, num_heads=H, block_size=bs, dtype=dtype,
                                latent_std=0.5 if dtype == "bf16" else 1.0)
    dc = rt.upload(case)
    plan = nb.mla_plan([L] * B, H, 1, bs, nb.mla_device_query(), max_partitions=64, dtype=dtype)
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    part, lse = rt.alloc_partials(plan.num_chunks, 1, H)
    out = torch.empty((B, 1, H, 512), dtype=torch.float32, device="cuda")
    ws = rt.alloc_decode_workspace(B, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, H)
    rt.decode(dc, part, lse, ind, out, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas, chunks_dev=chunks,
              subs=plan.clusters_per_chunk, workspace=ws, tables_ready=True)
    reqs, heads = [0, 13, 31], [0, H // 2 + 3, H - 1]
    sub = dataclasses.replace(case, q_abs=case.q_abs[reqs], q_pe=case.q_pe[reqs],
                                  block_table=case.block_table[reqs], context_lens=case.context_lens[reqs])
    ref, _ = orc.unsplit(sub, heads=heads)
    assert_close(out.cpu().numpy()[reqs][:, :, heads], ref[:, :, heads], f"B=32 H={H} {dtype}")


def test_largest_row_count_causal_window_of_32_over_128_heads():
    """q_len 32 x 128 heads = 4096 rows (32 row groups of the 128-row kernel) with the causal window rule,
    short and ragged contexts, every row against the oracle."""
    case = gen.make_decode_case(38, [300, 97], num_heads=128, q_len=32, block_size=16, dtype="bf16", latent_std=0.5,
                                causal=True)
    dc = rt.upload(case)
    P = 2
    ind = rt.uniform_indptr(2, P)
    part, lse = rt.alloc_partials(2 * P, 32, 128)
    out = torch.empty((2, 32, 128, 512), dtype=torch.float32, device="cuda")
    nb.mla_reset_counters()
    rt.decode(dc, part, lse, ind, out, num_partitions=P, kernel=nb.MLA_KERNEL_TC, cluster=2)
    assert nb.mla_get_counters()[nb.CTR_CTAS] == 2 * P * 32 * 2  # 32 row groups of one CTA pair per chunk
    ref, _ = orc.unsplit(case)
    assert_close(out.cpu().numpy(), ref, "4096 rows")


def prefix_pair(case, dc, plan, chunks, ind, num_partitions=1, C=None, k=None, out_dtype="f32"):
    """(out, out_lse) of mla_decode twice in a row without and then with prefix_ready (tables_ready on both)."""
    B, q, H = case.num_requests, case.q_len, case.num_heads
    N = plan.num_chunks if plan is not None else B * num_partitions
    C = plan.cluster_ctas if plan is not None else C
    k = plan.clusters_per_chunk if plan is not None else k
    res = []
    for early in (False, True):
        part, lse = rt.alloc_partials(N, q, H)
        out = torch.full((B, q, H, 512), float("nan"), dtype=TDT[out_dtype], device="cuda")
        out_lse = torch.full((B, q, H), float("nan"), device="cuda")
        ws = rt.alloc_decode_workspace(B, N, k, C, q, H)
        desc = rt.make_desc(dc, chunks, nb.MLA_KERNEL_TC, C, None, k, ws, True, prefix_ready=early)
        for _ in range(2):  # the second call follows a kernel of the first: its early loads overlap that kernel
            rt.decode(dc, part, lse, ind, out, out_lse, num_partitions=num_partitions, desc=desc)
        res.append((out, out_lse))
    return res


@pytest.mark.parametrize("L", [32768, 131072])
def test_prefix_ready_gives_the_same_bits(L):
    """prefix_ready only moves the loads of the first tiles before the dependency wait: the planner's plan at a
    bench context gives the same bits with and without it, and matches the oracle."""
    case = gen.make_decode_case(2, [L], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    plan = nb.mla_plan([L], 16, 1, 32, nb.mla_device_query())
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    (o0, l0), (o1, l1) = prefix_pair(case, dc, plan, chunks, ind)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    heads = [0, 9]
    ref, _ = orc.unsplit(case, heads=heads)
    assert_close(o1.cpu().numpy()[:, :, heads], ref[:, :, heads], f"prefix_ready L={L}")


@pytest.mark.parametrize("q_len,C,k", [(1, 2, 1), (1, 4, 3), (1, 16, 1), (4, 2, 1)])
def test_prefix_ready_ragged_windows(q_len, C, k):
    """Ragged requests (contexts shorter than a tile, one tile, a last tile that holds the new token with prefix
    positions, several tiles) on the paired kernel with and without spread partitions, and a causal window of
    4 rows (64 rows: the 128-row kernel, which reads every cache row after the wait): the same bits with and
    without prefix_ready, and the oracle on every row."""
    lens = [2, 100, 129, 383, 384, 385, 2000]
    case = gen.make_decode_case(39, lens, num_heads=16, q_len=q_len, block_size=32, dtype="f16", causal=q_len > 1)
    dc = rt.upload(case)
    P, B = 2, len(lens)
    ind = rt.uniform_indptr(B, P)
    (o0, l0), (o1, l1) = prefix_pair(case, dc, None, None, ind, num_partitions=P, C=C, k=k)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    ref, _ = orc.unsplit(case)
    assert_close(o1.cpu().numpy(), ref, f"prefix_ready windows q={q_len} C={C} k={k}")


def test_prefix_ready_after_the_cache_write_of_the_window():
    """The layer call's order: mla_cache_append writes the new tokens' rows, then mla_decode with prefix_ready
    (the window's rows are read only after the append kernel has finished). Against the oracle on the
    appended cache, on every row."""
    lens = [5000, 130, 64]
    q_len = 1  # 16 rows: the paired kernel, whose early loads stop before the new token's tile
    case = gen.make_decode_case(40, lens, num_heads=16, q_len=q_len, block_size=32, dtype="f16")
    dc = rt.upload(case)
    rng = np.random.default_rng(41)
    ckv_new = gen.to_bits(rng.standard_normal((3, q_len, 512)), "f16")
    kpe_new = gen.to_bits(rng.standard_normal((3, q_len, 64)), "f16")
    cn, kn = rt.to_device_16(ckv_new, "f16", "cuda"), rt.to_device_16(kpe_new, "f16", "cuda")
    P, B = 2, 3
    ind = rt.uniform_indptr(B, P)
    part, lse = rt.alloc_partials(B * P, q_len, 16)
    out = torch.empty((B, q_len, 16, 512), dtype=torch.float32, device="cuda")
    ws = rt.alloc_decode_workspace(B, B * P, 1, 2, q_len, 16)
    desc = rt.make_desc(dc, None, nb.MLA_KERNEL_TC, 2, None, 1, ws, True, prefix_ready=True)
    rt.decode(dc, part, lse, ind, out, num_partitions=P, desc=desc)  # a kernel before the append
    nb.mla_cache_append(cn.data_ptr(), kn.data_ptr(), dc.block_table.data_ptr(), dc.context_lens.data_ptr(), B, q_len,
                        case.block_size, case.num_blocks, case.max_blocks, dc.ckv.data_ptr(), dc.kpe.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    rt.decode(dc, part, lse, ind, out, num_partitions=P, desc=desc)
    c2, k2 = orc.cache_append(case.ckv, case.kpe, case.block_table, case.context_lens, ckv_new, kpe_new, 32)
    ref, _ = orc.unsplit(dataclasses.replace(case, ckv=c2, kpe=k2))
    assert_close(out.cpu().numpy(), ref, "append then decode with prefix_ready")


@pytest.mark.parametrize("L", [32768, 131072])
def test_bf16_on_the_paired_kernel_planner_plan(L):
    """bf16 at 16 rows runs on the paired kernel (probabilities as two bf16 terms): the planner's plan through
    mla_decode's default and its single launch, against the oracle on sampled heads, the single launch the
    same bits as the two ABI calls."""
    case = gen.make_decode_case(41, [L], num_heads=16, block_size=32, dtype="bf16", latent_std=0.5)
    dc = rt.upload(case)
    plan = nb.mla_plan([L], 16, 1, 32, nb.mla_device_query(), dtype="bf16")
    assert plan.cluster_ctas >= 2
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    nb.mla_reset_counters()
    out, out_lse = default_decode(case, dc, plan, chunks, ind)
    assert nb.mla_get_counters()[nb.CTR_PARTIAL_TC] == 1
    heads = [0, 6, 15]
    ref, ref_lse = orc.unsplit(case, heads=heads)
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], f"bf16 pairs L={L}")
    assert np.abs(out_lse.cpu().numpy()[:, :, heads] - ref_lse[:, :, heads]).max() <= MAX_ABS
    fused, plain = both_paths(case, dc, chunks, ind, plan.num_chunks, nb.MLA_KERNEL_TC, plan.cluster_ctas,
                              plan.clusters_per_chunk, "bf16", tables_ready=True)
    assert_same_bits(fused, plain)
