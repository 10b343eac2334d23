"""GPU parity: the CUDA path through the C ABI against the f64 oracle.

Tolerance (the stated target for fp16/bf16 inputs with fp32 accumulation):
max-abs error <= 2e-3 and relative L2 error <= 1e-3 on fp32 results (partials
and the fp32 merge output), and max-abs 2e-3 on every finite log2 LSE. A
16-bit merge output must equal the fp32 merge output rounded once
(nearest-even); its distance to the exact result rounded once is then at most
one unit in the last place plus the fp32 result's own error.
"""
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

MAX_ABS = 2e-3
REL_L2 = 1e-3
KERNELS = {"tc": nb.MLA_KERNEL_TC, "simt": nb.MLA_KERNEL_SIMT}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    nbuild.build()
    nb.load()
    yield
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_OK, f"device error word {code:#x}"


def assert_close(got, ref, what, mask=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
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


def assert_rounded_once(out16, out32, ref, dtype):
    """A 16-bit output is the fp32 output rounded once to nearest-even, hence within one ulp (plus the fp32
    output's own error) of the exact result rounded once."""
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    assert torch.equal(out16, out32.to(tdt)), f"{dtype} output is not the fp32 output rounded once"
    o32 = out32.cpu().double().numpy()
    exact16 = torch.from_numpy(ref).to(tdt).double().numpy()
    got16 = out16.cpu().double().numpy()
    if dtype == "f16":
        ulp = np.abs(np.spacing(exact16.astype(np.float16)).astype(np.float64))
    else:  # bfloat16: 8 significant bits, spacing 2^(e - 7) at |x| in [2^e, 2^(e+1))
        mag = np.maximum(np.abs(exact16), np.abs(got16))
        ulp = np.exp2(np.floor(np.log2(np.where(mag > 0, mag, 1e-38))) - 7)
    dist = np.abs(got16 - exact16)
    assert np.all(dist <= ulp + np.abs(o32 - ref) + 1e-12), f"{dtype}: {np.max(dist - ulp):.3e} past one ulp"


def run_uniform(case, P, kernel, cluster, dc=None, subs=1, ws=None):
    dc = dc or rt.upload(case)
    B, q, H = case.num_requests, case.q_len, case.num_heads
    part, lse = rt.alloc_partials(B * P, q, H)
    part.fill_(float("nan"))
    if subs > 1 and ws is None:
        ws = rt.alloc_workspace(B * P, subs, cluster, q, H)
    rt.decode_partial(dc, part, lse, num_partitions=P, kernel=kernel, cluster=cluster, subs=subs, workspace=ws)
    ind = rt.uniform_indptr(B, P)
    out = rt.merge_states(part, lse, ind, B, q, H, "f32")
    return part, lse, out, ind, dc


def oracle_uniform_chunks(case, P):
    return orc.plan_chunks(case.context_lens, [P] * case.num_requests, case.block_size)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("P", [1, 2, 4])
def test_tiny_config_partials_and_merge(kernel, P):
    """B=1, H=16, ctx 4096, block 32, shuffled table, fp16, partitions {1,2,4}."""
    case = gen.make_decode_case(1, [4096], num_heads=16, block_size=32, dtype="f16")
    nb.mla_reset_counters()
    part, lse, out, ind, dc = run_uniform(case, P, KERNELS[kernel], cluster=4)
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_PARTIAL_TC if kernel == "tc" else nb.CTR_PARTIAL_SIMT] == 1 and ctr[nb.CTR_MERGE] == 1
    chunks, indptr = oracle_uniform_chunks(case, P)
    ref_part, ref_lse = orc.partials(case, chunks)
    assert_close(part.cpu().numpy(), ref_part, f"partials {kernel} P={P}")
    assert_lse_close(lse.cpu().numpy(), ref_lse, f"lse {kernel} P={P}")
    ref, _ = orc.unsplit(case)
    out32 = out.cpu().numpy().astype(np.float64)
    assert_close(out32, ref, f"merged {kernel} P={P}")
    # 16-bit output: the fp32 result rounded once
    assert_rounded_once(rt.merge_states(part, lse, ind, 1, 1, 16, "f16"), out, ref, "f16")


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_bitwise_reproducible_for_one_plan(kernel):
    case = gen.make_decode_case(2, [9000, 3001], num_heads=16, block_size=32, dtype="f16")
    outs = []
    dc = rt.upload(case)
    for _ in range(3):
        _, _, out, _, _ = run_uniform(case, 3, KERNELS[kernel], cluster=4, dc=dc)
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_paging_invariance_bitwise(kernel):
    case = gen.make_decode_case(3, [5000, 777], num_heads=16, block_size=16, dtype="f16")
    _, _, a, _, _ = run_uniform(case, 2, KERNELS[kernel], cluster=2)
    _, _, b, _, _ = run_uniform(gen.permute_pool(case, 11), 2, KERNELS[kernel], cluster=2)
    assert torch.equal(a, b)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("bs", [16, 32, 64])
def test_ragged_lengths_and_empty_requests(kernel, bs):
    lens = [0, 1, 31, 33, 64, 65, 100, 1000]
    case = gen.make_decode_case(4, lens, num_heads=16, block_size=bs, dtype="f16")
    part, lse, out, _, _ = run_uniform(case, 3, KERNELS[kernel], cluster=2)
    chunks, _ = oracle_uniform_chunks(case, 3)
    ref_part, ref_lse = orc.partials(case, chunks)
    assert_close(part.cpu().numpy(), ref_part, "partials")
    assert_lse_close(lse.cpu().numpy(), ref_lse, "lse")
    ref, _ = orc.unsplit(case)
    got = out.cpu().numpy()
    assert np.all(got[0] == 0)  # empty request merges to zeros
    assert_close(got[1:], ref[1:], "merged")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("H", [16, 64, 128])
def test_heads_and_dtypes(dtype, H):
    case = gen.make_decode_case(5, [2500, 700], num_heads=H, block_size=64 if dtype == "bf16" else 32,
                                dtype=dtype, latent_std=0.5 if dtype == "bf16" else 1.0)
    ref, _ = orc.unsplit(case)
    for kernel in ("tc", "simt"):
        part, lse, out, _, _ = run_uniform(case, 2, KERNELS[kernel], cluster=2)
        assert_close(out.cpu().numpy(), ref, f"{kernel} H={H} {dtype}")


@pytest.mark.parametrize("H,bs", [(16, 32), (128, 64)])
def test_bf16_output_is_the_fp32_result_rounded_once(H, bs):
    """bf16 inputs and a bf16 merge output (the many-head workload's output type): every element is the
    fp32 merge output rounded once to nearest-even, and within one bf16 ulp of the exact result."""
    case = gen.make_decode_case(15, [3000, 1234], num_heads=H, block_size=bs, dtype="bf16", latent_std=0.5)
    B = case.num_requests
    part, lse, out, ind, _ = run_uniform(case, 2, nb.MLA_KERNEL_TC, cluster=2)
    ref, ref_lse = orc.unsplit(case)
    assert_close(out.cpu().numpy(), ref, f"bf16 H={H} fp32 output")
    out_lse = torch.empty((B, 1, H), dtype=torch.float32, device="cuda")
    out16 = rt.merge_states(part, lse, ind, B, 1, H, "bf16", out_lse=out_lse)
    assert_rounded_once(out16, out, ref, "bf16")
    assert_lse_close(out_lse.cpu().numpy(), ref_lse, f"bf16 H={H} merged lse")


@pytest.mark.parametrize("H,q_len,dtype,bs", [(128, 1, "bf16", 64), (64, 2, "f16", 32)])
def test_many_rows_pair_kernel_bitwise_reproducible(H, q_len, dtype, bs):
    """The 128-row pair kernel (the many-head workload's kernel): the same plan gives the same bits in the
    partials, the LSE and the merged output on every call."""
    case = gen.make_decode_case(16, [7000, 2049, 130], num_heads=H, q_len=q_len, block_size=bs, dtype=dtype,
                                latent_std=0.5)
    dc = rt.upload(case)
    runs = []
    for _ in range(3):
        nb.mla_reset_counters()
        part, lse, out, _, _ = run_uniform(case, 3, nb.MLA_KERNEL_TC, cluster=2, dc=dc)
        assert nb.mla_get_counters()[nb.CTR_CTAS] == 3 * 3 * 2  # one CTA pair per chunk: the 128-row kernel
        runs.append((part.clone(), lse.clone(), out.clone()))
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)


def test_out_lse_and_hierarchical_merge_is_associative():
    case = gen.make_decode_case(6, [6000], num_heads=16, block_size=32, dtype="f16")
    part, lse, out, _, _ = run_uniform(case, 4, nb.MLA_KERNEL_TC, cluster=2)
    # merge (0,1) and (2,3) separately, then merge the two results by their LSE
    ind2 = torch.tensor([0, 2, 4], dtype=torch.int32, device="cuda")
    lse2 = torch.empty((2, 1, 16), dtype=torch.float32, device="cuda")
    half = rt.merge_states(part, lse, ind2, 2, 1, 16, "f32", out_lse=lse2)
    ind1 = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    top = rt.merge_states(half.contiguous(), lse2, ind1, 1, 1, 16, "f32")
    assert_close(top.cpu().numpy(), out.cpu().numpy(), "hierarchical vs flat")
    lse1 = torch.empty((1, 1, 16), dtype=torch.float32, device="cuda")
    rt.merge_states(part, lse, rt.uniform_indptr(1, 4), 1, 1, 16, "f32", out_lse=lse1)
    _, ref_lse = orc.unsplit(case)
    assert_lse_close(lse1.cpu().numpy(), ref_lse, "merged lse")


def test_natural_log_lse_fails_parity_on_the_gpu_merge():
    """Negative control: natural-log LSE fed to the base-2 merge gives a wrong answer."""
    case = gen.make_decode_case(7, [4096], num_heads=16, block_size=32, dtype="f16")
    part, lse, out, ind, _ = run_uniform(case, 4, nb.MLA_KERNEL_TC, cluster=2)
    ref, _ = orc.unsplit(case)
    assert_close(out.cpu().numpy(), ref, "log2 merge")
    bad = rt.merge_states(part, lse * math.log(2.0), ind, 1, 1, 16, "f32").cpu().numpy()
    err = np.abs(bad - ref).max()
    rel = np.linalg.norm(bad - ref) / np.linalg.norm(ref)
    assert err > MAX_ABS or rel > REL_L2, "natural-log LSE should not pass parity"


@pytest.mark.parametrize("C", [2, 4, 8, 16])
@pytest.mark.parametrize("bs", [16, 32, 64])
def test_paired_kernel_ragged(C, bs):
    """16 fp16 rows, clusters of 2..16: the CTAs of a pair share each 128-token tile. The lengths end
    chunks at every kind of place in a tile's 32-token quarters (empty, partial, full)."""
    lens = [0, 1, 17, 31, 32, 33, 64, 95, 96, 97, 127, 128, 129, 1000, 4133]
    case = gen.make_decode_case(12, lens, num_heads=16, block_size=bs, dtype="f16")
    P = 3
    nb.mla_reset_counters()
    part, lse, out, _, _ = run_uniform(case, P, nb.MLA_KERNEL_TC, cluster=C)
    assert nb.mla_get_counters()[nb.CTR_CTAS] == len(lens) * P * C
    chunks, _ = oracle_uniform_chunks(case, P)
    ref_part, ref_lse = orc.partials(case, chunks)
    assert_close(part.cpu().numpy(), ref_part, f"partials C={C} bs={bs}")
    assert_lse_close(lse.cpu().numpy(), ref_lse, f"lse C={C} bs={bs}")
    ref, _ = orc.unsplit(case)
    assert_close(out.cpu().numpy(), ref, f"merged C={C} bs={bs}")


def plan_and_run(case, max_partitions=0, kernel=nb.MLA_KERNEL_TC, dc=None, ws=None, tables_ready=False):
    """The planner's plan as the bench runs it: its cluster size and clusters per partition."""
    dev = nb.mla_device_query()
    plan = nb.mla_plan(case.context_lens.tolist(), case.num_heads, case.q_len, case.block_size, dev,
                       max_partitions=max_partitions, dtype=case.dtype, merge_path=nb.MLA_MERGE_PARTIALS)
    dc = dc or rt.upload(case)
    chunks_dev = rt.chunks_to_device(plan.chunks)
    part, lse = rt.alloc_partials(plan.num_chunks, case.q_len, case.num_heads)
    k = plan.clusters_per_chunk if kernel != nb.MLA_KERNEL_SIMT else 1
    if k > 1 and ws is None:
        ws = rt.alloc_workspace(plan.num_chunks, k, plan.cluster_ctas, case.q_len, case.num_heads)
    rt.decode_partial(dc, part, lse, chunks_dev=chunks_dev, kernel=kernel, cluster=plan.cluster_ctas, subs=k,
                      workspace=ws, tables_ready=tables_ready)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    out = rt.merge_states(part, lse, ind, case.num_requests, case.q_len, case.num_heads, "f32")
    return plan, part, lse, out


@pytest.mark.parametrize("L", [32768, 49152, 65536, 81920, 98304, 131072])
def test_long_context_planned_full_size_sampled_heads(L):
    """Every context of the bench's sweep, in the bench's launch configuration (the planner's plan, tables
    read before the dependency wait), against the oracle on sampled heads."""
    case = gen.make_decode_case(2, [L], num_heads=16, block_size=32, dtype="f16")
    nb.mla_reset_counters()
    plan, part, lse, out = plan_and_run(case, tables_ready=True)
    assert 2 <= plan.num_chunks <= 8, plan.parts()
    if L == 131072:
        assert plan.clusters_per_chunk > 1  # the partitions are spread over clusters to fill the GPU
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_PARTIAL_TC] == 1
    assert ctr[nb.CTR_CTAS] == plan.num_chunks * plan.cluster_ctas * plan.clusters_per_chunk
    heads = [0, 7, 15]
    ref, _ = orc.unsplit(case, heads=heads)
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], f"L={L}")


@pytest.mark.parametrize("L,P,C,k,bs", [(4096, 2, 2, 4, 32), (4096, 1, 4, 2, 32), (20017, 3, 2, 5, 16),
                                         (20017, 2, 4, 3, 64), (9000, 2, 16, 2, 32)])
def test_spread_partitions_partials_match_oracle(L, P, C, k, bs):
    """Each partition over k clusters (every CTA pair's part merged by the last CTA to finish, up to 16 parts:
    more than one round of the merge) gives the partition's partial."""
    case = gen.make_decode_case(5, [L], num_heads=16, block_size=bs, dtype="f16")
    nb.mla_reset_counters()
    part, lse, out, ind, dc = run_uniform(case, P, nb.MLA_KERNEL_TC, cluster=C, subs=k)
    assert nb.mla_get_counters()[nb.CTR_CTAS] == P * C * k
    chunks, _ = oracle_uniform_chunks(case, P)
    ref_part, ref_lse = orc.partials(case, chunks)
    assert_close(part.cpu().numpy(), ref_part, f"partials L={L} P={P} C={C} k={k}")
    assert_lse_close(lse.cpu().numpy(), ref_lse, f"lse L={L} P={P} C={C} k={k}")
    ref, _ = orc.unsplit(case)
    assert_close(out.cpu().numpy(), ref, f"merged L={L} P={P} C={C} k={k}")


@pytest.mark.parametrize("L", [32768, 131072])
def test_tables_read_before_the_dependency_wait_give_the_same_bits(L):
    """tables_ready only moves the reads of the chunk table, the lengths and the block table before the
    wait for the preceding kernel: the same plan gives the same bits either way, also right behind
    another decode call (a merge, then this call's kernel as its programmatic dependent)."""
    case = gen.make_decode_case(7, [L], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    ref = plan_and_run(case, dc=dc)[1:]
    for _ in range(2):  # the second time behind the first call's merge in the stream
        got = plan_and_run(case, dc=dc, tables_ready=True)[1:]
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_OK, code


def test_spread_partitions_bitwise_reproducible_and_workspace_reused():
    """Same plan, same workspace, several calls: identical bits (the merge order does not depend on which
    pair finishes last, and every call leaves its tickets at zero)."""
    case = gen.make_decode_case(6, [131072], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    dev = nb.mla_device_query()
    plan = nb.mla_plan([131072], 16, 1, 32, dev, merge_path=nb.MLA_MERGE_PARTIALS)
    assert plan.clusters_per_chunk > 1
    ws = rt.alloc_workspace(plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, 16)
    outs = []
    for _ in range(3):
        _, part, lse, out = plan_and_run(case, dc=dc, ws=ws)
        outs.append((part.clone(), lse.clone(), out.clone()))
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a, b)
    tickets = ws[: 8 * plan.num_chunks].view(torch.int32)
    assert int(tickets.abs().sum()) == 0


@pytest.mark.parametrize("H,q_len,dtype,bs,lens,causal", [
    (128, 1, "bf16", 64, [5000, 777], False),
    (128, 1, "f16", 32, [4096], False),
    (128, 1, "bf16", 16, [2049, 130], False),
    (64, 2, "bf16", 32, [3000, 1500], True),
])
def test_many_rows_pair_kernel_partials(H, q_len, dtype, bs, lens, causal):
    """128 rows per CTA pair (rows on M, P in tensor memory): per-chunk partials against the oracle."""
    case = gen.make_decode_case(9, lens, num_heads=H, q_len=q_len, block_size=bs, dtype=dtype, latent_std=0.5,
                                causal=causal)
    P = 3
    nb.mla_reset_counters()
    part, lse, out, ind, dc = run_uniform(case, P, nb.MLA_KERNEL_TC, cluster=2)
    assert nb.mla_get_counters()[nb.CTR_CTAS] == len(lens) * P * 2  # one pair per chunk, all rows
    chunks, _ = oracle_uniform_chunks(case, P)
    ref_part, ref_lse = orc.partials(case, chunks)
    assert_close(part.cpu().numpy(), ref_part, f"partials H={H} q={q_len} {dtype} bs={bs}")
    assert_lse_close(lse.cpu().numpy(), ref_lse, f"lse H={H} q={q_len} {dtype} bs={bs}")
    ref, _ = orc.unsplit(case)
    assert_close(out.cpu().numpy(), ref, f"merged H={H} q={q_len} {dtype} bs={bs}")


@pytest.mark.parametrize("tables_ready", [False, True])
def test_mixed_batch_request_major(tables_ready):
    case = gen.make_decode_case(3, [32768, 20000], num_heads=16, block_size=32, dtype="f16")
    plan, part, lse, out = plan_and_run(case, max_partitions=4, tables_ready=tables_ready)
    assert all(2 <= p <= 4 for p in plan.parts()), plan.parts()
    heads = [0, 5, 10, 15]
    ref, _ = orc.unsplit(case, heads=heads)
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], "mixed batch")


def test_many_heads_bf16_planned_sampled():
    lens = gen.uniform_lengths(4, 8, 4096, 65536)
    case = gen.make_decode_case(4, lens, num_heads=128, block_size=64, dtype="bf16", latent_std=0.5)
    plan, part, lse, out = plan_and_run(case, max_partitions=64)
    heads = [0, 47, 48, 95, 96, 127]
    ref, _ = orc.unsplit(case, heads=heads)
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], "H=128 bf16")


def run_segments(seg, q_len, cluster=2):
    B, H = seg.base.num_requests, seg.base.num_heads
    nseg = len(seg.segments)
    part, lse = rt.alloc_partials(B * nseg, q_len, H)
    dc0 = rt.upload(seg.segments[0])
    for k, s in enumerate(seg.segments):
        dc = rt.upload(s, ckv=dc0.ckv, kpe=dc0.kpe)
        # one partition per (request, segment); slot = b * nseg + k (request-major)
        chunks = [(b, 0, int(s.context_lens[b]), b * nseg + k) for b in range(B)]
        rt.decode_partial(dc, part, lse, chunks_dev=rt.chunks_to_device(chunks), kernel=nb.MLA_KERNEL_TC,
                          cluster=cluster)
    ind = rt.uniform_indptr(B, nseg)
    out = rt.merge_states(part, lse, ind, B, q_len, H, "f32")
    return out, part, lse, ind, dc0


@pytest.mark.parametrize("q_len", [4, 9, 16, 32])
def test_verify_windows_over_segments(q_len):
    seg = gen.make_segmented_case(5, B=4, q_len=q_len, segment_tokens=(4096, 2048, 1024), num_heads=16,
                                  block_size=32)
    ref, _ = orc.unsplit(gen.concat_segments(seg))
    out, part, lse, ind, dc0 = run_segments(seg, q_len)
    assert_close(out.cpu().numpy(), ref, f"q_len={q_len}")
    # positive control: the tail without its causal mask gives a different answer
    B, nseg = 4, len(seg.segments)
    tail = seg.segments[-1]
    tail.causal = False
    dc = rt.upload(tail, ckv=dc0.ckv, kpe=dc0.kpe)
    chunks = [(b, 0, int(tail.context_lens[b]), b * nseg + nseg - 1) for b in range(B)]
    rt.decode_partial(dc, part, lse, chunks_dev=rt.chunks_to_device(chunks), kernel=nb.MLA_KERNEL_TC, cluster=1)
    bad = rt.merge_states(part, lse, ind, B, q_len, 16, "f32").cpu().numpy()
    assert np.abs(bad - ref).max() > 3 * MAX_ABS


def run_planned_segments(seg):
    """A verify window as the bench runs it: every segment planned by mla_plan (its own partitions, cluster
    size and row groups), one partial launch per segment into request-major slots, one merge."""
    base = seg.base
    B, q_len, H = base.num_requests, base.q_len, base.num_heads
    sp = rt.plan_segments(seg, nb.mla_device_query())
    part, lse = rt.alloc_partials(sp.num_slots, q_len, H)
    part.fill_(float("nan"))
    dc0 = rt.upload(base)
    for s, table, plan in zip(seg.segments, sp.chunk_tables, sp.plans):
        dc = rt.upload(s, ckv=dc0.ckv, kpe=dc0.kpe)
        ws = rt.alloc_workspace(plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, q_len, H)
        rt.decode_partial(dc, part, lse, chunks_dev=table, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas,
                          subs=plan.clusters_per_chunk, workspace=ws)
    out_lse = torch.empty((B, q_len, H), dtype=torch.float32, device="cuda")
    out = rt.merge_states(part, lse, sp.o_indptr, B, q_len, H, "f32", out_lse=out_lse)
    return out, out_lse, sp


@pytest.mark.parametrize("q_len", [4, 9, 16, 32])
def test_verify_window_full_prefix_sampled_heads(q_len):
    """The verify-window workload at full size, in the bench's launch configuration: prefix 81920 tokens in 3
    segments plus the causal window tail, B=4, every window length (a window of 16 or 32 rows over 16 heads
    runs on the 128-row pair kernel in 2 or 4 row groups), on sampled heads whose rows fall in different TMEM
    lane quadrants."""
    seg = gen.make_segmented_case(5, B=4, q_len=q_len, num_heads=16, block_size=32)
    heads = [0, 9] if q_len == 32 else [0, 7, 9, 14]
    ref, ref_lse = orc.unsplit(gen.concat_segments(seg), heads=heads)
    nb.mla_reset_counters()
    out, out_lse, sp = run_planned_segments(seg)
    assert nb.mla_get_counters()[nb.CTR_PARTIAL_TC] == 4
    assert all(p.num_chunks >= 4 for p in sp.plans[:3])  # every prefix segment split over the requests
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], f"full prefix q_len={q_len}")
    assert_lse_close(out_lse.cpu().numpy()[:, :, heads], ref_lse[:, :, heads], f"full prefix lse q_len={q_len}")


def test_out_of_range_page_reads_zeros_and_is_flagged():
    case = gen.make_decode_case(8, [300], num_heads=16, block_size=32, dtype="f16")
    case.block_table[0, 2] = case.num_blocks + 5  # a bad page id inside the context
    nb.mla_check_device_errors(None)
    part, lse, out, _, _ = run_uniform(case, 1, nb.MLA_KERNEL_TC, cluster=1)
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_ERR_DEVICE_CHECK and code & 2
    assert np.all(np.isfinite(out.cpu().numpy()))


def test_selfcheck_closed_form_case():
    """The library's built-in check (needle heads and a uniform head, fp16 and bf16, default and CUDA-core
    kernels) passes on this device; its closed form is confirmed by the oracle in the CPU tests."""
    nb.mla_check_device_errors(None)
    nb.mla_reset_counters()
    st, err = nb.mla_selfcheck()
    assert st == nb.MLA_OK, (st, err)
    assert err <= 2e-3
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_PARTIAL_TC] == 2 and ctr[nb.CTR_PARTIAL_SIMT] == 2 and ctr[nb.CTR_MERGE] == 4
