"""C-ABI library on the CPU: it loads, exports what the header declares, plans
correctly, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

from mla_split_kv_gb300 import binding as nb
from mla_split_kv_gb300 import build as nbuild
from mla_split_kv_gb300 import inputs as gen
from oracle import mla_oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nbuild.build()
    return nb.load()


def header_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?!typedef)[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_core_calls():
    names = header_functions()
    for must in ("mla_plan", "mla_decode_partial", "mla_merge_states", "mla_device_query",
                 "mla_check_device_errors", "mla_get_counters", "mla_selfcheck"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


# --- planner ------------------------------------------------------------------------

def fake_gb300():
    """Occupancy figures of the tensor-core kernel as measured on a GB300."""
    dev = nb.mla_device_info_t()
    dev.num_sms = 152
    for k, v in enumerate([152, 76, 36, 15, 7]):
        dev.max_clusters[k] = v
    return dev


def check_plan_tiles(plan, lens, bs):
    assert plan.o_indptr[0] == 0 and plan.o_indptr[-1] == plan.num_chunks
    for b, L in enumerate(lens):
        lo, hi = plan.o_indptr[b], plan.o_indptr[b + 1]
        ch = plan.chunks[lo:hi]
        assert all(c[0] == b for c in ch)
        assert ch[0][1] == 0 and ch[-1][2] == L
        for c0, c1 in zip(ch, ch[1:]):
            assert c0[2] == c1[1]
        for (bb, t0, t1, slot) in ch:
            assert t0 % bs == 0 and t0 <= t1
        # the chunk table is exactly the oracle's chunk rule for that P
        assert [(t0, t1) for (_, t0, t1, _) in ch] == orc.chunk_bounds(L, hi - lo, bs)
    assert [c[3] for c in plan.chunks] == list(range(plan.num_chunks))


@pytest.mark.parametrize("merge_path", [nb.MLA_MERGE_ENTRIES, nb.MLA_MERGE_PARTIALS])
@pytest.mark.parametrize("L", [32768, 49152, 65536, 81920, 98304, 131072])
def test_plan_long_context_single_request(lib, L, merge_path):
    plan = nb.mla_plan([L], 16, 1, 32, fake_gb300(), merge_path=merge_path)
    assert 2 <= plan.num_chunks <= 8
    busy = plan.num_chunks * plan.cluster_ctas * plan.clusters_per_chunk
    assert 100 <= busy <= 152  # most of the 152 SMs busy, with at most 8 partitions
    if merge_path == nb.MLA_MERGE_PARTIALS:
        if L >= 131072:  # long enough that spreading partitions over clusters pays for its merge tail
            assert plan.clusters_per_chunk > 1 and busy >= 140
        if L <= 65536:  # too short for that: one cluster of 16 per partition
            assert plan.clusters_per_chunk == 1 and plan.cluster_ctas == 16
    else:
        # with the pairs' parts merged as entries a spread costs nothing more: CTA pairs over the whole GPU,
        # and no plan of up to 8 partitions on the 76 co-resident pairs gives its busiest pair fewer tiles
        assert plan.cluster_ctas == 2 and plan.clusters_per_chunk > 1 and busy >= 140

        def busiest(P, k):  # 128-token tiles of the busiest pair: a chunk's tiles split evenly over its k pairs
            longest = max(t1 - t0 for t0, t1 in orc.chunk_bounds(L, P, 32))
            return -(-(-(-longest // 128)) // k)

        best = min(busiest(P, k) for P in range(2, 9) for k in range(1, 17) if P * k <= 76)
        assert busiest(plan.num_chunks, plan.clusters_per_chunk) == best
    check_plan_tiles(plan, [L], 32)
    # every CTA pair of every cluster keeps at least one 128-token tile of its partition
    k, C = plan.clusters_per_chunk, plan.cluster_ctas
    assert 1 <= k <= 16
    for (_, t0, t1, _) in plan.chunks:
        assert t1 - t0 >= k * (C // 2) * 128


def test_plan_rejects_an_unknown_merge_path(lib):
    dev = fake_gb300()
    lens = (ctypes.c_int32 * 1)(65536)
    plan = nb.mla_plan_t()
    plan.merge_path = 2
    assert lib.mla_plan(lens, 1, 16, 1, 32, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_INVALID_ARG


def test_plan_spreads_partitions_only_for_the_paired_kernel(lib):
    # the paired kernel runs for 16 rows per CTA (fp16 or bf16): 128 heads keep one cluster per partition
    p16 = nb.mla_plan([131072], 16, 1, 32, fake_gb300())
    assert p16.clusters_per_chunk > 1 and p16.cluster_ctas >= 2
    pb = nb.mla_plan([131072], 16, 1, 32, fake_gb300(), dtype="bf16")
    assert (pb.chunks, pb.cluster_ctas, pb.clusters_per_chunk) == (p16.chunks, p16.cluster_ctas, p16.clusters_per_chunk)
    p128 = nb.mla_plan([131072], 128, 1, 32, fake_gb300())
    assert p128.clusters_per_chunk == 1
    # a short request in the batch caps k so that, when a partition is spread, every pair still gets a tile
    pmix = nb.mla_plan([131072, 700], 16, 1, 32, fake_gb300())
    k, C = pmix.clusters_per_chunk, pmix.cluster_ctas
    if k > 1:
        for (_, t0, t1, _) in pmix.chunks:
            assert t1 - t0 >= k * (C // 2) * 128


@pytest.mark.parametrize("lens", [[131072], [700], [4096] * 8, [32768, 100, 9000, 0], [20000] * 64])
def test_plan_for_e4m3_caches_keeps_pairs(lib, lens):
    # E4M3 caches run on CTA pairs only: every plan uses clusters of 2 or more, and otherwise splits the
    # contexts as for fp16 caches whenever the fp16 plan already uses pairs
    pe = nb.mla_plan(lens, 16, 1, 32, fake_gb300(), dtype="e4m3")
    pf = nb.mla_plan(lens, 16, 1, 32, fake_gb300(), dtype="f16")
    assert pe.cluster_ctas >= 2
    check_plan_tiles(pe, lens, 32)
    if pf.cluster_ctas >= 2:
        assert (pe.chunks, pe.o_indptr, pe.cluster_ctas, pe.clusters_per_chunk) == \
            (pf.chunks, pf.o_indptr, pf.cluster_ctas, pf.clusters_per_chunk)


@pytest.mark.parametrize("lens", [[8192] * 8, [8192] * 32, [1000] * 8, [40000, 3000, 0, 129]])
def test_batch_plans_of_sixteen_rows_use_cta_pairs(lib, lens):
    # a batch at H=16 runs on the paired kernel (clusters of 2 or more) whenever the device has pairs
    plan = nb.mla_plan(lens, 16, 1, 32, fake_gb300())
    assert plan.cluster_ctas >= 2
    check_plan_tiles(plan, lens, 32)
    assert plan.num_chunks * plan.clusters_per_chunk <= 76  # one wave of the device's 76 pairs
    # without pairs on the device: one CTA per partition
    plan1 = nb.mla_plan(lens, 16, 1, 32, fake_device(152, [152, 0, 0, 0, 0]))
    assert plan1.cluster_ctas == 1
    # bf16 runs on the same pairs
    pb = nb.mla_plan(lens, 16, 1, 32, fake_gb300(), dtype="bf16")
    assert pb.cluster_ctas >= 2


def test_workspace_bytes(lib):
    assert nb.mla_workspace_bytes(8, 1, 4, 1, 16) == 0
    assert nb.mla_workspace_bytes(8, 4, 1, 1, 16) == 0
    # two tickets per chunk, one entry per CTA pair: O [rows][512] + two [rows][2] blocks
    n, k, C, rows = 8, 9, 4, 16
    e = n * k * (C // 2)
    assert nb.mla_workspace_bytes(n, k, C, 1, 16) == 256 + e * rows * 512 * 4 + e * 2 * rows * 2 * 4
    e = 100 * 2 * 8
    assert nb.mla_workspace_bytes(100, 2, 16, 2, 16) == 1024 + e * 32 * 512 * 4 + e * 2 * 32 * 2 * 4


def test_plan_mixed_batch_two_to_four(lib):
    lens = [32768, 20000]
    plan = nb.mla_plan(lens, 16, 1, 32, fake_gb300(), max_partitions=4)
    assert all(2 <= p <= 4 for p in plan.parts())
    check_plan_tiles(plan, lens, 32)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_plan_many_heads_batch(lib, dtype):
    lens = gen.uniform_lengths(4, 8, 4096, 65536)
    plan = nb.mla_plan(lens, 128, 1, 64, fake_gb300(), max_partitions=64, dtype=dtype)
    check_plan_tiles(plan, lens, 64)
    parts = plan.parts()
    assert all(1 <= p <= 64 for p in parts)
    order = np.argsort(lens)
    assert parts[order[-1]] >= parts[order[0]]


def test_plan_short_and_empty_requests_are_not_split(lib):
    lens = [0, 1, 100, 4095, 40000]
    plan = nb.mla_plan(lens, 16, 1, 16, fake_gb300())
    parts = plan.parts()
    assert parts[:4] == [1, 1, 1, 1] and parts[4] >= 2
    check_plan_tiles(plan, lens, 16)


def test_planner_host_timing_helper(lib):
    import bench
    us = bench.planner_host_us(nb, [131072], fake_gb300(), batches=2, reps=20)
    assert 0 < us < 1e4


def fake_device(num_sms, max_clusters):
    dev = nb.mla_device_info_t()
    dev.num_sms = num_sms
    for k, v in enumerate(max_clusters):
        dev.max_clusters[k] = v
    return dev


@pytest.mark.parametrize("sms,clusters", [
    (132, [132, 66, 33, 16, 8]),   # fewer SMs
    (148, [148, 74, 36, 18, 0]),   # clusters of 16 unavailable
    (20, [20, 10, 5, 2, 1]),       # a small part
    (152, [152, 76, 0, 0, 0]),     # pairs only
])
@pytest.mark.parametrize("L", [4096, 32768, 131072])
def test_plan_follows_the_device(lib, sms, clusters, L):
    dev = fake_device(sms, clusters)
    plan = nb.mla_plan([L], 16, 1, 32, dev)
    C, k, N = plan.cluster_ctas, plan.clusters_per_chunk, plan.num_chunks
    log2c = C.bit_length() - 1
    assert C in (1, 2, 4, 8, 16) and clusters[log2c] > 0  # never a size the device cannot launch
    assert 2 <= N <= 8  # the pages' 2..8 gate for a split request
    assert N * k <= clusters[log2c]  # every cluster of the launch is co-resident (one wave)
    assert N * k * C <= sms
    check_plan_tiles(plan, [L], 32)
    for (_, t0, t1, _) in plan.chunks:  # every CTA pair keeps at least one 128-token tile
        assert t1 - t0 >= k * max(1, C // 2) * 128


@pytest.mark.parametrize("sms,clusters", [
    (132, [132, 66, 33, 16, 8]),
    (148, [148, 74, 36, 18, 0]),
    (20, [20, 10, 5, 2, 1]),
])
@pytest.mark.parametrize("H,dtype,bs,maxp", [(128, "bf16", 64, 64), (16, "f16", 32, 4), (16, "bf16", 16, 8)])
def test_batch_plans_follow_the_device(lib, sms, clusters, H, dtype, bs, maxp):
    dev = fake_device(sms, clusters)
    lens = gen.uniform_lengths(4, 8, 4096, 65536) + [0, 1000]
    plan = nb.mla_plan(lens, H, 1, bs, dev, max_partitions=maxp, dtype=dtype)
    C = plan.cluster_ctas
    assert C in (1, 2, 4, 8, 16) and clusters[C.bit_length() - 1] > 0
    if H == 128:
        assert C == 2  # the 128-row kernel runs on one CTA pair
    parts = plan.parts()
    assert all(1 <= p <= maxp for p in parts) and parts[-2:] == [1, 1]
    check_plan_tiles(plan, lens, bs)


def test_plan_is_deterministic(lib):
    lens = gen.uniform_lengths(9, 5, 1000, 90000)
    a = nb.mla_plan(lens, 16, 4, 32, fake_gb300())
    b = nb.mla_plan(lens, 16, 4, 32, fake_gb300())
    assert a.chunks == b.chunks and a.o_indptr == b.o_indptr and a.cluster_ctas == b.cluster_ctas


def test_plan_capacity_and_argument_errors(lib):
    dev = fake_gb300()
    lens = (ctypes.c_int32 * 1)(65536)
    plan = nb.mla_plan_t()
    plan.capacity = 1
    chunks = (nb.mla_chunk_t * 1)()
    ind = (ctypes.c_int32 * 2)()
    plan.chunks = ctypes.cast(chunks, ctypes.POINTER(nb.mla_chunk_t))
    plan.o_indptr = ctypes.cast(ind, ctypes.POINTER(ctypes.c_int32))
    assert lib.mla_plan(lens, 1, 16, 1, 32, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_CAPACITY
    assert plan.num_chunks > 1
    assert lib.mla_plan(lens, 1, 24, 1, 32, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_UNSUPPORTED
    assert lib.mla_plan(lens, 1, 16, 33, 32, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_UNSUPPORTED
    assert lib.mla_plan(lens, 1, 16, 1, 48, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_UNSUPPORTED
    assert lib.mla_plan(lens, 0, 16, 1, 32, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_INVALID_ARG
    plan.dtype = 2
    assert lib.mla_plan(lens, 1, 16, 1, 32, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_UNSUPPORTED
    plan.dtype = nb.MLA_E4M3  # E4M3 caches run on CTA pairs: 128-row groups on clusters of 2
    assert lib.mla_plan(lens, 1, 64, 1, 32, ctypes.byref(dev), ctypes.byref(plan)) in (nb.MLA_OK, nb.MLA_ERR_CAPACITY)
    assert plan.cluster_ctas == 2
    plan.dtype = 0
    neg = (ctypes.c_int32 * 1)(-5)
    assert lib.mla_plan(neg, 1, 16, 1, 32, ctypes.byref(dev), ctypes.byref(plan)) == nb.MLA_ERR_INVALID_ARG


# --- argument checks before any launch ------------------------------------------------

FAKE = 0x10000  # 64 KiB-aligned fake device address: never dereferenced on a rejected call


def desc(**kw):
    d = nb.mla_decode_desc_t()
    d.num_requests, d.num_heads, d.q_len, d.block_size = 1, 16, 1, 32
    d.num_blocks, d.max_blocks_per_req, d.dtype, d.causal = 8, 8, nb.MLA_F16, 0
    d.chunks, d.num_chunks, d.cluster_ctas, d.kernel, d.stream = None, 0, 1, nb.MLA_KERNEL_TC, None
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def call_partial(lib, d, P=2, ptrs=None):
    p = [FAKE] * 8 if ptrs is None else ptrs
    return lib.mla_decode_partial(p[0], p[1], p[2], p[3], p[4], p[5], ctypes.c_float(0.07), P, p[6], p[7],
                                  ctypes.byref(d))


@pytest.mark.parametrize("kw,P,want", [
    (dict(num_heads=32), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(q_len=0), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(q_len=33), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(block_size=128), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(dtype=2), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(num_requests=0), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=3), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(kernel=7), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(causal=2), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(tables_ready=2), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(decode_merge=3), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(decode_merge=-1), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(prefix_ready=2, tables_ready=1), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(prefix_ready=1), 2, nb.MLA_ERR_INVALID_ARG),  # early cache reads need the tables early too
    (dict(), 0, nb.MLA_ERR_INVALID_ARG),
    (dict(num_requests=40000), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(dtype=4, cluster_ctas=2), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(score_exchange=4), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(score_exchange=-1), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(score_exchange=2, dtype=nb.MLA_E4M3, cluster_ctas=2, cache_scale=1.0), 2, nb.MLA_ERR_UNSUPPORTED),
    # E4M3 caches: the paired 16-row kernel only, and a cache scale in [2^-24, 2^24]
    (dict(dtype=nb.MLA_E4M3, cache_scale=1.0), 2, nb.MLA_ERR_UNSUPPORTED),  # clusters of 1
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=2, kernel=nb.MLA_KERNEL_SIMT, cache_scale=1.0), 2,
     nb.MLA_ERR_UNSUPPORTED),
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=4, num_heads=64, cache_scale=1.0), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=8, q_len=2, cache_scale=1.0), 2, nb.MLA_ERR_UNSUPPORTED),
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=2), 2, nb.MLA_ERR_INVALID_ARG),  # cache_scale left 0
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=2, cache_scale=-0.25), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=2, cache_scale=2.0 ** -25), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=2, cache_scale=2.0 ** 25), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=2, cache_scale=float("inf")), 2, nb.MLA_ERR_INVALID_ARG),
    (dict(dtype=nb.MLA_E4M3, cluster_ctas=2, cache_scale=float("nan")), 2, nb.MLA_ERR_INVALID_ARG),
])
def test_decode_partial_rejects_before_launch(lib, kw, P, want):
    nb.mla_reset_counters()
    assert call_partial(lib, desc(**kw), P) == want
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_PARTIAL_TC] == 0 and ctr[nb.CTR_PARTIAL_SIMT] == 0 and ctr[nb.CTR_REJECTED] == 1


BIG = 1 << 40


@pytest.mark.parametrize("kw,want", [
    (dict(clusters_per_chunk=17, cluster_ctas=2, workspace=FAKE, workspace_bytes=BIG), nb.MLA_ERR_INVALID_ARG),
    (dict(clusters_per_chunk=-1), nb.MLA_ERR_INVALID_ARG),
    (dict(clusters_per_chunk=4, cluster_ctas=2), nb.MLA_ERR_INVALID_ARG),  # no workspace
    (dict(clusters_per_chunk=4, cluster_ctas=2, workspace=FAKE, workspace_bytes=1024), nb.MLA_ERR_INVALID_ARG),
    (dict(clusters_per_chunk=4, cluster_ctas=2, workspace=FAKE + 8, workspace_bytes=BIG), nb.MLA_ERR_INVALID_ARG),
    (dict(clusters_per_chunk=4, cluster_ctas=0, workspace=FAKE, workspace_bytes=BIG), nb.MLA_ERR_INVALID_ARG),
    (dict(clusters_per_chunk=4, cluster_ctas=1, workspace=FAKE, workspace_bytes=BIG), nb.MLA_ERR_UNSUPPORTED),
    (dict(clusters_per_chunk=4, cluster_ctas=2, num_heads=64, workspace=FAKE, workspace_bytes=BIG),
     nb.MLA_ERR_UNSUPPORTED),
    (dict(clusters_per_chunk=4, cluster_ctas=2, kernel=nb.MLA_KERNEL_SIMT, workspace=FAKE, workspace_bytes=BIG),
     nb.MLA_ERR_UNSUPPORTED),
])
def test_decode_partial_rejects_bad_spread_partitions(lib, kw, want):
    nb.mla_reset_counters()
    assert call_partial(lib, desc(**kw), 2) == want
    assert nb.mla_get_counters()[nb.CTR_REJECTED] == 1


def test_decode_partial_rejects_null_and_misaligned(lib):
    nb.mla_reset_counters()
    ptrs = [FAKE] * 8
    ptrs[2] = 0
    assert call_partial(lib, desc(), 2, ptrs) == nb.MLA_ERR_INVALID_ARG
    ptrs = [FAKE] * 8
    ptrs[2] = FAKE + 8  # ckv not 16-byte aligned
    assert call_partial(lib, desc(), 2, ptrs) == nb.MLA_ERR_INVALID_ARG
    ptrs = [FAKE] * 8
    ptrs[6] = FAKE + 4  # partials not 16-byte aligned
    assert call_partial(lib, desc(), 2, ptrs) == nb.MLA_ERR_INVALID_ARG
    assert nb.mla_get_counters()[nb.CTR_PARTIAL_TC] == 0


def test_merge_rejects_before_launch(lib):
    nb.mla_reset_counters()
    f = lib.mla_merge_states
    assert f(FAKE, FAKE, FAKE, 1, 1, 24, FAKE, 0, None, None) == nb.MLA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, 1, 1, 16, FAKE, 5, None, None) == nb.MLA_ERR_UNSUPPORTED
    assert f(None, FAKE, FAKE, 1, 1, 16, FAKE, 0, None, None) == nb.MLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 0, 1, 16, FAKE, 0, None, None) == nb.MLA_ERR_INVALID_ARG
    assert f(FAKE + 4, FAKE, FAKE, 1, 1, 16, FAKE, 0, None, None) == nb.MLA_ERR_INVALID_ARG
    assert nb.mla_get_counters()[nb.CTR_MERGE] == 0


def test_sizes_and_strings(lib):
    assert nb.mla_partials_bytes(8, 1, 16) == 8 * 16 * 512 * 4
    assert lib.mla_lse_bytes(8, 2, 16) == 8 * 2 * 16 * 4
    assert nb.status_string(nb.MLA_ERR_TIMEOUT) == "device wait timed out"
    assert nb.mla_version() >= 1


def test_descriptor_keeps_its_tensors_alive():
    # a descriptor stores raw pointers to the partition table and the workspace: the tensors behind
    # them must live as long as the descriptor, whatever the caller keeps
    import gc
    import types
    import weakref
    import torch
    from mla_split_kv_gb300 import runtime as rt
    case = types.SimpleNamespace(num_requests=1, num_heads=16, q_len=1, block_size=32, dtype="f16", causal=False,
                                 cache_scale=1.0)
    dc = types.SimpleNamespace(case=case, ckv=torch.zeros(4, 1), block_table=torch.zeros(1, 4, dtype=torch.int32))
    chunks = torch.zeros(3, 4, dtype=torch.int32)
    ws = torch.zeros(256, dtype=torch.uint8)
    refs = (weakref.ref(chunks), weakref.ref(ws))
    desc = rt.make_desc(dc, chunks, nb.MLA_KERNEL_TC, 4, types.SimpleNamespace(cuda_stream=0), 2, ws)
    assert desc.chunks == chunks.data_ptr() and desc.workspace == ws.data_ptr()
    del chunks, ws
    gc.collect()
    assert all(r() is not None for r in refs)
    del desc
    gc.collect()
    assert all(r() is None for r in refs)


def call_static(lib, d, P=2, ptrs=None):
    p = [FAKE] * 8 if ptrs is None else ptrs
    return lib.mla_decode_partial_static(p[0], p[1], p[2], p[3], p[4], p[5], ctypes.c_float(0.07), P, p[6], p[7],
                                         ctypes.byref(d))


@pytest.mark.parametrize("kw,P", [
    (dict(clusters_per_chunk=4, cluster_ctas=0), 2),
    (dict(clusters_per_chunk=4, cluster_ctas=1), 2),
    (dict(clusters_per_chunk=4, cluster_ctas=2, num_heads=64), 2),
    (dict(clusters_per_chunk=4, cluster_ctas=2, kernel=nb.MLA_KERNEL_SIMT), 2),
    (dict(clusters_per_chunk=17, cluster_ctas=2), 2),
    (dict(clusters_per_chunk=4, cluster_ctas=2, num_requests=40000), 2),
    (dict(clusters_per_chunk=4, cluster_ctas=2, num_heads=32), 2),
    (dict(clusters_per_chunk=4, cluster_ctas=2), 0),
])
def test_static_entry_gives_the_plain_entrys_status_before_any_device_work(lib, kw, P):
    """The allocation-free variant validates the whole descriptor (all but the workspace, which it supplies)
    before its device set-up, so a bad descriptor gets the same status as from mla_decode_partial given a
    workspace, and nothing runs on a device (this machine may have none)."""
    d = desc(**kw)
    nb.mla_reset_counters()
    got = call_static(lib, d, P)
    plain = call_partial(lib, desc(workspace=FAKE, workspace_bytes=BIG, **kw), P)
    assert got == plain and got in (nb.MLA_ERR_INVALID_ARG, nb.MLA_ERR_UNSUPPORTED)
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_REJECTED] == 2 and ctr[nb.CTR_PARTIAL_TC] == 0


def test_static_entry_rejects_a_plan_beyond_its_scratch_before_any_device_work(lib):
    d = desc(clusters_per_chunk=16, cluster_ctas=2, num_requests=64, max_blocks_per_req=8)
    assert nb.mla_workspace_bytes(64, 16, 2, 1, 16) > nb.MLA_STATIC_WORKSPACE_BYTES
    nb.mla_reset_counters()
    assert call_static(lib, d, 1) == nb.MLA_ERR_CAPACITY
    assert nb.mla_get_counters()[nb.CTR_REJECTED] == 1


def call_decode(lib, d, P=2, o_indptr=FAKE, out=FAKE, out_dtype=nb.MLA_F16, out_lse=None):
    p = [FAKE] * 8
    return lib.mla_decode(p[0], p[1], p[2], p[3], p[4], p[5], ctypes.c_float(0.07), P, p[6], p[7], o_indptr, out,
                          out_dtype, out_lse, ctypes.byref(d))


@pytest.mark.parametrize("kw,args,want", [
    (dict(cluster_ctas=2), dict(o_indptr=None), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(out=None), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(out=FAKE + 8), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(out_lse=FAKE + 2), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(out_dtype=7), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=2, decode_merge=5), dict(), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2, decode_merge=1), dict(), nb.MLA_ERR_INVALID_ARG),                  # no workspace
    (dict(cluster_ctas=2, decode_merge=1, workspace=FAKE, workspace_bytes=64), dict(), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2, num_heads=24), dict(), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=4, clusters_per_chunk=4, decode_merge=1, workspace=FAKE, workspace_bytes=1024), dict(),
     nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=4, clusters_per_chunk=4), dict(), nb.MLA_ERR_INVALID_ARG),              # two launches, no ws
])
def test_decode_rejects_before_launch(lib, kw, args, want):
    nb.mla_reset_counters()
    assert call_decode(lib, desc(**kw), 2, **args) == want
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_REJECTED] == 1 and ctr[nb.CTR_PARTIAL_TC] == 0 and ctr[nb.CTR_DECODE_FUSED] == 0


def test_decode_workspace_layout():
    # one layout for mla_decode's two ways on the paired kernel: request tickets (16 per request) and a copy of
    # each chunk's LSE (the single launch's, each block 256-byte aligned), then the chunk tickets and one
    # [rows][512] fp32 entry per CTA pair (chunks x clusters per chunk x cluster / 2) with its [2][rows][2] row
    # maxima / sums
    def entries(N, k, C, rows):
        e = N * max(k, 1) * (C // 2)
        return -(-N * 8 // 256) * 256 + e * rows * 512 * 4 + e * 2 * rows * 2 * 4
    assert nb.mla_decode_workspace_bytes(1, 7, 1, 16, 1, 16) == 256 + 512 + entries(7, 1, 16, 16)
    assert nb.mla_decode_workspace_bytes(3, 7, 5, 4, 1, 16) == 256 + 512 + entries(7, 5, 4, 16)
    assert entries(7, 5, 4, 16) == nb.mla_workspace_bytes(7, 5, 4, 1, 16)  # the spread layout, for k > 1
    assert nb.mla_decode_workspace_bytes(0, 7, 1, 16, 1, 16) == 0


def call_decode_unembed(lib, d, P=2, o_indptr=FAKE, w=FAKE, w_dtype=nb.MLA_F16, v_head=128, out_v=FAKE,
                        out_dtype=nb.MLA_F16, out_lse=None):
    p = [FAKE] * 8
    return lib.mla_decode_unembed(p[0], p[1], p[2], p[3], p[4], p[5], ctypes.c_float(0.07), P, p[6], p[7], o_indptr,
                                  w, w_dtype, v_head, out_v, out_dtype, out_lse, ctypes.byref(d))


@pytest.mark.parametrize("kw,args,want", [
    (dict(cluster_ctas=2), dict(o_indptr=None), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(w=None), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(w=FAKE + 8), nb.MLA_ERR_INVALID_ARG),  # W_UV^T not 16-byte aligned
    (dict(cluster_ctas=2), dict(out_v=None), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(out_v=FAKE + 2), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(out_lse=FAKE + 2), nb.MLA_ERR_INVALID_ARG),
    (dict(cluster_ctas=2), dict(v_head=48), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=2), dict(v_head=544), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=2), dict(w_dtype=nb.MLA_F32), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=2), dict(out_dtype=7), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=2, num_heads=24), dict(), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=2), dict(), nb.MLA_ERR_INVALID_ARG),  # the paired kernel's entries need a workspace
    (dict(cluster_ctas=2, decode_merge=1, workspace=FAKE, workspace_bytes=BIG), dict(), nb.MLA_ERR_UNSUPPORTED),
    (dict(cluster_ctas=4, clusters_per_chunk=4), dict(), nb.MLA_ERR_INVALID_ARG),  # two launches, no workspace
])
def test_decode_unembed_rejects_before_launch(lib, kw, args, want):
    nb.mla_reset_counters()
    assert call_decode_unembed(lib, desc(**kw), 2, **args) == want
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_REJECTED] == 1 and ctr[nb.CTR_PARTIAL_TC] == 0 and ctr[nb.CTR_PARTIAL_SIMT] == 0
    assert ctr[nb.CTR_WRAP] == 0


def call_merge_unembed(lib, partials=FAKE, B=2, q_len=1, H=16, w=FAKE, w_dtype=nb.MLA_F16, v_head=128, out=FAKE,
                       out_dtype=nb.MLA_F16, out_lse=None):
    return lib.mla_merge_unembed(partials, FAKE, FAKE, B, q_len, H, w, w_dtype, v_head, out, out_dtype, out_lse, None)


@pytest.mark.parametrize("args,want", [
    (dict(partials=None), nb.MLA_ERR_INVALID_ARG),
    (dict(partials=FAKE + 4), nb.MLA_ERR_INVALID_ARG),
    (dict(w=FAKE + 8), nb.MLA_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), nb.MLA_ERR_INVALID_ARG),
    (dict(out_lse=FAKE + 1), nb.MLA_ERR_INVALID_ARG),
    (dict(B=0), nb.MLA_ERR_INVALID_ARG),
    (dict(H=24), nb.MLA_ERR_UNSUPPORTED),
    (dict(q_len=nb.MLA_MAX_Q_LEN + 1), nb.MLA_ERR_UNSUPPORTED),
    (dict(v_head=40), nb.MLA_ERR_UNSUPPORTED),
    (dict(v_head=0), nb.MLA_ERR_UNSUPPORTED),
    (dict(w_dtype=nb.MLA_E4M3), nb.MLA_ERR_UNSUPPORTED),
    (dict(out_dtype=9), nb.MLA_ERR_UNSUPPORTED),
    (dict(B=65535 * 16 + 1), nb.MLA_ERR_UNSUPPORTED),  # more row groups than a grid's z dimension holds
])
def test_merge_unembed_rejects_before_launch(lib, args, want):
    nb.mla_reset_counters()
    assert call_merge_unembed(lib, **args) == want
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_REJECTED] == 1 and ctr[nb.CTR_WRAP] == 0


def call_cache_append(lib, ckv_new=FAKE, B=2, q_len=1, bs=32, num_blocks=8, max_blocks=4, ckv=FAKE):
    return lib.mla_cache_append(ckv_new, FAKE, FAKE, FAKE, B, q_len, bs, num_blocks, max_blocks, ckv, FAKE, None)


@pytest.mark.parametrize("args,want", [
    (dict(ckv_new=None), nb.MLA_ERR_INVALID_ARG),
    (dict(ckv_new=FAKE + 8), nb.MLA_ERR_INVALID_ARG),
    (dict(ckv=None), nb.MLA_ERR_INVALID_ARG),
    (dict(B=0), nb.MLA_ERR_INVALID_ARG),
    (dict(num_blocks=0), nb.MLA_ERR_INVALID_ARG),
    (dict(max_blocks=0), nb.MLA_ERR_INVALID_ARG),
    (dict(q_len=0), nb.MLA_ERR_UNSUPPORTED),
    (dict(q_len=nb.MLA_MAX_Q_LEN + 1), nb.MLA_ERR_UNSUPPORTED),
    (dict(bs=48), nb.MLA_ERR_UNSUPPORTED),
])
def test_cache_append_rejects_before_launch(lib, args, want):
    nb.mla_reset_counters()
    assert call_cache_append(lib, **args) == want
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_REJECTED] == 1 and ctr[nb.CTR_WRAP] == 0
