"""Failure detection on the GPU without a fault: the bounded device waits run out.

Every wait in the partial kernels (mbarrier phases, the peer CTA's data, the
MMA issuer's idle time) gives up after the limit set with
mla_set_wait_timeout_ns; the kernel then flags MLA_ERR_TIMEOUT in its device
error word, drains what it has in flight and returns. Here the limit is set to
a few microseconds on a long context, far below the time the work takes, so
every role of every CTA gives up at its next wait: the call must come back
with MLA_ERR_TIMEOUT from mla_check_device_errors, and the next call on the
same context, with the default limit back, must be correct against the
oracle. Nothing here traps, asserts on the device, or waits without a bound.
"""
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
SHORT_NS = 2_000             # a few microseconds: far less than one call takes
DEFAULT_NS = 2_000_000_000   # the library's default limit


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    nbuild.build()
    nb.load()
    nb.mla_check_device_errors(None)
    yield
    nb.mla_set_wait_timeout_ns(DEFAULT_NS)
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_OK, f"device error word {code:#x}"


def close_to(got, ref):
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    return err <= MAX_ABS and rel <= REL_L2, (err, rel)


def planned_call(case, dc, max_partitions=0, score_exchange=0):
    dev = nb.mla_device_query()
    plan = nb.mla_plan(case.context_lens.tolist(), case.num_heads, case.q_len, case.block_size, dev,
                       max_partitions=max_partitions, dtype=case.dtype, merge_path=nb.MLA_MERGE_PARTIALS)
    chunks = rt.chunks_to_device(plan.chunks)
    ws = rt.alloc_workspace(plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, case.q_len, case.num_heads)
    part, lse = rt.alloc_partials(plan.num_chunks, case.q_len, case.num_heads)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")

    def call():
        rt.decode_partial(dc, part, lse, chunks_dev=chunks, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas,
                          subs=plan.clusters_per_chunk, workspace=ws, score_exchange=score_exchange)
        return rt.merge_states(part, lse, ind, case.num_requests, case.q_len, case.num_heads, "f32")

    return plan, ws, call


@pytest.mark.parametrize("which", ["pair_spread", "pair_cluster", "many_rows", "e4m3_pair", "many_rows_fp16_exchange",
                                   "many_rows_f32_exchange", "e4m3_many_rows"])
def test_bounded_waits_run_out_then_the_context_is_usable(which):
    if which == "pair_spread":      # 16 fp16 rows, 131072 tokens: partitions spread over clusters (tickets)
        case = gen.make_decode_case(21, [131072], num_heads=16, block_size=32, dtype="f16")
        heads = [0, 8, 15]
    elif which == "pair_cluster":   # 16 fp16 rows, 65536 tokens: partitions on clusters of 16 CTAs
        case = gen.make_decode_case(22, [65536], num_heads=16, block_size=32, dtype="f16")
        heads = [3, 12]
    elif which == "e4m3_pair":      # E4M3 caches on the pairs: the widening's meetings and loads give up too
        case = gen.make_decode_case(24, [131072], num_heads=16, block_size=32, dtype="e4m3")
        heads = [1, 14]
    elif which == "e4m3_many_rows":  # E4M3 caches on the 128-row kernel
        case = gen.make_decode_case(25, [65536, 40000], num_heads=128, block_size=64, dtype="e4m3")
        heads = [0, 77, 127]
    else:                           # 128 bf16 rows on a CTA pair (the many-head kernel)
        case = gen.make_decode_case(23, [65536, 40000], num_heads=128, block_size=64, dtype="bf16", latent_std=0.5)
        heads = [0, 77, 127]
    dc = rt.upload(case)
    plan, ws, call = planned_call(case, dc, max_partitions=64 if case.num_heads == 128 else 0,
                                  score_exchange={"many_rows_fp16_exchange": nb.MLA_SCORE_EXCHANGE_F16,
                                                  "many_rows_f32_exchange": nb.MLA_SCORE_EXCHANGE_F32}.get(which, 0))
    if which == "pair_spread":
        assert plan.clusters_per_chunk > 1
    if which == "pair_cluster":
        assert plan.clusters_per_chunk == 1 and plan.cluster_ctas >= 4
    if which.startswith("many_rows") or which == "e4m3_many_rows":
        assert plan.cluster_ctas == 2
    nb.mla_check_device_errors(None)
    nb.mla_reset_counters()
    try:
        nb.mla_set_wait_timeout_ns(SHORT_NS)
        call()
        st, code = nb.mla_check_device_errors(None)
    finally:
        nb.mla_set_wait_timeout_ns(DEFAULT_NS)
    assert nb.mla_get_counters()[nb.CTR_PARTIAL_TC] == 1  # the kernel did launch
    assert st == nb.MLA_ERR_TIMEOUT and code & 1, (st, code)
    # the owner of a workspace zeroes it again after a device error (the header's contract)
    if ws is not None:
        ws.zero_()
    out = call()
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_OK, code
    ref, _ = orc.unsplit(case, heads=heads)
    ok, e = close_to(out.cpu().numpy()[:, :, heads].astype(np.float64), ref[:, :, heads])
    assert ok, f"after the timeout: max-abs {e[0]:.3e} rel-L2 {e[1]:.3e}"
    if ws is not None:  # a completed call leaves its tickets at zero
        assert int(ws[: 8 * plan.num_chunks].view(torch.int32).abs().sum()) == 0

