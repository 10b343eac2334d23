"""The allocation-free entry point (mla_decode_partial_static) against mla_decode_partial.

Collected last on purpose: the first call of the static variant on a device
does its set-up (symbol lookup and clearing of the library's scratch), and
this file must pass both alone in a fresh process and after every other test.
"""
import ctypes

import pytest
import torch

from mla_split_kv_gb300 import binding as nb
from mla_split_kv_gb300 import build as nbuild
from mla_split_kv_gb300 import inputs as gen
from mla_split_kv_gb300 import runtime as rt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    nbuild.build()
    nb.load()
    yield
    st, code = nb.mla_check_device_errors(None)
    assert st == nb.MLA_OK, f"device error word {code:#x}"


def call_static(dc, part, lse, desc, P):
    nb.mla_decode_partial_static(dc.q_abs.data_ptr(), dc.q_pe.data_ptr(), dc.ckv.data_ptr(), dc.kpe.data_ptr(),
                                 dc.block_table.data_ptr(), dc.context_lens.data_ptr(), float(dc.case.scale), P,
                                 part.data_ptr(), lse.data_ptr(), desc)


@pytest.mark.parametrize("L,P,C,k", [(65536, 6, 4, 6), (20017, 3, 2, 5)])
def test_static_entry_matches_workspace_entry_two_calls_in_a_row(L, P, C, k):
    case = gen.make_decode_case(7, [L], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    assert nb.mla_workspace_bytes(P, k, C, 1, 16) <= nb.MLA_STATIC_WORKSPACE_BYTES
    # the existing entry point, with a caller workspace
    ref_part, ref_lse = rt.alloc_partials(P, 1, 16)
    ws = rt.alloc_workspace(P, k, C, 1, 16)
    rt.decode_partial(dc, ref_part, ref_lse, num_partitions=P, kernel=nb.MLA_KERNEL_TC, cluster=C, subs=k,
                      workspace=ws)
    # the static variant, twice in a row on the same stream (its tickets must be back at zero in between)
    desc = rt.make_desc(dc, None, nb.MLA_KERNEL_TC, C, None, k, None)
    for _ in range(2):
        part, lse = rt.alloc_partials(P, 1, 16)
        part.fill_(float("nan"))
        nb.mla_reset_counters()
        call_static(dc, part, lse, desc, P)
        torch.cuda.synchronize()
        ctr = nb.mla_get_counters()
        assert ctr[nb.CTR_PARTIAL_TC] == 1 and ctr[nb.CTR_CTAS] == P * C * k
        assert torch.equal(part, ref_part)
        assert torch.equal(lse, ref_lse)


def test_static_entry_rejects_plans_beyond_its_scratch():
    case = gen.make_decode_case(8, [4096], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    P, k = 64, 16  # 64 * 16 sub-partials of 16 x 513 floats: more than 4 MiB
    assert nb.mla_workspace_bytes(P, k, 2, 1, 16) > nb.MLA_STATIC_WORKSPACE_BYTES
    part, lse = rt.alloc_partials(P, 1, 16)
    desc = rt.make_desc(dc, None, nb.MLA_KERNEL_TC, 2, None, k, None)
    nb.mla_reset_counters()
    with pytest.raises(nb.MlaError) as e:
        call_static(dc, part, lse, desc, P)
    assert e.value.status == nb.MLA_ERR_CAPACITY
    ctr = nb.mla_get_counters()
    assert ctr[nb.CTR_REJECTED] == 1 and ctr[nb.CTR_PARTIAL_TC] == 0


def test_static_entry_is_usable_again_after_a_device_error():
    """A static call cut short by its bounded waits (a limit of a few microseconds) is reported by
    mla_check_device_errors, which then clears the library's scratch; the next two calls match the
    workspace entry point bit for bit."""
    L, P, C, k = 65536, 6, 4, 6
    case = gen.make_decode_case(7, [L], num_heads=16, block_size=32, dtype="f16")
    dc = rt.upload(case)
    ref_part, ref_lse = rt.alloc_partials(P, 1, 16)
    ws = rt.alloc_workspace(P, k, C, 1, 16)
    rt.decode_partial(dc, ref_part, ref_lse, num_partitions=P, kernel=nb.MLA_KERNEL_TC, cluster=C, subs=k,
                      workspace=ws)
    desc = rt.make_desc(dc, None, nb.MLA_KERNEL_TC, C, None, k, None)
    part, lse = rt.alloc_partials(P, 1, 16)
    nb.mla_check_device_errors(None)
    try:
        nb.mla_set_wait_timeout_ns(2_000)
        call_static(dc, part, lse, desc, P)
        st, code = nb.mla_check_device_errors(None)
    finally:
        nb.mla_set_wait_timeout_ns(2_000_000_000)
    assert st == nb.MLA_ERR_TIMEOUT and code & 1, (st, code)
    for _ in range(2):
        part.fill_(float("nan"))
        call_static(dc, part, lse, desc, P)
        torch.cuda.synchronize()
        assert torch.equal(part, ref_part)
        assert torch.equal(lse, ref_lse)
