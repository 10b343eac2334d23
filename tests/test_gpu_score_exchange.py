"""The 128-row kernel's score exchange options: partial scores exchanged as fp16
(score_exchange = MLA_SCORE_EXCHANGE_F16), and none exchanged (MLA_SCORE_EXCHANGE_NONE: each CTA of a
pair computes the full scores, part of the queries in tensor memory).

Each CTA of a pair rounds its partial dot product of a tile to fp16 once and
both add the same rounded values, so they still take the same decisions. The
rounding adds |s| x 2^-12 per half before the softmax scale; on the test
inputs (latents N(0, 1) or N(0, 0.5), queries N(0, 1)) the results stay within
the stated tolerance: max-abs 2e-3 and rel-L2 1e-3 on fp32 results against the
f64 oracle. The default exchange (fp32) is untouched: the two give different
bits, and each is bitwise repeatable.
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
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e} rel-L2 {rel:.3e}"


def planned(case, exchange, max_partitions=16):
    lens = case.context_lens.tolist()
    plan = nb.mla_plan(lens, case.num_heads, case.q_len, case.block_size, nb.mla_device_query(),
                       max_partitions=max_partitions, dtype=case.dtype)
    dc = rt.upload(case)
    chunks = rt.chunks_to_device(plan.chunks)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    part, lse = rt.alloc_partials(plan.num_chunks, case.q_len, case.num_heads)
    out = torch.empty((case.num_requests, case.q_len, case.num_heads, 512), dtype=torch.float32, device="cuda")
    nb.mla_reset_counters()
    rt.decode(dc, part, lse, ind, out, kernel=nb.MLA_KERNEL_TC, cluster=plan.cluster_ctas, chunks_dev=chunks,
              score_exchange=exchange)
    assert nb.mla_get_counters()[nb.CTR_PARTIAL_TC] == 1
    return part, lse, out


@pytest.mark.parametrize("H,q_len,dtype,bs,std,heads", [
    (128, 1, "bf16", 64, 0.5, [0, 37, 64, 127]),   # the many-head decode's shape
    (64, 1, "f16", 32, 1.0, [0, 21, 42, 63]),       # a 64-row group: half its rows padding
    (16, 16, "f16", 32, 1.0, [0, 7, 15]),           # a verify window of 16 rows per request, causal
    (16, 9, "f16", 16, 1.0, [0, 15]),               # 144 rows: a full group and a 16-row one
])
def test_fp16_exchange_against_the_oracle(H, q_len, dtype, bs, std, heads):
    lens = [9000, 2500, 130]
    case = gen.make_decode_case(81, lens, num_heads=H, q_len=q_len, block_size=bs, dtype=dtype, latent_std=std,
                                causal=q_len > 1)
    part, lse, out = planned(case, nb.MLA_SCORE_EXCHANGE_F16)
    ref, _ = orc.unsplit(case, heads=heads)
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], f"fp16 exchange H={H} q_len={q_len} {dtype}")
    # the default exchange on the same case: other bits (the fp16 rounding is real), same tolerance
    _, _, out32 = planned(case, nb.MLA_SCORE_EXCHANGE_F32)
    assert not torch.equal(out, out32)
    assert_close(out32.cpu().numpy()[:, :, heads], ref[:, :, heads], "fp32 exchange")


def test_fp16_exchange_bitwise_repeatable():
    case = gen.make_decode_case(82, [7000, 2049], num_heads=128, block_size=64, dtype="bf16", latent_std=0.5)
    runs = [planned(case, nb.MLA_SCORE_EXCHANGE_F16) for _ in range(3)]
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)


@pytest.mark.parametrize("H,q_len,dtype,bs,std,heads,lens", [
    (128, 1, "bf16", 64, 0.5, [0, 37, 64, 127], [9000, 2500, 130]),  # the many-head decode's shape
    (128, 1, "f16", 16, 1.0, [0, 77, 127], [4099, 1, 2222]),          # block 16, a one-token request
    (64, 1, "f16", 32, 1.0, [0, 21, 42, 63], [9000, 2500, 130]),      # a 64-row group: half its rows padding
    (64, 2, "bf16", 32, 0.5, [0, 40, 63], [3000, 65]),                 # two window rows per request, causal
    (16, 16, "f16", 32, 1.0, [0, 7, 15], [9000, 2500, 130]),           # a verify window of 16, causal
    (16, 32, "f16", 64, 1.0, [0, 15], [6000, 777]),                    # 512 rows: four groups, causal
])
def test_no_exchange_against_the_oracle(H, q_len, dtype, bs, std, heads, lens):
    """No exchange: exact (within the stated tolerance of the oracle, like the fp32 exchange) and within
    fp32 rounding of the fp32 exchange's results (only the order of the 576-term sums differs)."""
    case = gen.make_decode_case(83, lens, num_heads=H, q_len=q_len, block_size=bs, dtype=dtype, latent_std=std,
                                causal=q_len > 1)
    part, lse, out = planned(case, nb.MLA_SCORE_EXCHANGE_NONE)
    ref, ref_lse = orc.unsplit(case, heads=heads)
    assert_close(out.cpu().numpy()[:, :, heads], ref[:, :, heads], f"no exchange H={H} q_len={q_len} {dtype}")
    # the two exact ways differ only by the order of fp32 sums: well inside the stated tolerance (a quarter)
    part32, lse32, out32 = planned(case, nb.MLA_SCORE_EXCHANGE_F32)
    assert (out - out32).abs().max().item() <= MAX_ABS / 4
    live = torch.isfinite(lse32)
    assert torch.equal(torch.isfinite(lse), live) and (lse - lse32)[live].abs().max().item() <= MAX_ABS / 4


def test_no_exchange_bitwise_repeatable():
    case = gen.make_decode_case(84, [7000, 2049], num_heads=128, block_size=64, dtype="bf16", latent_std=0.5)
    runs = [planned(case, nb.MLA_SCORE_EXCHANGE_NONE) for _ in range(3)]
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)
