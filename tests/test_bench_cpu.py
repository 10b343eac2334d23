"""The benchmark's bookkeeping on the CPU: algorithmic bytes, the profiled
traffic lookup and the whole-job figure (no GPU needed)."""
import json
import os

import bench


def test_algorithmic_bytes_match_the_stated_formula():
    # per layer call: latent stream + block table + queries + partials and lse written and read back + output
    for L, N in [(32768, 7), (131072, 7), (4096, 2), (1000, 1)]:
        part, merge = bench.algorithmic_bytes(L, N)
        want = (L * 576 * 2 + -(-L // 32) * 4 + 16 * 576 * 2 + 2 * N * 16 * 513 * 4 + 16 * 512 * 2)
        assert part + merge == want
        assert merge == N * 16 * 513 * 4 + 16 * 512 * 2


def test_latent_stream_of_the_sweep():
    # 37.7 / 56.6 / 75.5 / 94.4 / 113.2 / 151.0 MB for the six contexts
    mb = [round(L * bench.LATENT_BYTES_PER_TOKEN / 1e6, 1) for L in bench.CONTEXTS]
    assert mb == [37.7, 56.6, 75.5, 94.4, 113.2, 151.0]


def test_profiled_traffic_only_for_the_profiled_source():
    path = os.path.join(bench.ROOT, "profiles", "mla_partial_tc128_kernel_dram_traffic.json")
    prof = json.load(open(path))
    got = bench.profiled_traffic("mla_partial_tc128_kernel", 1000)
    if prof["kernel_source_hash"] == bench.kernel_source_hash():
        assert got == round(prof["dram_bytes_per_token"] * 1000)
    else:  # the kernel changed since the counters were taken: no traffic figure
        assert got is None
    assert bench.profiled_traffic("no_such_kernel", 1000) is None


def test_whole_job_figure_counts_every_replica():
    # 2 ranks each replaying 60 calls in 1.2 ms: the job did 120 calls in 1.2 ms
    assert abs(bench.job_us_per_call(1.2, 60, 2) - 10.0) < 1e-12
    assert abs(bench.job_us_per_call(1.2, 60, 1) - 20.0) < 1e-12
