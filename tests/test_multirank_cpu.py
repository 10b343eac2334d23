"""The N-replica path of bench.py on CPU ranks (gloo, world size 2).

Decode requests are independent, so N GPUs run N replicas of the workload
with no collective on the data path; the only cross-rank steps are the
barrier around the timed region and the max over ranks of the timed
duration. These run here on CPU ranks over gloo, together with the host-side
planner each rank uses and the reference arm's rank rule.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from mla_split_kv_gb300 import binding as nb

        # the slowest rank's time is the job's time
        local_ms = 10.0 + 5.0 * rank
        dist.barrier()
        job_ms = bench.max_over_ranks(local_ms, "cpu")
        # each replica plans its own copy of the workload: identical host plans on every rank
        dev = nb.mla_device_info_t()
        dev.num_sms = 152
        for k, v in enumerate([152, 76, 36, 15, 7]):
            dev.max_clusters[k] = v
        plans = [nb.mla_plan([L], 16, 1, 32, dev) for L in bench.CONTEXTS]
        sig = torch.tensor([[p.num_chunks, p.cluster_ctas, p.clusters_per_chunk, p.chunks[-1][2]] for p in plans],
                           dtype=torch.int64)
        gathered = [torch.zeros_like(sig) for _ in range(world)]
        dist.all_gather(gathered, sig)
        # the reference arm runs on rank 0 only; the other ranks return without work
        class A:
            steps = 1
        ref = bench.run_reference(A(), rank, world) if rank != 0 else "rank0"
        out[rank] = (job_ms, bench.job_us_per_call(job_ms, 6 * 20, world),
                     all(torch.equal(g, gathered[0]) for g in gathered), ref)
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_max_time_identical_plans_reference_on_rank0():
    world, port = 2, _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert set(out.keys()) == {0, 1}
    for r in range(world):
        job_ms, us, same_plans, ref = out[r]
        assert job_ms == pytest.approx(15.0)           # max over ranks, seen by every rank
        assert us == pytest.approx(15.0 * 1e3 / (6 * 20 * 2))
        assert same_plans
    assert out[1][3] is None                           # non-zero ranks of the reference arm do nothing


PROBE = """
import json, os, sys
sys.path.insert(0, {root!r})
import bench
rank, world, local = bench.init_ranks()
job_ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
if rank == 0:
    print(json.dumps({{"n_gpus": world, "job_ms": job_ms, "local_ranks": local,
                      "backend": __import__("torch").distributed.get_backend()}}))
bench.finish_ranks(world)
"""


def test_launcher_starts_one_rank_per_gpu_on_cpu_ranks(tmp_path):
    """bench.py --gpus N with no launcher around it starts N ranks through torch's launcher (rendezvous on
    127.0.0.1); each binds to its LOCAL_RANK and joins the group (gloo here, no GPU), and rank 0 sees the
    slowest rank's time. The same launch and rank set-up serve the benchmark."""
    import json
    import subprocess
    import sys
    sys.path.insert(0, ROOT)
    import bench

    probe = tmp_path / "probe.py"
    probe.write_text(PROBE.format(root=ROOT))
    res = bench.launch_replicas(2, [], script=str(probe), stdout=subprocess.PIPE)
    assert res.returncode == 0
    line = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(line) == 1, res.stdout
    got = json.loads(line[0])
    assert got["n_gpus"] == 2 and got["job_ms"] == 15.0 and got["local_ranks"] == 0 and got["backend"] == "gloo"
    cmd = bench.replica_command(4, "bench.py", ["--gpus", "4"], 29500)
    assert "--nproc-per-node=4" in cmd and "--master-addr=127.0.0.1" in cmd and cmd[-2:] == ["--gpus", "4"]


def test_bench_refuses_a_gpu_count_that_differs_from_the_launcher(monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert "does not match" in str(e.value)
