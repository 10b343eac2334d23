"""Benchmark: MLA split-KV decode layer calls on one GB300 (or N replicas).

Workload: B=1, H=16, kv_lora_rank 512, rope 64, fp16, block 32, contexts
32768 / 49152 / 65536 / 81920 / 98304 / 131072 tokens (N(0,1) latents, random
block permutation), partitions chosen by the planner. One step = one layer
call at each of the six contexts through mla_decode's default (the paired
partial kernel writing every CTA pair's part, the entries merge kernel, its
programmatic dependent, merging them); the six caches live in disjoint memory (528 MB together, > L2),
so every call streams its latent from HBM. Each call's tables and the cache
rows before its window are complete before the step (tables_ready,
prefix_ready).

Printed: one JSON line. `value` = mean microseconds per layer call over the
sweep (device time, inputs resident, each step replayed from one CUDA graph);
`e2e` = the same through mla_decode with host buffers (queries, block tables
and plan of the six calls copied in with one copy from one pinned buffer, the
six outputs copied out with one copy, every step; the step replayed from a
CUDA graph captured through those calls, host wall clock with a synchronize
per step; `eager_us` launches them one by one); `roofline` = the layer
call's algorithmic HBM bytes / its CUDA-event time in the timed graph against
the measured copy bandwidth; `cpu_baseline` = the f64 oracle on the host
cores. Outside the timed region: `without_prefix_ready_us` (every cache read after the preceding kernel has
finished), `single_launch_us` (one launch per call whose last CTAs merge the
chunk partials), `partial_kernel_alone` (the ABI's mla_decode_partial),
`per_ctx` (each context alone, its planned split, a single cold call after an
L2 flush and the host planner's time per call), `trials` (median / min / max
over five more K-step trials), `many_heads` (the many-head workload),
`verify_windows`, `batch_grid`, `e4m3_caches` (the same sweep on 8-bit E4M3
caches), `bf16` (the same sweep in bf16) and `layer_with_append_and_unembed`
(the new token's cache write, the partial decode and the merge with the
W_UV^T unembed at 32K and 131K). `--impl reference` times the oracle itself
on the same workload; `--gpus N` without a launcher starts N ranks (one
replica per GPU).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONTEXTS = [32768, 49152, 65536, 81920, 98304, 131072]
H, BS, DTYPE, SEED = 16, 32, "f16", 2
LATENT_BYTES_PER_TOKEN = (512 + 64) * 2
WORKLOAD = "mla_decode_ctx_sweep_B1_H16_r512_rope64_fp16_bs32"
METRIC = "us per MLA decode layer call (mean over ctx 32K-131K), HBM GB/s as fraction of peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", default="tc", choices=["tc", "simt"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-ctx", type=int, default=0,
                    help="profiling case: only --launches plain layer calls at this context (of the sweep), then exit")
    ap.add_argument("--profile-many-heads", action="store_true",
                    help="profiling case: only --launches plain layer calls of the many-head workload, then exit")
    ap.add_argument("--profile-verify", type=int, default=0,
                    help="profiling case: only --launches plain verify-window calls of this q_len, then exit")
    ap.add_argument("--launches", type=int, default=5)
    ap.add_argument("--profile-exchange", default="f32", choices=["f32", "f16", "none", "exact"],
                    help="profiling case of the many-head workload: the 128-row kernel's partial-score exchange")
    ap.add_argument("--profile-cache", default="f16", choices=["f16", "e4m3"],
                    help="profiling case at --profile-ctx: the cache type (e4m3: 8-bit caches, scale 1/4)")
    ap.add_argument("--profile-layer", action="store_true",
                    help="profiling case at --profile-ctx: each call is the layer call with the cache write and the "
                         "unembed (mla_cache_append + mla_decode_unembed, v_head 128)")
    ap.add_argument("--profile-split", default="",
                    help="profiling case: 'P,C' = a uniform split into P partitions on clusters of C CTAs instead of "
                         "the planner's plan")
    ap.add_argument("--skip-extra", action="store_true",
                    help="leave out the verify-window and batch-grid timings (reported beside the headline)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# CPU oracle timing (bounded sample), run in a spawned pool over shared memory
# ---------------------------------------------------------------------------

def _oracle_worker(args):
    import numpy as np
    from multiprocessing import shared_memory

    from mla_split_kv_gb300.inputs import DecodeCase
    from oracle import mla_oracle as orc

    meta, heads = args
    shms, arrays = [], {}
    for key, (name, shape, dt) in meta["arrays"].items():
        shm = shared_memory.SharedMemory(name=name)
        shms.append(shm)
        arrays[key] = np.ndarray(shape, dtype=np.dtype(dt), buffer=shm.buf)
    case = DecodeCase(dtype=meta["dtype"], num_heads=meta["H"], q_len=1, block_size=meta["bs"],
                      scale=meta["scale"], causal=False, **arrays)
    out, _ = orc.unsplit(case, heads=heads)
    s = float(np.nansum(out))
    del arrays, case, out
    for shm in shms:
        shm.close()
    return s


class OraclePool:
    """Process pool (spawn) that runs the oracle, one head group per worker."""

    def __init__(self, cores):
        import multiprocessing as mp

        os.environ["OPENBLAS_NUM_THREADS"] = "1"
        os.environ["OMP_NUM_THREADS"] = "1"
        self.cores = cores
        self.pool = mp.get_context("spawn").Pool(cores)

    def share(self, case):
        import numpy as np
        from multiprocessing import shared_memory

        meta = {"dtype": case.dtype, "H": case.num_heads, "bs": case.block_size, "scale": case.scale, "arrays": {}}
        shms = []
        for key in ("q_abs", "q_pe", "ckv", "kpe", "block_table", "context_lens"):
            a = np.ascontiguousarray(getattr(case, key))
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            meta["arrays"][key] = (shm.name, a.shape, a.dtype.str)
            shms.append(shm)
        return meta, shms

    def layer_call(self, meta, num_heads):
        groups = [list(range(h, num_heads, self.cores)) for h in range(min(self.cores, num_heads))]
        t0 = time.perf_counter()
        self.pool.map(_oracle_worker, [(meta, g) for g in groups])
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def make_case(i, L, dtype=DTYPE):
    """Context i of the sweep: seeded latents, a pool 25% larger than needed, random page order (E4M3 caches:
    cache scale 1/4)."""
    from mla_split_kv_gb300 import inputs as gen

    pages = gen.pages_for(L, BS)
    return gen.make_decode_case(SEED * 100 + i, [L], num_heads=H, block_size=BS, dtype=dtype,
                                pool_blocks=pages + pages // 4, cache_scale=0.25)


def make_cases():
    return [make_case(i, L) for i, L in enumerate(CONTEXTS)]


# many-head decode (the tensor-core-bound shape): B=8, H=128, bf16, block 64, contexts uniform in
# [4096, 65536] from the seed, latents N(0, 0.5), partitions planned per request
MH_B, MH_H, MH_BS, MH_SEED = 8, 128, 64, 4
MANY_HEADS = "mla_decode_B8_H128_bf16_bs64_ctx_U4K_64K"


def make_many_heads_case(dtype="bf16"):
    """The many-head workload; dtype "e4m3": the same lengths and pages over an E4M3 cache (scale 1/4) beside
    fp16 queries."""
    from mla_split_kv_gb300 import inputs as gen

    lens = gen.uniform_lengths(MH_SEED, MH_B, 4096, 65536)
    return gen.make_decode_case(MH_SEED, lens, num_heads=MH_H, block_size=MH_BS, dtype=dtype, latent_std=0.5,
                                cache_scale=0.25)


def many_heads_call(nb, rt, torch, stream=None, exchange=0, dtype="bf16"):
    """Upload the many-head case, plan it, and return a closure doing one layer call (partial + merge kernels);
    `exchange`: the 128-row kernel's score exchange (0: the exact default, no exchange on 16-bit caches; 1: fp16;
    2: none; 3: fp32)."""
    case = make_many_heads_case(dtype)
    dev = nb.mla_device_query()
    plan = nb.mla_plan(case.context_lens.tolist(), MH_H, 1, MH_BS, dev, max_partitions=64, dtype=dtype)
    dc = rt.upload(case)
    chunks_dev = rt.chunks_to_device(plan.chunks)
    part, lse = rt.alloc_partials(plan.num_chunks, 1, MH_H)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    out = torch.empty((MH_B, 1, MH_H, 512), dtype=torch.bfloat16 if dtype == "bf16" else torch.float16, device="cuda")
    desc = rt.make_desc(dc, chunks_dev, nb.MLA_KERNEL_TC, plan.cluster_ctas, stream, score_exchange=exchange)

    def call():  # mla_decode: the 128-row kernel, then the merge kernel
        rt.decode(dc, part, lse, ind, out, desc=desc)

    tokens = int(case.context_lens.sum())
    return call, plan, tokens


# verify windows (the tensor-core-bound shape at 16 and 32 rows): B=4 requests, H=16, fp16, block 32, a
# prefix of 81920 tokens in 3 non-contiguous segments (40960 / 28672 / 12288) and the window's own q_len
# tokens as a causal tail segment; every segment planned on its own, all merged per request by LSE
VW_B, VW_SEED, VW_QLENS = 4, 5, [4, 9, 16, 32]
VERIFY = "mla_verify_windows_B4_H16_fp16_bs32_prefix81920_in_3_segments"


def window_work(seg):
    """(flops, bytes) one window call must do: every visible (row, token) pair, and the latent stream plus
    tables, queries, partials written and read back, and the output."""
    segs = seg.segments
    B, q, Hh = segs[0].num_requests, segs[0].q_len, segs[0].num_heads
    prefix = sum(int(s.context_lens[0]) for s in segs[:-1])
    pairs = B * sum(prefix + i + 1 for i in range(q))  # row i of the window sees the prefix and i + 1 window tokens
    flops = pairs * Hh * 2 * (576 + 512)
    tokens = B * (prefix + q)
    pages = sum(-(-int(L) // s.block_size) for s in segs for L in s.context_lens)
    return flops, tokens * LATENT_BYTES_PER_TOKEN + pages * 4 + B * q * Hh * (576 * 2 + 512 * 2)


def verify_window_call(nb, rt, torch, stream, full, dc_base, q):
    """One verify-window layer call of q_len q over the segmented prefix: one partial launch per segment and
    one merge. Returns (call, the window's view of the case, the number of partial launches)."""
    from mla_split_kv_gb300 import inputs as gen

    dev = nb.mla_device_query()
    seg = gen.window_view(full, q)
    sp = rt.plan_segments(seg, dev, max_partitions=64)  # as the many-head timing: enough pairs to fill the GPU
    part, lse = rt.alloc_partials(sp.num_slots, q, H)
    out = torch.empty((VW_B, q, H, 512), dtype=torch.float16, device="cuda")
    launches = []
    for s, table, plan in zip(seg.segments, sp.chunk_tables, sp.plans):
        dc = rt.upload(s, ckv=dc_base.ckv, kpe=dc_base.kpe)
        ws = rt.alloc_workspace(plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, q, H)
        desc = rt.make_desc(dc, table, nb.MLA_KERNEL_TC, plan.cluster_ctas, stream, plan.clusters_per_chunk, ws,
                            tables_ready=True)
        launches.append((dc, desc))

    def call():
        for dc, desc in launches:
            rt.decode_partial(dc, part, lse, desc=desc)
        rt.merge_states(part, lse, sp.o_indptr, VW_B, q, H, "f16", out=out, stream=stream)

    call.plans = sp.plans
    return call, seg, len(launches)


def time_verify_windows(nb, rt, torch, stream, peaks, reps=5):
    from mla_split_kv_gb300 import inputs as gen

    full = gen.make_segmented_case(VW_SEED, B=VW_B, q_len=max(VW_QLENS), num_heads=H, block_size=BS)
    dc_base = rt.upload(full.base)  # the cache pool, shared by every window length
    rows = []
    for q in VW_QLENS:
        call, seg, nlaunch = verify_window_call(nb, rt, torch, stream, full, dc_base, q)
        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                call()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            g.replay()
            e[0].record(stream)
            g.replay()
            e[1].record(stream)
        stream.synchronize()
        us = e[0].elapsed_time(e[1]) * 1e3 / reps
        flops, nbytes = window_work(seg)
        tf = flops / (us * 1e-6) / 1e12
        gbs = nbytes / (us * 1e-6) / 1e9
        frac_t = tf / peaks["tensor_tflops"]
        frac_h = gbs / peaks["hbm_gbs"]
        rows.append({"q_len": q, "us_per_call": round(us, 3), "tflops": round(tf, 1), "hbm_gbs": round(gbs, 1),
                     "bound": "tensor" if flops / nbytes > peaks["tensor_tflops"] * 1e3 / peaks["hbm_gbs"] else "hbm",
                     "frac_tensor": round(frac_t, 4), "frac_hbm": round(frac_h, 4),
                     "flop_per_byte": round(flops / nbytes, 1),
                     "partitions_per_segment": [p.num_chunks for p in call.plans],
                     "launches": nlaunch + 1})
    return {"workload": VERIFY, "per_q_len": rows,
            "peaks": {"tensor_tflops": peaks["tensor_tflops"], "hbm_gbs": peaks["hbm_gbs"],
                      "source": peaks["source"]},
            "note": "each window call: one partial launch per segment (3 prefix segments + the causal window tail) "
                    "and one merge; the 377 MB prefix cache is larger than L2; fp16 tensor peak = the measured bf16 "
                    "dense peak (the same nominal rate)"}


# the batch grid of the many-head comparison (heads x batch), at an 8192-token context per request
GRID_HEADS, GRID_BATCH, GRID_CTX = [16, 64, 128], [1, 8, 32], 8192
GRID = "mla_decode_grid_H16_64_128_x_B1_8_32_ctx8192"


def time_batch_grid(nb, rt, torch, stream, reps=10):
    from mla_split_kv_gb300 import inputs as gen

    dev = nb.mla_device_query()
    rows = []
    for Hh in GRID_HEADS:
        dtype = "bf16" if Hh == 128 else "f16"
        for B in GRID_BATCH:
            case = gen.make_decode_case(40 + Hh + B, [GRID_CTX] * B, num_heads=Hh, block_size=BS if dtype == "f16" else 64,
                                        dtype=dtype, latent_std=0.5 if dtype == "bf16" else 1.0)
            plan = nb.mla_plan(case.context_lens.tolist(), Hh, 1, case.block_size, dev, max_partitions=64, dtype=dtype)
            dc = rt.upload(case)
            chunks = rt.chunks_to_device(plan.chunks)
            part, lse = rt.alloc_partials(plan.num_chunks, 1, Hh)
            ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
            out = torch.empty((B, 1, Hh, 512), dtype=rt.TORCH_DTYPE[dtype], device="cuda")
            ws = rt.alloc_decode_workspace(B, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, Hh)
            desc = rt.make_desc(dc, chunks, nb.MLA_KERNEL_TC, plan.cluster_ctas, stream, plan.clusters_per_chunk, ws,
                                tables_ready=True)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    rt.decode(dc, part, lse, ind, out, desc=desc)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    rt.decode(dc, part, lse, ind, out, desc=desc)
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            with torch.cuda.stream(stream):
                g.replay()
                e[0].record(stream)
                g.replay()
                e[1].record(stream)
            stream.synchronize()
            us = e[0].elapsed_time(e[1]) * 1e3 / reps
            tokens = B * GRID_CTX
            rows.append({"H": Hh, "B": B, "dtype": dtype, "us_per_call": round(us, 3),
                         "hbm_gbs": round(tokens * LATENT_BYTES_PER_TOKEN / (us * 1e-6) / 1e9, 1),
                         "tflops": round(tokens * Hh * 2 * (576 + 512) / (us * 1e-6) / 1e12, 1),
                         "partitions": plan.num_chunks, "cluster": plan.cluster_ctas,
                         "clusters_per_partition": plan.clusters_per_chunk,
                         "l2_resident": tokens * LATENT_BYTES_PER_TOKEN < 129e6})
    return {"workload": GRID, "cells": rows,
            "note": "repeats of one cache per cell; caches smaller than L2 (129 MB) are partly L2-resident"}


def oracle_timing(cases, steps, cores, budget_s=30.0):
    """Seconds per layer call of the oracle: every context once per step, bounded by budget_s."""
    pool = OraclePool(cores)
    shared = [pool.share(c) for c in cases]
    try:
        pool.layer_call(shared[0][0], H)  # worker start-up, imports
        per_call, t_start, done_steps = [], time.perf_counter(), 0
        for _ in range(max(1, steps)):
            for meta, _ in shared:
                per_call.append(pool.layer_call(meta, H))
            done_steps += 1
            if time.perf_counter() - t_start > budget_s:
                break
    finally:
        pool.close()
        for _, shms in shared:
            for s in shms:
                s.close()
                s.unlink()
    return per_call, done_steps


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def planner_host_us(nb, lens, dev, batches=5, reps=400):
    """Host time of one mla_plan call (median over batches of the per-call mean), with the
    ctypes arguments built once so that mostly the C planner is timed."""
    import ctypes

    lib = nb.load()
    B = len(lens)
    arr = (ctypes.c_int32 * B)(*[int(x) for x in lens])
    cap = 8 * B + 64
    chunks = (nb.mla_chunk_t * cap)()
    indptr = (ctypes.c_int32 * (B + 1))()
    plan = nb.mla_plan_t()
    plan.capacity = cap
    plan.dtype = nb.DTYPE_CODES[DTYPE]
    plan.chunks = ctypes.cast(chunks, ctypes.POINTER(nb.mla_chunk_t))
    plan.o_indptr = ctypes.cast(indptr, ctypes.POINTER(ctypes.c_int32))
    pdev, pplan = ctypes.byref(dev), ctypes.byref(plan)
    per = []
    for _ in range(batches):
        t0 = time.perf_counter_ns()
        for _ in range(reps):
            if lib.mla_plan(arr, B, H, 1, BS, pdev, pplan) != nb.MLA_OK:
                raise RuntimeError("mla_plan failed")
        per.append((time.perf_counter_ns() - t0) / reps / 1e3)
    return statistics.median(per)


def algorithmic_bytes(L, n_chunks, latent_per_token=LATENT_BYTES_PER_TOKEN):
    """(partial kernel bytes, merge kernel bytes) one layer call must move."""
    pages = (L + BS - 1) // BS
    latent = L * latent_per_token
    table = pages * 4
    queries = H * 576 * 2
    partial_io = n_chunks * H * 513 * 4  # partials + lse written
    merge = n_chunks * H * 513 * 4 + H * 512 * 2  # read back, output written
    return latent + table + queries + partial_io, merge


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("partial_tc.cu", "partial_tc128.cu", "device_common.cuh", "kernels.h"):
        h.update(open(os.path.join(ROOT, "mla_split_kv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_name, tokens_per_launch):
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel."""
    try:
        prof = json.load(open(os.path.join(ROOT, "profiles", f"{kernel_name}_dram_traffic.json")))
    except (OSError, ValueError):
        return None
    if prof.get("kernel") != kernel_name or prof.get("kernel_source_hash") != kernel_source_hash():
        return None
    bpt = prof.get("dram_bytes_per_token")
    return None if bpt is None else round(bpt * tokens_per_launch)


def free_port():
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def replica_command(nprocs, script, script_args, port):
    """One process per GPU on this node: torch's launcher, rendezvous on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={nprocs}",
            "--master-addr=127.0.0.1", f"--master-port={port}", script, *script_args]


def launch_replicas(nprocs, script_args, script=None, stdout=None):
    """Run `script` (this file by default) as `nprocs` ranks and wait for them; returns the exit status.
    Each rank reads RANK / LOCAL_RANK / WORLD_SIZE from the environment the launcher sets."""
    cmd = replica_command(nprocs, script or os.path.abspath(__file__), list(script_args), free_port())
    return subprocess.run(cmd, stdout=stdout, text=True)


def init_ranks():
    """(rank, world, local rank) of this process. Under a launcher (WORLD_SIZE > 1) it binds the process to GPU
    LOCAL_RANK and joins the process group (NCCL on GPUs, gloo on a machine without them); the group carries
    only the barrier around the timed region and the max over ranks."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            torch.distributed.init_process_group("nccl")
        else:
            torch.distributed.init_process_group("gloo")
    return rank, world, local


def finish_ranks(world):
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


def max_over_ranks(value, device):
    """The largest of one float over all ranks (the job's time is its slowest rank's)."""
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(max_ms, calls_per_rank, world):
    """Whole-job figure: every rank replays the same calls (replicas), so the job did world x calls in the
    slowest rank's time."""
    return max_ms * 1e3 / (calls_per_rank * world)


def partial_kernel_name(kernel, plans):
    """The partial kernel the library dispatches for this workload (16 fp16 rows per CTA)."""
    if kernel == "simt":
        return "mla_partial_simt_kernel"
    if all(2 <= p.cluster_ctas <= 16 for p in plans):
        return "mla_partial_tc128_kernel"
    return "mla_partial_tc_kernel"


def run_profile_case(args):
    """A few plain layer calls at one context: the workload of the ncu captures in profiles/."""
    import torch

    from mla_split_kv_gb300 import binding as nb
    from mla_split_kv_gb300 import build as nbuild
    from mla_split_kv_gb300 import runtime as rt

    nbuild.build()
    nb.load()
    L = args.profile_ctx
    i = CONTEXTS.index(L) if L in CONTEXTS else 0
    case = make_case(i, L, args.profile_cache)
    dev = nb.mla_device_query()
    plan = nb.mla_plan([L], H, 1, BS, dev, dtype=args.profile_cache)
    num_partitions = 1
    if args.profile_split:  # the library's uniform split instead: P partitions on clusters of C CTAs, one each
        P, C = (int(x) for x in args.profile_split.split(","))
        plan = nb.Plan([(0, 0, 0, n) for n in range(P)], [0, P], C, nb.MLA_KERNEL_TC, 1)
        num_partitions = P
    kernel = {"tc": nb.MLA_KERNEL_TC, "simt": nb.MLA_KERNEL_SIMT}[args.kernel]
    dc = rt.upload(case)
    chunks_dev = rt.chunks_to_device(plan.chunks) if not args.profile_split else None
    part, lse = rt.alloc_partials(plan.num_chunks, 1, H)
    ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
    out = torch.empty((1, 1, H, 512), dtype=torch.float16, device="cuda")
    k = plan.clusters_per_chunk if kernel != nb.MLA_KERNEL_SIMT else 1
    ws = rt.alloc_decode_workspace(1, plan.num_chunks, k, plan.cluster_ctas, 1, H)
    if args.profile_layer:  # the layer call with its ends: cache write, decode, merge with the unembed
        import numpy as np

        from mla_split_kv_gb300 import inputs as gen

        rng = np.random.default_rng(SEED + 77)
        new_c = rt.to_device_16(gen.to_bits(rng.standard_normal((1, 1, 512)), "f16"), "f16", "cuda")
        new_k = rt.to_device_16(gen.to_bits(rng.standard_normal((1, 1, 64)), "f16"), "f16", "cuda")
        w = rt.to_device_16(gen.to_bits(rng.standard_normal((H, 512, 128)) / 512 ** 0.5, "f16"), "f16", "cuda")
        out_v = torch.empty((1, 1, H, 128), dtype=torch.float16, device="cuda")
    for _ in range(args.launches):  # the bench's layer call: mla_decode's default (partial kernel + entries merge)
        if args.profile_layer:
            nb.mla_cache_append(new_c.data_ptr(), new_k.data_ptr(), dc.block_table.data_ptr(),
                                dc.context_lens.data_ptr(), 1, 1, BS, case.num_blocks, case.max_blocks,
                                dc.ckv.data_ptr(), dc.kpe.data_ptr(), None)
            rt.decode_unembed(dc, part, lse, ind, w, out_v, num_partitions=num_partitions, kernel=kernel,
                              cluster=plan.cluster_ctas, chunks_dev=chunks_dev, subs=k, workspace=ws,
                              tables_ready=True, prefix_ready=True)
            continue
        rt.decode(dc, part, lse, ind, out, num_partitions=num_partitions, kernel=kernel, cluster=plan.cluster_ctas,
                  chunks_dev=chunks_dev, subs=k, workspace=ws, tables_ready=True, prefix_ready=True)
    torch.cuda.synchronize()
    st, code = nb.mla_check_device_errors(None)
    print(json.dumps({"profile_ctx": L, "cache": args.profile_cache, "launches": args.launches,
                      "layer_with_append_and_unembed": args.profile_layer, "partitions": plan.num_chunks,
                      "cluster": plan.cluster_ctas, "clusters_per_partition": k,
                      "kernel": partial_kernel_name(args.kernel, [plan]),
                      "device_status": st, "device_error": code}))
    if st != nb.MLA_OK:
        raise SystemExit(1)


def run_profile_verify(args):
    """A few plain verify-window calls of q_len args.profile_verify: the workload of the ncu capture of the
    window kernels' DRAM traffic in profiles/."""
    import torch

    from mla_split_kv_gb300 import binding as nb
    from mla_split_kv_gb300 import build as nbuild
    from mla_split_kv_gb300 import inputs as gen
    from mla_split_kv_gb300 import runtime as rt

    nbuild.build()
    nb.load()
    q = args.profile_verify
    full = gen.make_segmented_case(VW_SEED, B=VW_B, q_len=max(VW_QLENS), num_heads=H, block_size=BS)
    dc_base = rt.upload(full.base)
    stream = torch.cuda.current_stream()
    call, seg, nlaunch = verify_window_call(nb, rt, torch, stream, full, dc_base, q)
    for _ in range(args.launches):
        call()
    torch.cuda.synchronize()
    st, code = nb.mla_check_device_errors(None)
    flops, nbytes = window_work(seg)
    print(json.dumps({"profile": VERIFY, "q_len": q, "calls": args.launches, "partial_launches_per_call": nlaunch,
                      "algorithmic_bytes_per_call": nbytes, "algorithmic_flops_per_call": flops,
                      "partitions_per_segment": [p.num_chunks for p in call.plans],
                      "device_status": st, "device_error": code}))
    if st != nb.MLA_OK:
        raise SystemExit(1)


def run_profile_many_heads(args):
    import torch

    from mla_split_kv_gb300 import binding as nb
    from mla_split_kv_gb300 import build as nbuild
    from mla_split_kv_gb300 import runtime as rt

    nbuild.build()
    nb.load()
    call, plan, tokens = many_heads_call(nb, rt, torch, exchange={"exact": 0, "f16": 1, "none": 2, "f32": 3}[args.profile_exchange])
    for _ in range(args.launches):
        call()
    torch.cuda.synchronize()
    st, code = nb.mla_check_device_errors(None)
    print(json.dumps({"profile": MANY_HEADS, "launches": args.launches, "partitions": plan.num_chunks,
                      "cluster": plan.cluster_ctas, "tokens": tokens, "device_status": st, "device_error": code}))
    if st != nb.MLA_OK:
        raise SystemExit(1)


def time_many_heads(nb, rt, torch, stream, reps=20):
    """Device time of one many-head layer call (graph of `reps` calls, CUDA events), and its flop rate; beside
    it the same call with the partial scores exchanged as fp16 (an opt-in of the ABI)."""
    def timed(exchange, dtype="bf16"):
        with torch.cuda.stream(stream):
            call, plan, tokens = many_heads_call(nb, rt, torch, stream, exchange, dtype)
            for _ in range(3):
                call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                call()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            g.replay()
            e[0].record(stream)
            g.replay()
            e[1].record(stream)
        stream.synchronize()
        return e[0].elapsed_time(e[1]) * 1e3 / reps, plan, tokens

    us, plan, tokens = timed(0)  # the exact default: on 16-bit caches no partial scores cross the pair
    us16, _, _ = timed(1)
    us32, _, _ = timed(3)
    us8, _, _ = timed(0, "e4m3")
    flops = tokens * MH_H * 2 * (576 + 512)
    return {"workload": MANY_HEADS, "us_per_call": round(us, 3), "partitions": plan.num_chunks,
            "cluster": plan.cluster_ctas, "tokens": tokens, "tflops": round(flops / (us * 1e-6) / 1e12, 1),
            "hbm_gbs": round(tokens * LATENT_BYTES_PER_TOKEN / (us * 1e-6) / 1e9, 1),
            "fp32_exchange_us": round(us32, 3),
            "fp16_exchange_us": round(us16, 3),
            "fp16_exchange_tflops": round(flops / (us16 * 1e-6) / 1e12, 1),
            "e4m3_cache_us": round(us8, 3),
            "note": "a parity workload timed beside the headline one; repeats of one cache (323 MB, > L2); "
                    "us_per_call: the exact default (each CTA of a pair computes the full scores, nothing crosses "
                    "the pair); fp32_exchange: score_exchange = MLA_SCORE_EXCHANGE_F32 (half the columns a CTA, "
                    "fp32 partial scores exchanged); fp16_exchange: MLA_SCORE_EXCHANGE_F16; e4m3_cache: the same "
                    "lengths over an E4M3 cache (scale 1/4) beside fp16 queries"}


# the headline sweep with 8-bit E4M3 caches (576 bytes a token, power-of-two cache scale 1/4) beside fp16
# queries: the same contexts, seeds and pools, planned for E4M3 caches
E4M3_SWEEP = "mla_decode_ctx_sweep_B1_H16_e4m3_cache_fp16_q_bs32"
BF16_SWEEP = "mla_decode_ctx_sweep_B1_H16_r512_rope64_bf16_bs32"


def time_e4m3_sweep(nb, rt, torch, stream, dev, peak, reps=20, dtype="e4m3"):
    """The headline sweep on another cache type (E4M3 caches with fp16 queries, or bf16 throughout)."""
    calls, per_ctx = [], []
    with torch.cuda.stream(stream):
        for i, L in enumerate(CONTEXTS):
            case = make_case(i, L, dtype)
            plan = nb.mla_plan([L], H, 1, BS, dev, dtype=dtype)
            dc = rt.upload(case)
            chunks = rt.chunks_to_device(plan.chunks)
            part, lse = rt.alloc_partials(plan.num_chunks, 1, H)
            ws = rt.alloc_decode_workspace(1, plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, H)
            desc = rt.make_desc(dc, chunks, nb.MLA_KERNEL_TC, plan.cluster_ctas, stream, plan.clusters_per_chunk, ws,
                                tables_ready=True, prefix_ready=True)
            out = torch.empty((1, 1, H, 512), dtype=torch.bfloat16 if dtype == "bf16" else torch.float16,
                              device="cuda")
            ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
            calls.append(dict(L=L, plan=plan, dc=dc, part=part, lse=lse, ind=ind, out=out, desc=desc))
        for _ in range(3):
            for c in calls:
                rt.decode(c["dc"], c["part"], c["lse"], c["ind"], c["out"], desc=c["desc"])
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            rt.decode(c["dc"], c["part"], c["lse"], c["ind"], c["out"], desc=c["desc"])
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        g.replay()
        e[0].record(stream)
        for _ in range(reps):
            g.replay()
        e[1].record(stream)
    stream.synchronize()
    us = e[0].elapsed_time(e[1]) * 1e3 / (reps * len(calls))
    per_token = 576 if dtype == "e4m3" else LATENT_BYTES_PER_TOKEN
    nbytes = sum(sum(algorithmic_bytes(c["L"], c["plan"].num_chunks, per_token)) for c in calls) / len(calls)
    for c in calls:  # each context alone: a graph of four calls on its cache
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            for _ in range(4):
                rt.decode(c["dc"], c["part"], c["lse"], c["ind"], c["out"], desc=c["desc"])
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            g1.replay()
            e1[0].record(stream)
            g1.replay()
            e1[1].record(stream)
        stream.synchronize()
        per_ctx.append({"ctx": c["L"], "us_per_call": round(e1[0].elapsed_time(e1[1]) * 1e3 / 4, 3),
                        "partitions": c["plan"].num_chunks, "cluster": c["plan"].cluster_ctas,
                        "clusters_per_partition": c["plan"].clusters_per_chunk})
    achieved = nbytes / (us * 1e-6) / 1e9
    if dtype != "e4m3":
        return {"workload": BF16_SWEEP, "us_per_call": round(us, 3), "bytes_per_token": per_token,
                "achieved_gbs": round(achieved, 1), "frac": round(achieved / peak, 4), "per_ctx": per_ctx,
                "note": "timed like the headline step; the same seeds and pools drawn in bf16"}
    return {"workload": E4M3_SWEEP, "us_per_call": round(us, 3), "bytes_per_token": 576, "cache_scale": 0.25,
            "achieved_gbs": round(achieved, 1), "frac": round(achieved / peak, 4), "per_ctx": per_ctx,
            "note": "timed like the headline step (a graph of the six layer calls through mla_decode, tables and "
                    "first tiles read early); caches 354 MB in all, > L2"}


# the steps either side of attention: one new token written into its page (mla_cache_append), then the
# decode over the cache that now holds it with the W_UV^T unembed after it (mla_decode_unembed, v_head
# 128, fp16 weights); beside it the same through chunk partials (mla_decode_partial + mla_merge_unembed)
WRAP = "mla_layer_append_decode_unembed_B1_H16_fp16_bs32_vhead128"


def time_wrap(nb, rt, torch, stream, dev, reps=20):
    import numpy as np

    from mla_split_kv_gb300 import inputs as gen

    rows = []
    for i, L in ((0, CONTEXTS[0]), (len(CONTEXTS) - 1, CONTEXTS[-1])):
        case = make_case(i, L)
        rng = np.random.default_rng(SEED + 77)
        with torch.cuda.stream(stream):
            dc = rt.upload(case)
            new_c = rt.to_device_16(gen.to_bits(rng.standard_normal((1, 1, 512)), "f16"), "f16", "cuda")
            new_k = rt.to_device_16(gen.to_bits(rng.standard_normal((1, 1, 64)), "f16"), "f16", "cuda")
            w = rt.to_device_16(gen.to_bits(rng.standard_normal((H, 512, 128)) / 512 ** 0.5, "f16"), "f16", "cuda")
            plan = nb.mla_plan([L], H, 1, BS, dev, merge_path=nb.MLA_MERGE_PARTIALS)
            chunks = rt.chunks_to_device(plan.chunks)
            ind = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
            part, lse = rt.alloc_partials(plan.num_chunks, 1, H)
            ws = rt.alloc_workspace(plan.num_chunks, plan.clusters_per_chunk, plan.cluster_ctas, 1, H)
            desc = rt.make_desc(dc, chunks, nb.MLA_KERNEL_TC, plan.cluster_ctas, stream, plan.clusters_per_chunk, ws,
                                tables_ready=True)
            out = torch.empty((1, 1, H, 128), dtype=torch.float16, device="cuda")
            # the default plan: pair entries merged and unembedded by one dependent launch
            plan_d = nb.mla_plan([L], H, 1, BS, dev)
            chunks_d = rt.chunks_to_device(plan_d.chunks)
            ind_d = torch.tensor(plan_d.o_indptr, dtype=torch.int32, device="cuda")
            part_d, lse_d = rt.alloc_partials(plan_d.num_chunks, 1, H)
            ws_d = rt.alloc_decode_workspace(1, plan_d.num_chunks, plan_d.clusters_per_chunk, plan_d.cluster_ctas, 1, H)
            desc_d = rt.make_desc(dc, chunks_d, nb.MLA_KERNEL_TC, plan_d.cluster_ctas, stream,
                                  plan_d.clusters_per_chunk, ws_d, tables_ready=True, prefix_ready=True)
        s = stream.cuda_stream

        def append():
            nb.mla_cache_append(new_c.data_ptr(), new_k.data_ptr(), dc.block_table.data_ptr(),
                                dc.context_lens.data_ptr(), 1, 1, BS, case.num_blocks, case.max_blocks, dc.ckv.data_ptr(),
                                dc.kpe.data_ptr(), s)

        def unembed():
            nb.mla_merge_unembed(part.data_ptr(), lse.data_ptr(), ind.data_ptr(), 1, 1, H, w.data_ptr(), nb.MLA_F16,
                                 128, out.data_ptr(), nb.MLA_F16, None, s)

        def layer_partials():
            append()
            rt.decode_partial(dc, part, lse, desc=desc)
            unembed()

        def layer():
            append()
            rt.decode_unembed(dc, part_d, lse_d, ind_d, w, out, desc=desc_d)

        def timed(fn):
            with torch.cuda.stream(stream):
                for _ in range(3):
                    fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    fn()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            with torch.cuda.stream(stream):
                g.replay()
                e[0].record(stream)
                g.replay()
                e[1].record(stream)
            stream.synchronize()
            return e[0].elapsed_time(e[1]) * 1e3 / reps

        rows.append({"ctx": L, "us_per_call": round(timed(layer), 3),
                     "plan": [plan_d.num_chunks, plan_d.cluster_ctas, plan_d.clusters_per_chunk],
                     "us_per_call_chunk_partials": round(timed(layer_partials), 3),
                     "append_us": round(timed(append), 3), "merge_unembed_us": round(timed(unembed), 3),
                     "partials_plan": [plan.num_chunks, plan.cluster_ctas, plan.clusters_per_chunk]})
        del dc
    return {"workload": WRAP, "per_ctx": rows,
            "note": "us_per_call: mla_cache_append + mla_decode_unembed (the planner's default plan, pair entries "
                    "merged and unembedded by one dependent launch, prefix_ready); us_per_call_chunk_partials: "
                    "mla_cache_append + mla_decode_partial (a plan for chunk partials) + mla_merge_unembed; "
                    "append_us and merge_unembed_us: each call alone, repeated in a graph (latency-bound: one "
                    "token's 1152 bytes; 2 MB of W_UV^T and the partials)"}


def run_ours(args, rank, world):
    import numpy as np
    import torch

    from mla_split_kv_gb300 import binding as nb
    from mla_split_kv_gb300 import build as nbuild
    from mla_split_kv_gb300 import runtime as rt

    nbuild.build()
    nb.load()
    dev_index = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_index)
    kernel = {"tc": nb.MLA_KERNEL_TC, "simt": nb.MLA_KERNEL_SIMT}[args.kernel]

    cases = make_cases()
    dev = nb.mla_device_query()
    stream = torch.cuda.Stream()
    calls = []
    with torch.cuda.stream(stream):
        for case in cases:
            L = int(case.context_lens[0])
            dc = rt.upload(case)
            out = torch.empty((1, 1, H, 512), dtype=torch.float16, device="cuda")
            c = dict(L=L, dc=dc, out=out)
            # the timed step (mla_decode's default: pair entries merged by the entries kernel) and the paths
            # that merge chunk partials (mla_decode_partial + mla_merge_states, the single launch), each
            # planned for its merge
            for tag, mp in (("", nb.MLA_MERGE_ENTRIES), ("p", nb.MLA_MERGE_PARTIALS)):
                plan = nb.mla_plan([L], H, 1, BS, dev, merge_path=mp)
                chunks_dev = rt.chunks_to_device(plan.chunks)
                part, lse = rt.alloc_partials(plan.num_chunks, 1, H)
                k = plan.clusters_per_chunk if kernel != nb.MLA_KERNEL_SIMT else 1
                c[tag + "plan"] = plan
                c[tag + "chunks"] = chunks_dev
                c[tag + "part"], c[tag + "lse"] = part, lse
                c[tag + "ind"] = torch.tensor(plan.o_indptr, dtype=torch.int32, device="cuda")
                c[tag + "ws"] = rt.alloc_workspace(plan.num_chunks, k, plan.cluster_ctas, 1, H)
                c[tag + "dws"] = rt.alloc_decode_workspace(1, plan.num_chunks, k, plan.cluster_ctas, 1, H)
            # the tables are uploaded before the step and no kernel of the step writes them or the caches:
            # each call may read its tables and its first cache tiles while the kernel before it finishes
            for key, early in (("ldesc", True), ("ldesc0", False)):
                c[key] = rt.make_desc(dc, c["chunks"], kernel, c["plan"].cluster_ctas, stream,
                                      c["plan"].clusters_per_chunk if kernel != nb.MLA_KERNEL_SIMT else 1, c["dws"],
                                      tables_ready=True, prefix_ready=early)
            pk = c["pplan"].clusters_per_chunk if kernel != nb.MLA_KERNEL_SIMT else 1
            c["desc"] = rt.make_desc(dc, c["pchunks"], kernel, c["pplan"].cluster_ctas, stream, pk, c["pws"],
                                     tables_ready=True)
            c["sdesc"] = rt.make_desc(dc, c["pchunks"], kernel, c["pplan"].cluster_ctas, stream, pk, c["pdws"],
                                      tables_ready=True, decode_merge=nb.MLA_DECODE_MERGE_TICKETS)
            calls.append(c)
    torch.cuda.synchronize()

    def layer(c):  # one decode layer call through mla_decode (its default: partial kernel, then merge kernel)
        rt.decode(c["dc"], c["part"], c["lse"], c["ind"], c["out"], desc=c["ldesc"])

    def layer0(c):  # the same call with every cache read after the preceding kernel has finished
        rt.decode(c["dc"], c["part"], c["lse"], c["ind"], c["out"], desc=c["ldesc0"])

    def single(c):  # one launch that merges the chunk partials (their last CTAs merge)
        rt.decode(c["dc"], c["ppart"], c["plse"], c["pind"], c["out"], desc=c["sdesc"])

    def partial(c):  # the ABI's two calls: mla_decode_partial ...
        rt.decode_partial(c["dc"], c["ppart"], c["plse"], desc=c["desc"])

    def merge(c):  # ... and mla_merge_states
        rt.merge_states(c["ppart"], c["plse"], c["pind"], 1, 1, H, "f16", out=c["out"], stream=stream)

    # warm-up through the plain calls (also sets kernel attributes before capture)
    nb.mla_reset_counters()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            for c in calls:
                layer(c)
                layer0(c)
                partial(c)
                merge(c)
                single(c)
    stream.synchronize()
    st, code = nb.mla_check_device_errors(stream.cuda_stream)
    if st != nb.MLA_OK:
        raise RuntimeError(f"device error word {code:#x} after warm-up")

    # One CUDA graph per step (all six layer calls through mla_decode): `value`, and the roofline of
    # the layer call (its algorithmic bytes over its time in this graph). A graph of the six partial
    # launches of the two-launch ABI path (mla_decode_partial) alone, and a graph of the step with
    # single-launch calls, are reported beside it. Every graph sweeps the six disjoint caches, so
    # every launch streams its latent from HBM.
    g_step, g_part, g_two = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    g_late = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        for c in calls:
            layer(c)
    with torch.cuda.graph(g_late, stream=stream):
        for c in calls:
            layer0(c)
    with torch.cuda.graph(g_part, stream=stream):
        for c in calls:
            partial(c)
    with torch.cuda.graph(g_two, stream=stream):
        for c in calls:
            single(c)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g_step.replay()
            g_part.replay()
            g_two.replay()
            g_late.replay()
    stream.synchronize()

    K = args.steps
    # repeat the K-step loop so the timed region lasts long enough for the clock sampler
    probe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        probe[0].record(stream)
        g_step.replay()
        probe[1].record(stream)
    stream.synchronize()
    step_s = max(probe[0].elapsed_time(probe[1]) * 1e-3, 1e-6)
    reps = max(1, int(0.6 / (step_s * K)) + 1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev_index) as clocks:
        time.sleep(0.2)
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for _ in range(K * reps):
                g_step.replay()
            ev[1].record(stream)
            for _ in range(K * reps):
                g_part.replay()
            ev[2].record(stream)
        stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = ev[0].elapsed_time(ev[1]) / reps  # per K steps
    part_ms_all = ev[1].elapsed_time(ev[2]) / reps  # the ABI path's partial kernel alone
    if world > 1:
        total_ms = max_over_ranks(total_ms, "cuda")
    st, code = nb.mla_check_device_errors(stream.cuda_stream)
    if st != nb.MLA_OK:
        raise RuntimeError(f"device error word {code:#x} in the timed region")

    # the same step with single-launch layer calls (the merge inside the paired kernel), outside the
    # timed region, for comparison
    e2 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with torch.cuda.stream(stream):
        e2[0].record(stream)
        for _ in range(K):
            g_two.replay()
        e2[1].record(stream)
        for _ in range(K):
            g_late.replay()
        e2[2].record(stream)
    stream.synchronize()
    single_launch_us = e2[0].elapsed_time(e2[1]) * 1e3 / (K * len(calls))
    late_cache_us = e2[1].elapsed_time(e2[2]) * 1e3 / (K * len(calls))

    # per-context breakdown (not part of the timed region): one graph per call
    per_ctx = []
    kern_bytes_all = 0
    for c in calls:
        pb, mb = algorithmic_bytes(c["L"], c["plan"].num_chunks)
        kern_bytes_all += (pb + mb) * K
        g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            for _ in range(4):  # the other caches sit between repeats in the sweep; here each repeat re-reads
                layer(c)
        with torch.cuda.graph(g2, stream=stream):
            for _ in range(4):
                single(c)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        with torch.cuda.stream(stream):
            g1.replay()
            g2.replay()
            e[0].record(stream)
            g1.replay()
            e[1].record(stream)
            g2.replay()
            e[2].record(stream)
        stream.synchronize()
        us = e[0].elapsed_time(e[1]) * 1e3 / 4
        tus = e[1].elapsed_time(e[2]) * 1e3 / 4
        per_ctx.append({"ctx": c["L"], "partitions": c["plan"].num_chunks, "cluster": c["plan"].cluster_ctas,
                        "clusters_per_partition": c["ldesc"].clusters_per_chunk,
                        "partials_plan": [c["pplan"].num_chunks, c["pplan"].cluster_ctas, c["pplan"].clusters_per_chunk],
                        "us_per_call": round(us, 3), "single_launch_us": round(tus, 3),
                        "layer_gbs": round((pb + mb) / (us * 1e-6) / 1e9, 1),
                        "note": "repeats of one cache; caches <= 113 MB may be partly L2-resident"})

    # a single cold call per context: L2 flushed by writing 512 MB, then one un-graphed layer call
    # (host launch included), event-timed; median of three. And the host planner's time per call.
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for c, row in zip(calls, per_ctx):
        cold = []
        for t in range(3):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            with torch.cuda.stream(stream):
                flush.fill_(t + 1)
                e[0].record(stream)
                layer(c)
                e[1].record(stream)
            stream.synchronize()
            cold.append(e[0].elapsed_time(e[1]) * 1e3)
        row["cold_us"] = round(statistics.median(cold), 3)
        row["planner_host_us"] = round(planner_host_us(nb, [c["L"]], dev), 3)
    del flush
    # spread of the step time: five more trials of K graph replays each (outside the timed region)
    trial_us = []
    for _ in range(5):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            e[0].record(stream)
            for _ in range(K):
                g_step.replay()
            e[1].record(stream)
        stream.synchronize()
        trial_us.append(e[0].elapsed_time(e[1]) * 1e3 / (K * len(calls)))
    trials = {"n": 5, "median_us": round(statistics.median(trial_us), 3), "min_us": round(min(trial_us), 3),
              "max_us": round(max(trial_us), 3)}
    st, code = nb.mla_check_device_errors(stream.cuda_stream)
    if st != nb.MLA_OK:
        raise RuntimeError(f"device error word {code:#x} in the cold-call timing")

    # end to end through the C ABI with host buffers (pinned), every step: the inputs of the six calls
    # (queries, block tables, lengths, partition tables, merge offsets) sit in one pinned host buffer
    # that mirrors one device buffer, so a step uploads them with one copy; the six outputs come back
    # with one copy as well
    e2e_steps = max(1, args.e2e_steps)
    segs, off = [], 0

    def seg(arr):
        nonlocal off
        a = np.ascontiguousarray(arr)
        segs.append((off, a))
        off += (a.nbytes + 15) // 16 * 16  # every device input 16-byte aligned
        return len(segs) - 1

    layout = []
    for c in calls:
        cs = c["dc"].case
        layout.append(dict(q_abs=seg(cs.q_abs.view(np.int16)), q_pe=seg(cs.q_pe.view(np.int16)),
                           bt=seg(cs.block_table), lens=seg(cs.context_lens),
                           chunks=seg(c["plan"].chunk_array()),
                           ind=seg(np.asarray(c["plan"].o_indptr, dtype=np.int32))))
    hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
    hview = hbuf.numpy()
    for o, a in segs:
        hview[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
    dbuf = torch.empty(off, dtype=torch.uint8, device="cuda")

    def dview(i, dtype):
        o, a = segs[i]
        return dbuf[o:o + a.nbytes].view(dtype).view(a.shape)

    dout = torch.empty((len(calls), 1, 1, H, 512), dtype=torch.float16, device="cuda")
    hout = torch.empty(dout.shape, dtype=torch.float16).pin_memory()
    e2e_calls = []
    for j, (c, lay) in enumerate(zip(calls, layout)):
        dc = c["dc"]
        edc = rt.DeviceCase(q_abs=dview(lay["q_abs"], torch.int16).view(torch.float16),
                            q_pe=dview(lay["q_pe"], torch.int16).view(torch.float16),
                            ckv=dc.ckv, kpe=dc.kpe, block_table=dview(lay["bt"], torch.int32),
                            context_lens=dview(lay["lens"], torch.int32), case=dc.case)
        chunks = dview(lay["chunks"], torch.int32)
        desc = rt.make_desc(edc, chunks, kernel, c["plan"].cluster_ctas, stream, c["ldesc"].clusters_per_chunk,
                            c["dws"], tables_ready=True, prefix_ready=True)
        e2e_calls.append(dict(dc=edc, desc=desc, ind=dview(lay["ind"], torch.int32), out=dout[j],
                              part=c["part"], lse=c["lse"]))
    h2d = off
    d2h = dout.numel() * 2
    nb.mla_reset_counters()

    def e2e_step():
        with torch.cuda.stream(stream):
            dbuf.copy_(hbuf, non_blocking=True)
            for e in e2e_calls:
                rt.decode(e["dc"], e["part"], e["lse"], e["ind"], e["out"], desc=e["desc"])
            hout.copy_(dout, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_eager_s = time.perf_counter() - t0
    # the results of the last step are the graph's results (same inputs)
    for j, c in enumerate(calls):
        if not torch.equal(hout[j], c["out"].cpu()):
            raise RuntimeError(f"end-to-end output of call {j} differs from the timed graph's")
    ctr = nb.mla_get_counters()
    expect = (3 + e2e_steps) * len(calls)
    ctr_key = nb.CTR_PARTIAL_SIMT if kernel == nb.MLA_KERNEL_SIMT else nb.CTR_PARTIAL_TC
    # every layer call: one partial launch, and either the merge at the end of it or a merge launch
    if ctr[ctr_key] != expect or ctr[nb.CTR_MERGE] + ctr[nb.CTR_DECODE_FUSED] != expect:
        print(f"WARNING: path counters {ctr} disagree with {expect} layer calls on the {args.kernel} kernel",
              file=sys.stderr)
    launches_per_call = (ctr[ctr_key] + ctr[nb.CTR_MERGE]) / max(expect, 1)
    # the same step captured once through the same calls into a CUDA graph (the upload from the pinned
    # buffer, the six layer calls, the download), then replayed and waited for every step: how a decode
    # loop would run it; the copies still move every step's inputs and outputs
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        dbuf.copy_(hbuf, non_blocking=True)
        for e in e2e_calls:
            rt.decode(e["dc"], e["part"], e["lse"], e["ind"], e["out"], desc=e["desc"])
        hout.copy_(dout, non_blocking=True)
    # (outputs cleared on both sides first, so the check below sees what the replays computed)
    with torch.cuda.stream(stream):
        dout.zero_()
        hout.zero_()
        for _ in range(3):
            g_e2e.replay()
            stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            g_e2e.replay()
            stream.synchronize()
        e2e_s = time.perf_counter() - t0
    for j, c in enumerate(calls):
        if not torch.equal(hout[j], c["out"].cpu()):
            raise RuntimeError(f"graphed end-to-end output of call {j} differs from the timed graph's")

    many_heads = time_many_heads(nb, rt, torch, stream)
    st, code = nb.mla_check_device_errors(stream.cuda_stream)
    if st != nb.MLA_OK:
        raise RuntimeError(f"device error word {code:#x} in the many-head timing")
    peaks = measured_peaks()
    tpk = {"hbm_gbs": float(peaks["hbm_gbs"]), "tensor_tflops": float(peaks["bf16_tflops"]), "source": "measured"} \
        if peaks and peaks.get("hbm_gbs") and peaks.get("bf16_tflops") else \
        {"hbm_gbs": 6800.0, "tensor_tflops": 1900.0, "source": "fallback"}
    verify = time_verify_windows(nb, rt, torch, stream, tpk) if not args.skip_extra else None
    e4m3 = time_e4m3_sweep(nb, rt, torch, stream, dev, tpk["hbm_gbs"]) if not args.skip_extra else None
    bf16 = time_e4m3_sweep(nb, rt, torch, stream, dev, tpk["hbm_gbs"], dtype="bf16") if not args.skip_extra else None
    wrap = time_wrap(nb, rt, torch, stream, dev) if not args.skip_extra else None
    grid = time_batch_grid(nb, rt, torch, stream) if not args.skip_extra else None
    st, code = nb.mla_check_device_errors(stream.cuda_stream)
    if st != nb.MLA_OK:
        raise RuntimeError(f"device error word {code:#x} in the verify-window / batch-grid timing")

    n_calls = K * len(calls)
    value_us = job_us_per_call(total_ms, n_calls, world)
    achieved = kern_bytes_all / (total_ms * 1e-3) / 1e9  # whole layer calls in the timed region
    peaks = measured_peaks()
    if peaks and peaks.get("hbm_gbs"):
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        peak, peak_src = 6800.0, "fallback"
    kname = partial_kernel_name(args.kernel, [c["plan"] for c in calls])
    part_bytes = sum(algorithmic_bytes(c["L"], c["pplan"].num_chunks)[0] for c in calls) * K
    partial_only = {"kernel": kname + " (mla_decode_partial: in-cluster combine, normalized partials)",
                    "us_per_launch": round(part_ms_all * 1e3 / (K * len(calls)), 3),
                    "achieved_gbs": round(part_bytes / (part_ms_all * 1e-3) / 1e9, 1),
                    "frac": round(part_bytes / (part_ms_all * 1e-3) / 1e9 / peak, 4)}
    result = {
        "metric": METRIC,
        "value": round(value_us, 3),
        "unit": "us/layer-call",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "contexts": CONTEXTS, "B": 1, "H": H, "kv_lora_rank": 512, "rope_dim": 64,
                   "block_size": BS, "partitions": "planner", "kernel": args.kernel,
                   "launches_per_layer_call": round(launches_per_call, 3),
                   "l2": "inputs larger than L2: each step streams six disjoint caches, 528 MB",
                   "timing": "CUDA graph per step (6 layer calls through mla_decode), CUDA events on the launching "
                             "stream; the roofline over the same graph"},
        "per_ctx": per_ctx,
        "trials": trials,
        "single_launch_us": round(single_launch_us, 3),
        "without_prefix_ready_us": round(late_cache_us, 3),
        "many_heads": many_heads,
        "verify_windows": verify,
        "batch_grid": grid,
        "e4m3_caches": e4m3,
        "bf16": bf16,
        "layer_with_append_and_unembed": wrap,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(kname, sum(CONTEXTS) / len(CONTEXTS)),
                     "peak_source": peak_src,
                     "kernel": kname + " (with its dependent mla_merge_entries_kernel: the whole layer call)",
                     "bytes": "latent + block table + queries + partials and LSE written and read back + output",
                     "time": "the timed step graph: every launch of both kernels and the gaps between them"},
        "partial_kernel_alone": partial_only,
        "e2e": {"value": round(e2e_s * 1e6 / (e2e_steps * len(calls)), 3), "unit": "us/layer-call",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "eager_us": round(e2e_eager_s * 1e6 / (e2e_steps * len(calls)), 3),
                "how": "host wall clock per step: the pinned upload, the six mla_decode calls and the download, "
                       "replayed from one CUDA graph captured through those calls, then a stream synchronize; "
                       "eager_us: the same calls launched one by one every step"},
        # the step graphs (launches_per_call each layer call) and the partial-only graphs (one each)
        "gpu_launches": int(round((launches_per_call + 1) * n_calls * reps)),
        "timed_repeats": reps,
        "clocks": clocks.summary(),
    }
    return result, cases


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cases = make_cases()
    cores = os.cpu_count() or 1
    per_call, steps = oracle_timing(cases, max(1, args.steps), cores, budget_s=90.0)
    us = statistics.mean(per_call) * 1e6
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(us, 1),
        "unit": "us/layer-call",
        "n_gpus": world,
        "steps": steps,
        "warmup": 1,
        "ms_per_step": round(us * len(CONTEXTS) / 1e3, 3),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "contexts": CONTEXTS, "B": 1, "H": H, "block_size": BS},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/layer-call", "cores": cores, "kind": "oracle",
                         "sample": f"{steps} sweep(s) of the six contexts, all 16 heads, f64 numpy oracle, "
                                   f"{cores} spawned single-threaded workers (heads split across them)"},
        "e2e": {"value": round(us, 1), "unit": "us/layer-call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.profile_ctx:
        run_profile_case(args)
        return
    if args.profile_many_heads:
        run_profile_many_heads(args)
        return
    if args.profile_verify:
        run_profile_verify(args)
        return
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # no launcher around this process: start one rank per GPU (this file again, same arguments)
        raise SystemExit(launch_replicas(args.gpus, sys.argv[1:]).returncode)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} does not match the launcher's WORLD_SIZE {world}")
    if args.impl == "reference":
        res = run_reference(args, int(os.environ.get("RANK", "0")), world)
        if res is not None:
            print(json.dumps(res))
        return
    rank, world, _ = init_ranks()
    res, cases = run_ours(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        per_call, steps = oracle_timing(cases, 1, cores, budget_s=30.0)
        res["cpu_baseline"] = {"value": round(statistics.mean(per_call) * 1e6, 1), "unit": "us/layer-call",
                               "cores": cores, "kind": "oracle",
                               "sample": f"{steps} sweep of the six contexts (one layer call each, all 16 heads), "
                                         f"f64 numpy oracle in {cores} spawned single-threaded workers"}
    finish_ranks(world)
    if rank == 0:
        assert res["n_gpus"] == args.gpus
        print(json.dumps(res))


if __name__ == "__main__":
    main()
