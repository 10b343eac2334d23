"""The exchange format of context parallelism, on CPU ranks (gloo, world size 2).

One long request's pages split into contiguous, block-aligned spans, one per
rank; every rank computes the partials of the partitions of its span, the
ranks all-gather their (partial, log2 LSE) pairs, and the LSE merge of the
gathered set is the attention over the whole context ("[kernel] Wire MLA
split-KV decode", *What changed*: the reduce combines slices by their LSE so
the result equals ordinary attention; merge associativity across regroupings,
mlxcel PR #995). Not built on GPUs (every run here has one GPU); this pins the
format a multi-GPU version would exchange, with the oracle on both sides.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
L, H, BS, SEED, PARTS_PER_RANK = 2100, 16, 32, 21, 2


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
        from mla_split_kv_gb300 import inputs as gen
        from oracle import mla_oracle as orc

        case = gen.make_decode_case(SEED, [L], num_heads=H, block_size=BS, dtype="f16")
        # this rank's span of the context, then its partitions inside the span (block-aligned)
        s0, s1 = orc.chunk_bounds(L, world, BS)[rank]
        local = [(0, s0 + a, s0 + b) for (a, b) in orc.chunk_bounds(s1 - s0, PARTS_PER_RANK, BS)]
        part, lse = orc.partials(case, local)
        # the exchange: every rank gathers every rank's (partial, lse) in rank order
        pt, lt = torch.from_numpy(np.ascontiguousarray(part)), torch.from_numpy(np.ascontiguousarray(lse))
        parts = [torch.zeros_like(pt) for _ in range(world)]
        lses = [torch.zeros_like(lt) for _ in range(world)]
        dist.all_gather(parts, pt)
        dist.all_gather(lses, lt)
        allp = torch.cat(parts).numpy()
        alll = torch.cat(lses).numpy()
        merged, merged_lse = orc.merge(allp, alll, [0, allp.shape[0]])
        ref, ref_lse = orc.unsplit(case)
        out[rank] = (float(np.max(np.abs(merged - ref))), float(np.max(np.abs(merged_lse - ref_lse))),
                     allp.shape[0], (s0, s1))
    finally:
        dist.destroy_process_group()


def test_spans_on_two_ranks_gather_and_merge_to_the_whole_context():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    spans = sorted(out[r][3] for r in range(world))
    assert spans[0][0] == 0 and spans[-1][1] == L and spans[0][1] == spans[1][0] and spans[0][1] % BS == 0
    for r in range(world):
        err, err_lse, n, _ = out[r]
        assert n == world * PARTS_PER_RANK
        assert err < 1e-12 and err_lse < 1e-12, (r, err, err_lse)
