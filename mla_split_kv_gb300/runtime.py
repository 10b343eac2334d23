"""Device buffers and one decode layer call through the C ABI.

torch supplies device memory and streams; the binding passes raw pointers;
all computation happens in the CUDA library.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

from . import binding as nb
from .inputs import DecodeCase

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


def to_device_16(bits: np.ndarray, dtype: str, device) -> torch.Tensor:
    """uint16 bit patterns -> a 16-bit float tensor on `device` (bit-exact)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DTYPE[dtype])


@dataclasses.dataclass
class DeviceCase:
    q_abs: torch.Tensor
    q_pe: torch.Tensor
    ckv: torch.Tensor
    kpe: torch.Tensor
    block_table: torch.Tensor
    context_lens: torch.Tensor
    case: DecodeCase


def to_device_cache(bits: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Cache patterns -> device: 16-bit floats (bit-exact), or E4M3 bytes as uint8."""
    if dtype == "e4m3":
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).to(device)
    return to_device_16(bits, dtype, device)


def query_dtype(dtype: str) -> str:
    """The queries' 16-bit type beside a cache of `dtype`: fp16 beside E4M3."""
    return "f16" if dtype == "e4m3" else dtype


def upload(case: DecodeCase, device="cuda", ckv: torch.Tensor = None, kpe: torch.Tensor = None) -> DeviceCase:
    """Copy a case to the device. A resident cache (ckv/kpe) can be shared."""
    qdt = query_dtype(case.dtype)
    return DeviceCase(
        q_abs=to_device_16(case.q_abs, qdt, device),
        q_pe=to_device_16(case.q_pe, qdt, device),
        ckv=ckv if ckv is not None else to_device_cache(case.ckv, case.dtype, device),
        kpe=kpe if kpe is not None else to_device_cache(case.kpe, case.dtype, device),
        block_table=torch.from_numpy(np.ascontiguousarray(case.block_table)).to(device),
        context_lens=torch.from_numpy(np.ascontiguousarray(case.context_lens)).to(device),
        case=case,
    )


def chunks_to_device(chunks: Sequence[Sequence[int]], device="cuda") -> torch.Tensor:
    arr = np.asarray(chunks, dtype=np.int32).reshape(-1, 4)
    return torch.from_numpy(arr).to(device)


def make_desc(dc: DeviceCase, chunks_dev: Optional[torch.Tensor], kernel: int, cluster: int,
              stream: Optional[torch.cuda.Stream] = None, subs: int = 1,
              workspace: Optional[torch.Tensor] = None, tables_ready: bool = False,
              decode_merge: int = 0, prefix_ready: bool = False,
              score_exchange: int = 0) -> nb.mla_decode_desc_t:
    c = dc.case
    d = nb.mla_decode_desc_t()
    d.num_requests = c.num_requests
    d.num_heads = c.num_heads
    d.q_len = c.q_len
    d.block_size = c.block_size
    d.num_blocks = int(dc.ckv.shape[0])
    d.max_blocks_per_req = int(dc.block_table.shape[1])
    d.dtype = nb.DTYPE_CODES[c.dtype]
    d.causal = 1 if c.causal else 0
    d.chunks = chunks_dev.data_ptr() if chunks_dev is not None else None
    d.num_chunks = int(chunks_dev.shape[0]) if chunks_dev is not None else 0
    d.cluster_ctas = cluster
    d.kernel = kernel
    s = stream if stream is not None else torch.cuda.current_stream()
    d.stream = s.cuda_stream
    d.clusters_per_chunk = subs
    d.workspace = workspace.data_ptr() if workspace is not None else None
    d.workspace_bytes = workspace.numel() if workspace is not None else 0
    d.tables_ready = 1 if tables_ready else 0
    d.decode_merge = decode_merge
    d.prefix_ready = 1 if prefix_ready else 0
    d.cache_scale = float(c.cache_scale)
    d.score_exchange = score_exchange
    # the descriptor holds raw device pointers: keep their tensors alive as long as it lives
    d._keep = (chunks_dev, workspace)
    return d


def alloc_workspace(num_chunks: int, subs: int, cluster: int, q_len: int, H: int,
                    device="cuda") -> Optional[torch.Tensor]:
    """Zeroed workspace for partitions spread over `subs` clusters of `cluster` CTAs (None when subs <= 1)."""
    n = nb.mla_workspace_bytes(num_chunks, subs, cluster, q_len, H)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def alloc_decode_workspace(B: int, num_chunks: int, subs: int, cluster: int, q_len: int, H: int,
                           device="cuda") -> torch.Tensor:
    """Zeroed workspace of mla_decode on the paired kernel (request tickets and LSE copies of its single-launch
    way, then the chunk tickets and the pair entries)."""
    n = nb.mla_decode_workspace_bytes(B, num_chunks, subs, cluster, q_len, H)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode(dc: DeviceCase, part: torch.Tensor, lse: torch.Tensor, o_indptr_dev: torch.Tensor, out: torch.Tensor,
           out_lse: Optional[torch.Tensor] = None, num_partitions: int = 1, desc: Optional[nb.mla_decode_desc_t] = None,
           **desc_kw) -> torch.Tensor:
    """One decode layer call through mla_decode (its ways on the paired kernel chosen by decode_merge)."""
    d = desc if desc is not None else make_desc(dc, desc_kw.get("chunks_dev"), desc_kw.get("kernel", nb.MLA_KERNEL_AUTO),
                                                desc_kw.get("cluster", 0), desc_kw.get("stream"),
                                                desc_kw.get("subs", 1), desc_kw.get("workspace"),
                                                desc_kw.get("tables_ready", False), desc_kw.get("decode_merge", 0),
                                                desc_kw.get("prefix_ready", False),
                                                desc_kw.get("score_exchange", 0))
    out_code = {torch.float32: nb.MLA_F32, torch.float16: nb.MLA_F16, torch.bfloat16: nb.MLA_BF16}[out.dtype]
    nb.mla_decode(dc.q_abs.data_ptr(), dc.q_pe.data_ptr(), dc.ckv.data_ptr(), dc.kpe.data_ptr(),
                  dc.block_table.data_ptr(), dc.context_lens.data_ptr(), float(dc.case.scale), num_partitions,
                  part.data_ptr(), lse.data_ptr(), o_indptr_dev.data_ptr(), out.data_ptr(), out_code,
                  out_lse.data_ptr() if out_lse is not None else None, d)
    return out


def decode_unembed(dc: DeviceCase, part: torch.Tensor, lse: torch.Tensor, o_indptr_dev: torch.Tensor,
                   w_uv_t: torch.Tensor, out_v: torch.Tensor, out_lse: Optional[torch.Tensor] = None,
                   num_partitions: int = 1, desc: Optional[nb.mla_decode_desc_t] = None, **desc_kw) -> torch.Tensor:
    """One decode layer call through mla_decode_unembed: attention, then W_UV^T [H, 512, v_head] per head."""
    d = desc if desc is not None else make_desc(dc, desc_kw.get("chunks_dev"), desc_kw.get("kernel", nb.MLA_KERNEL_AUTO),
                                                desc_kw.get("cluster", 0), desc_kw.get("stream"),
                                                desc_kw.get("subs", 1), desc_kw.get("workspace"),
                                                desc_kw.get("tables_ready", False), desc_kw.get("decode_merge", 0),
                                                desc_kw.get("prefix_ready", False),
                                                desc_kw.get("score_exchange", 0))
    codes = {torch.float32: nb.MLA_F32, torch.float16: nb.MLA_F16, torch.bfloat16: nb.MLA_BF16}
    nb.mla_decode_unembed(dc.q_abs.data_ptr(), dc.q_pe.data_ptr(), dc.ckv.data_ptr(), dc.kpe.data_ptr(),
                          dc.block_table.data_ptr(), dc.context_lens.data_ptr(), float(dc.case.scale), num_partitions,
                          part.data_ptr(), lse.data_ptr(), o_indptr_dev.data_ptr(), w_uv_t.data_ptr(),
                          codes[w_uv_t.dtype], int(w_uv_t.shape[-1]), out_v.data_ptr(), codes[out_v.dtype],
                          out_lse.data_ptr() if out_lse is not None else None, d)
    return out_v


def alloc_partials(num_slots: int, q_len: int, H: int, device="cuda"):
    part = torch.empty((num_slots, q_len, H, 512), dtype=torch.float32, device=device)
    lse = torch.empty((num_slots, q_len, H), dtype=torch.float32, device=device)
    return part, lse


def decode_partial(dc: DeviceCase, part: torch.Tensor, lse: torch.Tensor, num_partitions: int = 1,
                   chunks_dev: Optional[torch.Tensor] = None, kernel: int = nb.MLA_KERNEL_AUTO,
                   cluster: int = 0, stream=None, desc: Optional[nb.mla_decode_desc_t] = None, subs: int = 1,
                   workspace: Optional[torch.Tensor] = None, tables_ready: bool = False,
                   score_exchange: int = 0) -> None:
    d = desc if desc is not None else make_desc(dc, chunks_dev, kernel, cluster, stream, subs, workspace,
                                                tables_ready, score_exchange=score_exchange)
    nb.mla_decode_partial(dc.q_abs.data_ptr(), dc.q_pe.data_ptr(), dc.ckv.data_ptr(), dc.kpe.data_ptr(),
                          dc.block_table.data_ptr(), dc.context_lens.data_ptr(), float(dc.case.scale),
                          num_partitions, part.data_ptr(), lse.data_ptr(), d)


def merge_states(part: torch.Tensor, lse: torch.Tensor, o_indptr_dev: torch.Tensor, B: int, q_len: int, H: int,
                 out_dtype: str = "f32", out: Optional[torch.Tensor] = None, out_lse: Optional[torch.Tensor] = None,
                 stream=None):
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[out_dtype]
    if out is None:
        out = torch.empty((B, q_len, H, 512), dtype=tdt, device=part.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    nb.mla_merge_states(part.data_ptr(), lse.data_ptr(), o_indptr_dev.data_ptr(), B, q_len, H, out.data_ptr(),
                        nb.DTYPE_CODES[out_dtype], out_lse.data_ptr() if out_lse is not None else None,
                        s.cuda_stream)
    return out


def uniform_indptr(B: int, P: int, device="cuda") -> torch.Tensor:
    return torch.arange(0, (B + 1) * P, P, dtype=torch.int32, device=device)


@dataclasses.dataclass
class SegmentPlan:
    """Partitions of a verify window over a segmented prefix: each segment planned on its own,
    chunk slots request-major over all segments, so one merge of o_indptr combines them."""
    chunk_tables: list       # per segment, device int32 [n, 4] {b, t0, t1, slot}
    plans: list              # per segment, the planner's Plan
    o_indptr: torch.Tensor   # device [B+1]
    num_slots: int


def plan_segments(seg, dev: nb.mla_device_info_t, max_partitions: int = 0, device="cuda") -> SegmentPlan:
    segs = seg.segments
    B = segs[0].num_requests
    plans = [nb.mla_plan(s.context_lens.tolist(), s.num_heads, s.q_len, s.block_size, dev,
                         max_partitions=max_partitions, dtype=s.dtype) for s in segs]
    # request b's slots: its chunks of segment 0, then of segment 1, ...
    per = [[p.o_indptr[b + 1] - p.o_indptr[b] for b in range(B)] for p in plans]
    indptr = [0]
    for b in range(B):
        indptr.append(indptr[-1] + sum(per[k][b] for k in range(len(segs))))
    tables = []
    for k, p in enumerate(plans):
        rows = []
        for b in range(B):
            base = indptr[b] + sum(per[j][b] for j in range(k))
            for i, (cb, t0, t1, _) in enumerate(p.chunks[p.o_indptr[b]:p.o_indptr[b + 1]]):
                rows.append((cb, t0, t1, base + i))
        tables.append(chunks_to_device(rows, device))
    return SegmentPlan(chunk_tables=tables, plans=plans,
                       o_indptr=torch.tensor(indptr, dtype=torch.int32, device=device), num_slots=indptr[-1])
