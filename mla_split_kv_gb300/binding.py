"""Thin ctypes binding of the C ABI in ``include/mla_split_kv.h``.

Argument marshalling only: every step of the decode runs in the CUDA library.
The function names match the C entry points. Device buffers are passed as raw
pointers (``tensor.data_ptr()``), streams as ``cudaStream_t`` handles
(``torch.cuda.current_stream().cuda_stream``). Loading fails loudly when the
library has not been built; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmla_split_kv.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_CUDA = 3
MLA_ERR_TIMEOUT = 4
MLA_ERR_DEVICE_CHECK = 5
MLA_ERR_CAPACITY = 6

MLA_F16, MLA_BF16, MLA_F32, MLA_E4M3 = 0, 1, 2, 3
MLA_MAX_Q_LEN = 32  # rows of a verify window per request, at most
MLA_STATIC_WORKSPACE_BYTES = 4 * 1024 * 1024
MLA_KERNEL_AUTO, MLA_KERNEL_SIMT, MLA_KERNEL_TC = 0, 1, 2
MLA_MERGE_ENTRIES, MLA_MERGE_PARTIALS = 0, 1
MLA_DECODE_MERGE_ENTRIES, MLA_DECODE_MERGE_TICKETS = 0, 1
MLA_SCORE_EXCHANGE_EXACT, MLA_SCORE_EXCHANGE_F16, MLA_SCORE_EXCHANGE_NONE, MLA_SCORE_EXCHANGE_F32 = 0, 1, 2, 3

CTR_PARTIAL_SIMT, CTR_PARTIAL_TC, CTR_MERGE, CTR_REJECTED, CTR_CTAS, CTR_DECODE_FUSED, CTR_WRAP = range(7)
NUM_COUNTERS = 7

DTYPE_CODES = {"f16": MLA_F16, "bf16": MLA_BF16, "f32": MLA_F32, "e4m3": MLA_E4M3}


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({status_string(status)})")
        self.status = status


class mla_chunk_t(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int32), ("t0", ctypes.c_int32), ("t1", ctypes.c_int32), ("out_slot", ctypes.c_int32)]


class mla_device_info_t(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("max_clusters", ctypes.c_int32 * 5)]


class mla_plan_t(ctypes.Structure):
    _fields_ = [
        ("max_partitions", ctypes.c_int32),
        ("min_partitions", ctypes.c_int32),
        ("split_min_tokens", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("chunks", ctypes.POINTER(mla_chunk_t)),
        ("o_indptr", ctypes.POINTER(ctypes.c_int32)),
        ("merge_path", ctypes.c_int32),
        ("num_chunks", ctypes.c_int32),
        ("cluster_ctas", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("clusters_per_chunk", ctypes.c_int32),
    ]


class mla_decode_desc_t(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_req", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("chunks", ctypes.c_void_p),
        ("num_chunks", ctypes.c_int32),
        ("cluster_ctas", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("stream", ctypes.c_void_p),
        ("clusters_per_chunk", ctypes.c_int32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_uint64),
        ("tables_ready", ctypes.c_int32),
        ("decode_merge", ctypes.c_int32),
        ("prefix_ready", ctypes.c_int32),
        ("cache_scale", ctypes.c_float),
        ("score_exchange", ctypes.c_int32),
    ]


_lib = None


def load() -> ctypes.CDLL:
    """Load the built library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("MLA_SPLIT_KV_LIB", LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run mla_split_kv_gb300.build.build())")
    lib = ctypes.CDLL(path)
    i32, u64, vp, f32 = ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_float
    lib.mla_device_query.argtypes = [i32, ctypes.POINTER(mla_device_info_t)]
    lib.mla_device_query.restype = i32
    lib.mla_plan.argtypes = [ctypes.POINTER(i32), i32, i32, i32, i32, ctypes.POINTER(mla_device_info_t),
                             ctypes.POINTER(mla_plan_t)]
    lib.mla_plan.restype = i32
    lib.mla_decode_partial.argtypes = [vp, vp, vp, vp, vp, vp, f32, i32, vp, vp, ctypes.POINTER(mla_decode_desc_t)]
    lib.mla_decode_partial.restype = i32
    lib.mla_decode_partial_static.argtypes = [vp, vp, vp, vp, vp, vp, f32, i32, vp, vp,
                                              ctypes.POINTER(mla_decode_desc_t)]
    lib.mla_decode_partial_static.restype = i32
    lib.mla_decode.argtypes = [vp, vp, vp, vp, vp, vp, f32, i32, vp, vp, vp, vp, i32, vp,
                               ctypes.POINTER(mla_decode_desc_t)]
    lib.mla_decode.restype = i32
    lib.mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.mla_decode_workspace_bytes.restype = u64
    lib.mla_cache_append.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.mla_cache_append.restype = i32
    lib.mla_merge_unembed.argtypes = [vp, vp, vp, i32, i32, i32, vp, i32, i32, vp, i32, vp, vp]
    lib.mla_merge_unembed.restype = i32
    lib.mla_decode_unembed.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, i32, vp, vp, vp, vp, i32, i32, vp, i32,
                                       vp, ctypes.POINTER(mla_decode_desc_t)]
    lib.mla_decode_unembed.restype = i32
    lib.mla_merge_states.argtypes = [vp, vp, vp, i32, i32, i32, vp, i32, vp, vp]
    lib.mla_merge_states.restype = i32
    lib.mla_check_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.mla_check_device_errors.restype = i32
    lib.mla_selfcheck.argtypes = [ctypes.POINTER(f32)]
    lib.mla_selfcheck.restype = i32
    lib.mla_get_counters.argtypes = [ctypes.POINTER(u64), i32]
    lib.mla_get_counters.restype = None
    lib.mla_reset_counters.argtypes = []
    lib.mla_reset_counters.restype = None
    lib.mla_set_wait_timeout_ns.argtypes = [u64]
    lib.mla_set_wait_timeout_ns.restype = None
    lib.mla_partials_bytes.argtypes = [i32, i32, i32]
    lib.mla_partials_bytes.restype = ctypes.c_size_t
    lib.mla_lse_bytes.argtypes = [i32, i32, i32]
    lib.mla_lse_bytes.restype = ctypes.c_size_t
    lib.mla_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.mla_workspace_bytes.restype = u64
    lib.mla_status_string.argtypes = [i32]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_version.argtypes = []
    lib.mla_version.restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().mla_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status != MLA_OK:
        raise MlaError(status, where)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------


def mla_device_query(device: int = -1) -> mla_device_info_t:
    info = mla_device_info_t()
    _check(load().mla_device_query(device, ctypes.byref(info)), "mla_device_query")
    return info


class Plan:
    """Host result of :func:`mla_plan`."""

    def __init__(self, chunks, o_indptr, cluster_ctas, kernel, clusters_per_chunk=1):
        self.chunks = chunks  # list of (b, t0, t1, out_slot)
        self.o_indptr = o_indptr  # list of B+1 ints
        self.cluster_ctas = cluster_ctas
        self.kernel = kernel
        self.clusters_per_chunk = clusters_per_chunk

    @property
    def num_chunks(self) -> int:
        return len(self.chunks)

    def parts(self):
        return [self.o_indptr[b + 1] - self.o_indptr[b] for b in range(len(self.o_indptr) - 1)]

    def chunk_array(self):
        import numpy as np
        return np.asarray(self.chunks, dtype=np.int32).reshape(-1, 4)


def mla_plan(context_lens: Sequence[int], num_heads: int, q_len: int, block_size: int,
             dev: mla_device_info_t, max_partitions: int = 0, min_partitions: int = 0,
             split_min_tokens: int = 0, dtype: str = "f16", merge_path: int = MLA_MERGE_ENTRIES) -> Plan:
    lib = load()
    B = len(context_lens)
    lens = (ctypes.c_int32 * B)(*[int(x) for x in context_lens])
    plan = mla_plan_t()
    plan.max_partitions = max_partitions
    plan.min_partitions = min_partitions
    plan.split_min_tokens = split_min_tokens
    plan.dtype = DTYPE_CODES[dtype]
    plan.merge_path = merge_path
    plan.capacity = 0
    st = lib.mla_plan(lens, B, num_heads, q_len, block_size, ctypes.byref(dev), ctypes.byref(plan))
    if st not in (MLA_OK, MLA_ERR_CAPACITY):
        raise MlaError(st, "mla_plan")
    cap = max(1, plan.num_chunks)
    chunks = (mla_chunk_t * cap)()
    indptr = (ctypes.c_int32 * (B + 1))()
    plan.capacity = cap
    plan.chunks = ctypes.cast(chunks, ctypes.POINTER(mla_chunk_t))
    plan.o_indptr = ctypes.cast(indptr, ctypes.POINTER(ctypes.c_int32))
    _check(lib.mla_plan(lens, B, num_heads, q_len, block_size, ctypes.byref(dev), ctypes.byref(plan)), "mla_plan")
    out = [(c.b, c.t0, c.t1, c.out_slot) for c in chunks[: plan.num_chunks]]
    return Plan(out, list(indptr), plan.cluster_ctas, plan.kernel, plan.clusters_per_chunk)


def mla_decode_partial(q_absorbed: int, q_pe: int, ckv_cache: int, kpe_cache: int, block_table: int,
                       context_lens: int, scale: float, num_partitions: int, partials: int, lse: int,
                       desc: mla_decode_desc_t) -> None:
    _check(load().mla_decode_partial(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens,
                                     ctypes.c_float(scale), num_partitions, partials, lse, ctypes.byref(desc)),
           "mla_decode_partial")


def mla_decode_partial_static(q_absorbed: int, q_pe: int, ckv_cache: int, kpe_cache: int, block_table: int,
                              context_lens: int, scale: float, num_partitions: int, partials: int, lse: int,
                              desc: mla_decode_desc_t) -> None:
    _check(load().mla_decode_partial_static(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens,
                                            ctypes.c_float(scale), num_partitions, partials, lse, ctypes.byref(desc)),
           "mla_decode_partial_static")


def mla_decode(q_absorbed: int, q_pe: int, ckv_cache: int, kpe_cache: int, block_table: int, context_lens: int,
               scale: float, num_partitions: int, partials: int, lse: int, o_indptr: int, out: int, out_dtype: int,
               out_lse: Optional[int], desc: mla_decode_desc_t) -> None:
    _check(load().mla_decode(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens, ctypes.c_float(scale),
                             num_partitions, partials, lse, o_indptr, out, out_dtype, out_lse or None,
                             ctypes.byref(desc)), "mla_decode")


def mla_decode_unembed(q_absorbed: int, q_pe: int, ckv_cache: int, kpe_cache: int, block_table: int,
                       context_lens: int, scale: float, num_partitions: int, partials: int, lse: int, o_indptr: int,
                       w_uv_t: int, w_dtype: int, v_head: int, out_v: int, out_dtype: int, out_lse: Optional[int],
                       desc: mla_decode_desc_t) -> None:
    _check(load().mla_decode_unembed(q_absorbed, q_pe, ckv_cache, kpe_cache, block_table, context_lens,
                                     ctypes.c_float(scale), num_partitions, partials, lse, o_indptr, w_uv_t, w_dtype,
                                     v_head, out_v, out_dtype, out_lse or None, ctypes.byref(desc)),
           "mla_decode_unembed")


def mla_decode_workspace_bytes(num_requests: int, num_chunks: int, clusters_per_chunk: int, cluster_ctas: int,
                               q_len: int, num_heads: int) -> int:
    return int(load().mla_decode_workspace_bytes(num_requests, num_chunks, clusters_per_chunk, cluster_ctas, q_len,
                                                 num_heads))


def mla_merge_states(partials: int, lse: int, o_indptr: int, B: int, q_len: int, num_heads: int, out: int,
                     out_dtype: int, out_lse: Optional[int], stream: Optional[int]) -> None:
    _check(load().mla_merge_states(partials, lse, o_indptr, B, q_len, num_heads, out, out_dtype,
                                   out_lse or None, stream or None), "mla_merge_states")


def mla_cache_append(ckv_new: int, kpe_new: int, block_table: int, context_lens: int, B: int, q_len: int,
                     block_size: int, num_blocks: int, max_blocks_per_req: int, ckv_cache: int, kpe_cache: int,
                     stream: Optional[int]) -> None:
    _check(load().mla_cache_append(ckv_new, kpe_new, block_table, context_lens, B, q_len, block_size, num_blocks,
                                   max_blocks_per_req, ckv_cache, kpe_cache, stream or None), "mla_cache_append")


def mla_merge_unembed(partials: int, lse: int, o_indptr: int, B: int, q_len: int, num_heads: int, w_uv_t: int,
                      w_dtype: int, v_head: int, out: int, out_dtype: int, out_lse: Optional[int],
                      stream: Optional[int]) -> None:
    _check(load().mla_merge_unembed(partials, lse, o_indptr, B, q_len, num_heads, w_uv_t, w_dtype, v_head, out,
                                    out_dtype, out_lse or None, stream or None), "mla_merge_unembed")


def mla_check_device_errors(stream: Optional[int] = None):
    """Synchronize and read/clear the device error word; returns (status, word)."""
    code = ctypes.c_uint32(0)
    return load().mla_check_device_errors(stream or None, ctypes.byref(code)), code.value


def mla_selfcheck():
    """Run the library's closed-form decode check on the current device; returns (status, max-abs error)."""
    err = ctypes.c_float(0.0)
    return load().mla_selfcheck(ctypes.byref(err)), err.value


def mla_get_counters():
    arr = (ctypes.c_uint64 * NUM_COUNTERS)()
    load().mla_get_counters(arr, NUM_COUNTERS)
    return list(arr)


def mla_reset_counters() -> None:
    load().mla_reset_counters()


def mla_set_wait_timeout_ns(ns: int) -> None:
    load().mla_set_wait_timeout_ns(ns)


def mla_workspace_bytes(num_chunks: int, clusters_per_chunk: int, cluster_ctas: int, q_len: int, num_heads: int) -> int:
    return int(load().mla_workspace_bytes(num_chunks, clusters_per_chunk, cluster_ctas, q_len, num_heads))


def mla_partials_bytes(num_slots: int, q_len: int, num_heads: int) -> int:
    return load().mla_partials_bytes(num_slots, q_len, num_heads)


def mla_version() -> int:
    return load().mla_version()
