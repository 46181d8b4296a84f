"""Python binding of libkvp (paged-KV-cache decode for GB300, sm_103a).

Thin marshalling over the C ABI in ``include/kvp.h``: every function here has
the C entry point's name, turns torch tensors into pointers and sizes, passes
torch's current CUDA stream, and raises :class:`KvpError` on a non-OK status.
All computation happens in the library's CUDA kernels; there is no fallback.
If ``_lib/libkvp.so`` has not been built, the first call raises
``RuntimeError`` (build it with ``__graft_entry__.build()`` or
``python -m pagedattention_decode_kvp_gb300._build``).

Block manager: :class:`BlockManager` wraps the host allocator (``kvp_bm_*``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libkvp.so")

KVP_OK = 0
KVP_ERR_INVALID_ARG = 1
KVP_ERR_UNSUPPORTED = 2
KVP_ERR_CUDA = 3
KVP_ERR_BAD_BLOCK = 4
KVP_ERR_TIMEOUT = 5
KVP_ERR_OOM = 6
KVP_ERR_REFCOUNT = 7
KVP_ERR_NOT_FOUND = 8
KVP_ERR_SCRATCH_LIMIT = 9
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
KVP_F16 = 0
KVP_BF16 = 1
KVP_PHASE_PARTIAL = 1
KVP_PHASE_REDUCE = 2
KVP_PHASE_ALL = 3
KVP_DECODE_MERGE_RUNS = 8  # or'ed into `phases`: one copy per run of consecutive blocks
BLOCK_SIZE = 16


class kvp_cache_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class kvp_bm_stats_t(ctypes.Structure):
    _fields_ = [("total_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32),
                ("free_blocks", ctypes.c_int32), ("active_requests", ctypes.c_int32),
                ("block_refs", ctypes.c_int64), ("utilization", ctypes.c_double),
                ("bytes_per_block", ctypes.c_int64), ("total_memory_gb", ctypes.c_double)]


class KvpError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        super().__init__(f"{where}: {kvp_status_string(status)} ({status})")


# (name, restype, argtypes) of every exported symbol
_P, _I32, _I64, _SZ, _F = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                            ctypes.c_float)
_D = kvp_cache_desc
SIGNATURES = {
    "kvp_status_string": (ctypes.c_char_p, [_I32]),
    "kvp_version": (_I32, []),
    "kvp_append": (_I32, [_P, _P, _P, _P, _P, _I32, _D, _I32, _P, _P]),
    "kvp_append_int8": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _I32, _D, _P, _P]),
    "kvp_append_int8_fixed": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _F, _F, _P, _I32, _D, _P,
                                     _P]),
    "kvp_append_fp8": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _I32, _D, _P, _P]),
    "kvp_copy_blocks": (_I32, [_P, _P, _P, _P, _I32, _P, _I32, _D, _P, _P]),
    "kvp_decode_partition_blocks": (_I32, [_I32, _I32, _D, _I32, _I32]),
    "kvp_decode_workspace_bytes": (_SZ, [_I32, _I32, _D, _I32, _I32, _I32]),
    "kvp_attention_decode": (_I32, [_P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _F, _D, _I32, _I32,
                                    _P, _SZ, _I32, _P, _P]),
    "kvp_append_attention_decode": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _F,
                                           _D, _I32, _I32, _P, _SZ, _I32, _P, _P]),
    "kvp_attention_decode_int8": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32,
                                         _F, _D, _I32, _P, _SZ, _I32, _P, _P]),
    "kvp_attention_decode_fp8": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32,
                                        _F, _D, _I32, _P, _SZ, _I32, _P, _P]),
    "kvp_attention_decode_noalloc": (_I32, [_P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _F, _D,
                                            _I32, _I32, _P, _P]),
    "kvp_attention_prefill": (_I32, [_P, _P, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                     _I32, _F, _D, _I32, _P, _P]),
    "kvp_decode_shared_prefix_workspace_bytes": (_SZ, [_I32, _I32, _D, _I32, _I32, _I32]),
    "kvp_attention_decode_shared_prefix": (_I32, [_P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _F,
                                                  _D, _I32, _I32, _I32, _P, _SZ, _P, _P]),
    "kvp_read_status": (_I32, [_P, _P]),
    "kvp_selftest_wait_timeout": (_I32, [_P, _I64, _P]),
    "kvp_bm_create": (_P, [_I32, _I32, _I64]),
    "kvp_bm_destroy": (None, [_P]),
    "kvp_bm_allocate": (_I32, [_P, _I64, _I32, _I32]),
    "kvp_bm_share_prefix": (_I32, [_P, _I64, _I64, _I32]),
    "kvp_bm_append_slot": (_I32, [_P, _I64, _P, _P, _P]),
    "kvp_bm_free": (_I32, [_P, _I64]),
    "kvp_bm_release_block": (_I32, [_P, _I64, _I32]),
    "kvp_bm_block_table": (_I32, [_P, _I64, _P, _I32]),
    "kvp_bm_num_tokens": (_I32, [_P, _I64]),
    "kvp_bm_ref_count": (_I32, [_P, _I32]),
    "kvp_bm_stats": (None, [_P, ctypes.POINTER(kvp_bm_stats_t)]),
}

_lock = threading.Lock()
_lib = None


def load_library():
    """Load libkvp.so (once).  Raises RuntimeError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libkvp.so is not built ({LIB_PATH}); run __graft_entry__.build() or "
                "python -m pagedattention_decode_kvp_gb300._build")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def kvp_status_string(status: int) -> str:
    try:
        return load_library().kvp_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def kvp_version() -> int:
    return load_library().kvp_version()


# ------------------------------------------------------------------ marshalling
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return KVP_F16
    if t.dtype == torch.bfloat16:
        return KVP_BF16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors passed to the GPU entry points must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("tensors passed to the GPU entry points must be contiguous")


def cache_desc(k_cache) -> kvp_cache_desc:
    """kvp_cache_desc of a pool tensor [NB, Hkv, block_size, D]."""
    if k_cache.dim() != 4:
        raise ValueError("cache pools are [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = (int(x) for x in k_cache.shape)
    return kvp_cache_desc(nb, hkv, bs, d)


def _check(status: int, where: str) -> None:
    if status != KVP_OK:
        raise KvpError(status, where)


# ------------------------------------------------------------------ GPU entry points
def kvp_append(key, value, k_cache, v_cache, slot_mapping, *, status=None, stream=None) -> None:
    """Scatter key/value [T, Hkv, D] into the fp16/bf16 pools at slot_mapping [T] int32."""
    lib = load_library()
    _need_cuda(key, value, k_cache, v_cache, slot_mapping, status)
    if key.dtype != k_cache.dtype or value.dtype != v_cache.dtype:
        raise TypeError("key/value must have the pool's dtype")
    T = int(slot_mapping.numel())
    _check(lib.kvp_append(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                          _ptr(slot_mapping), T, cache_desc(k_cache), _dtype_code(k_cache),
                          _ptr(status), _stream_ptr(stream)), "kvp_append")


def kvp_append_int8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, *,
                    status=None, stream=None) -> None:
    """Quantise key/value [T, Hkv, D] (fp16/bf16) per token and head and scatter
    codes into the int8 pools and scales into k_scale/v_scale [NB, Hkv, bs]."""
    lib = load_library()
    _need_cuda(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, status)
    T = int(slot_mapping.numel())
    _check(lib.kvp_append_int8(_ptr(key), _ptr(value), _dtype_code(key), _ptr(k_cache),
                               _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping),
                               T, cache_desc(k_cache), _ptr(status), _stream_ptr(stream)),
           "kvp_append_int8")


def kvp_append_int8_fixed(key, value, k_cache, v_cache, k_scale_pool, v_scale_pool, k_scale,
                          v_scale, slot_mapping, *, status=None, stream=None) -> None:
    """Per-tensor INT8: quantise key/value with the given scales (also written to
    the scale pools at each slot) and scatter the codes."""
    lib = load_library()
    _need_cuda(key, value, k_cache, v_cache, k_scale_pool, v_scale_pool, slot_mapping, status)
    T = int(slot_mapping.numel())
    _check(lib.kvp_append_int8_fixed(_ptr(key), _ptr(value), _dtype_code(key), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(k_scale_pool), _ptr(v_scale_pool),
                                     float(k_scale), float(v_scale), _ptr(slot_mapping), T,
                                     cache_desc(k_cache), _ptr(status), _stream_ptr(stream)),
           "kvp_append_int8_fixed")


def kvp_append_fp8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, *,
                   status=None, stream=None) -> None:
    """Quantise key/value [T, Hkv, D] to FP8 E4M3 per token and head (uint8 or
    float8_e4m3fn pools) with float32 scales [NB, Hkv, bs], then scatter."""
    lib = load_library()
    _need_cuda(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, status)
    T = int(slot_mapping.numel())
    _check(lib.kvp_append_fp8(_ptr(key), _ptr(value), _dtype_code(key), _ptr(k_cache),
                              _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping),
                              T, cache_desc(k_cache), _ptr(status), _stream_ptr(stream)),
           "kvp_append_fp8")


def kvp_copy_blocks(k_cache, v_cache, pairs, *, k_scale=None, v_scale=None, status=None,
                    stream=None) -> None:
    """Copy block pairs[i, 0] onto pairs[i, 1] in both pools (and scale pools)."""
    lib = load_library()
    _need_cuda(k_cache, v_cache, pairs, k_scale, v_scale, status)
    P = int(pairs.shape[0]) if pairs.dim() == 2 else int(pairs.numel()) // 2
    _check(lib.kvp_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                               k_cache.element_size(), _ptr(pairs), P, cache_desc(k_cache),
                               _ptr(status), _stream_ptr(stream)), "kvp_copy_blocks")


def _kv_8bit(kv_int8, kv_fp8):
    return 2 if kv_fp8 else (1 if kv_int8 else 0)


def kvp_decode_partition_blocks(batch, num_q_heads, desc: kvp_cache_desc, max_blocks,
                                kv_int8=False, kv_fp8=False) -> int:
    """kv_int8 / kv_fp8: the pools hold INT8 / FP8 codes (their decodes are
    shaped differently)."""
    return load_library().kvp_decode_partition_blocks(int(batch), int(num_q_heads), desc,
                                                      int(max_blocks), _kv_8bit(kv_int8, kv_fp8))


def kvp_decode_workspace_bytes(batch, num_q_heads, desc: kvp_cache_desc, max_blocks,
                               partition_blocks=0, kv_int8=False, kv_fp8=False) -> int:
    return int(load_library().kvp_decode_workspace_bytes(int(batch), int(num_q_heads), desc,
                                                         int(max_blocks), int(partition_blocks),
                                                         _kv_8bit(kv_int8, kv_fp8)))


def kvp_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, *,
                         workspace=None, partition_blocks=0, phases=KVP_PHASE_ALL, status=None,
                         stream=None) -> None:
    """out[B, Hq, D] = paged decode attention of q[B, Hq, D] over fp16/bf16 pools."""
    lib = load_library()
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, workspace, status)
    if q.dtype != k_cache.dtype or out.dtype != q.dtype:
        raise TypeError("q, out and the pools must share one dtype")
    B, Hq, _ = (int(x) for x in q.shape)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.kvp_attention_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens), B, Hq, float(scale), cache_desc(k_cache),
        _dtype_code(q), int(partition_blocks), _ptr(workspace), ws_bytes, int(phases),
        _ptr(status), _stream_ptr(stream)), "kvp_attention_decode")


def kvp_decode_shared_prefix_workspace_bytes(batch, num_q_heads, desc: kvp_cache_desc, max_blocks,
                                             shared_prefix_blocks, partition_blocks=0) -> int:
    return int(load_library().kvp_decode_shared_prefix_workspace_bytes(
        int(batch), int(num_q_heads), desc, int(max_blocks), int(shared_prefix_blocks),
        int(partition_blocks)))


def kvp_attention_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens,
                                       scale, shared_prefix_blocks, *, workspace,
                                       partition_blocks=0, status=None, stream=None) -> None:
    """kvp_attention_decode for requests whose first shared_prefix_blocks table
    entries name the same physical blocks (the prefix part runs once per kv
    head for all requests)."""
    lib = load_library()
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, workspace, status)
    if q.dtype != k_cache.dtype or out.dtype != q.dtype:
        raise TypeError("q, out and the pools must share one dtype")
    B, Hq, _ = (int(x) for x in q.shape)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.kvp_attention_decode_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens), B, Hq, float(scale), cache_desc(k_cache),
        _dtype_code(q), int(shared_prefix_blocks), int(partition_blocks), _ptr(workspace),
        ws_bytes, _ptr(status), _stream_ptr(stream)), "kvp_attention_decode_shared_prefix")


def kvp_append_attention_decode(key, value, out, q, k_cache, v_cache, block_tables, context_lens,
                                scale, *, workspace=None, partition_blocks=0,
                                phases=KVP_PHASE_ALL, status=None, stream=None) -> None:
    """One fused decode step over fp16/bf16 pools: request b's new token
    key/value[b] ([B, Hkv, D]) is written at position context_lens[b] - 1, then
    out = paged decode attention of q."""
    lib = load_library()
    _need_cuda(key, value, out, q, k_cache, v_cache, block_tables, context_lens, workspace,
               status)
    if q.dtype != k_cache.dtype or out.dtype != q.dtype or key.dtype != k_cache.dtype:
        raise TypeError("key, value, q, out and the pools must share one dtype")
    B, Hq, _ = (int(x) for x in q.shape)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.kvp_append_attention_decode(
        _ptr(key), _ptr(value), _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), B, Hq, float(scale),
        cache_desc(k_cache), _dtype_code(q), int(partition_blocks), _ptr(workspace), ws_bytes,
        int(phases), _ptr(status), _stream_ptr(stream)), "kvp_append_attention_decode")


def kvp_attention_decode_int8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                              context_lens, scale, *, workspace=None, partition_blocks=0,
                              phases=KVP_PHASE_ALL, status=None, stream=None) -> None:
    """As kvp_attention_decode over int8 pools with float32 scales [NB, Hkv, bs]."""
    lib = load_library()
    _need_cuda(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, workspace,
               status)
    if out.dtype != q.dtype:
        raise TypeError("out must have q's dtype")
    B, Hq, _ = (int(x) for x in q.shape)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.kvp_attention_decode_int8(
        _ptr(out), _ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), B, Hq,
        float(scale), cache_desc(k_cache), int(partition_blocks), _ptr(workspace), ws_bytes,
        int(phases), _ptr(status), _stream_ptr(stream)), "kvp_attention_decode_int8")


def kvp_attention_decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                             context_lens, scale, *, workspace=None, partition_blocks=0,
                             phases=KVP_PHASE_ALL, status=None, stream=None) -> None:
    """As kvp_attention_decode over FP8 (E4M3) pools with float32 scales."""
    lib = load_library()
    _need_cuda(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, workspace,
               status)
    if out.dtype != q.dtype:
        raise TypeError("out must have q's dtype")
    B, Hq, _ = (int(x) for x in q.shape)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.kvp_attention_decode_fp8(
        _ptr(out), _ptr(q), _dtype_code(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), B, Hq,
        float(scale), cache_desc(k_cache), int(partition_blocks), _ptr(workspace), ws_bytes,
        int(phases), _ptr(status), _stream_ptr(stream)), "kvp_attention_decode_fp8")


def kvp_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale, *,
                                 partition_blocks=0, status=None, stream=None) -> None:
    """kvp_attention_decode without a workspace argument, for callers that cannot
    allocate device memory: the library's built-in scratch array
    (NOALLOC_SCRATCH_BYTES per GPU) holds the split-context partials.  Calls that
    overlap on the GPU share that array and race; serialise them."""
    lib = load_library()
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, status)
    if q.dtype != k_cache.dtype or out.dtype != q.dtype:
        raise TypeError("q, out and the pools must share one dtype")
    B, Hq, _ = (int(x) for x in q.shape)
    _check(lib.kvp_attention_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens), B, Hq, float(scale), cache_desc(k_cache),
        _dtype_code(q), int(partition_blocks), _ptr(status), _stream_ptr(stream)),
        "kvp_attention_decode_noalloc")


def kvp_attention_prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                          max_query_len, scale, *, shared_prefix_blocks=0, status=None,
                          stream=None) -> None:
    """out[T, Hq, D] = causal multi-query paged attention of q[T, Hq, D] over
    fp16/bf16 pools; request b's rows are q[query_start[b]:query_start[b+1]]
    and sit at the last positions of its context_lens[b] cached tokens.
    shared_prefix_blocks > 0: the first that many table entries of every
    request are the same physical blocks (packs all rows into dense tiles)."""
    lib = load_library()
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, query_start, status)
    if q.dtype != k_cache.dtype or out.dtype != q.dtype:
        raise TypeError("q, out and the pools must share one dtype")
    T, Hq, _ = (int(x) for x in q.shape)
    if int(out.shape[0]) < T:
        raise ValueError("out needs as many rows as q")
    B = int(context_lens.shape[0])
    _check(lib.kvp_attention_prefill(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens), _ptr(query_start), T, B, Hq,
        int(max_query_len), int(shared_prefix_blocks), float(scale), cache_desc(k_cache),
        _dtype_code(q), _ptr(status), _stream_ptr(stream)), "kvp_attention_prefill")


def kvp_selftest_wait_timeout(status, limit_ns, stream=None):
    """Run the library's bounded mbarrier wait on a barrier nothing arrives
    on, giving up after limit_ns: it records KVP_ERR_TIMEOUT in `status`."""
    _need_cuda(status)
    _check(load_library().kvp_selftest_wait_timeout(_ptr(status), int(limit_ns),
                                                     _stream_ptr(stream)),
           "kvp_selftest_wait_timeout")


def kvp_read_status(status, stream=None) -> int:
    """Synchronise the stream and return the device status word's kvp_status."""
    return int(load_library().kvp_read_status(_ptr(status), _stream_ptr(stream)))


# ------------------------------------------------------------------ block manager
class BlockManager:
    """Host block allocator (kvp_bm_*): free pool, block tables, reference
    counts and copy-on-write decisions."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE, bytes_per_block: int = 0):
        self._lib = load_library()
        self._h = self._lib.kvp_bm_create(int(num_blocks), int(block_size), int(bytes_per_block))
        if not self._h:
            raise KvpError(KVP_ERR_INVALID_ARG, "kvp_bm_create")
        self.block_size = int(block_size)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.kvp_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def allocate(self, req: int, num_tokens: int, reserve_blocks: int = 0) -> None:
        _check(self._lib.kvp_bm_allocate(self._h, int(req), int(num_tokens), int(reserve_blocks)),
               "kvp_bm_allocate")

    def share_prefix(self, src: int, dst: int, num_tokens: int) -> None:
        _check(self._lib.kvp_bm_share_prefix(self._h, int(src), int(dst), int(num_tokens)),
               "kvp_bm_share_prefix")

    def append_slot(self, req: int):
        """Returns (slot, cow_src, cow_dst); cow_* are -1 when no copy is needed."""
        slot, cs, cd = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.kvp_bm_append_slot(self._h, int(req), ctypes.byref(slot),
                                            ctypes.byref(cs), ctypes.byref(cd)),
               "kvp_bm_append_slot")
        return slot.value, cs.value, cd.value

    def free(self, req: int) -> None:
        _check(self._lib.kvp_bm_free(self._h, int(req)), "kvp_bm_free")

    def release_block(self, req: int, block: int) -> None:
        _check(self._lib.kvp_bm_release_block(self._h, int(req), int(block)),
               "kvp_bm_release_block")

    def block_table(self, req: int) -> list:
        n = self._lib.kvp_bm_block_table(self._h, int(req), None, 0)
        if n < 0:
            raise KvpError(KVP_ERR_NOT_FOUND, "kvp_bm_block_table")
        buf = (ctypes.c_int32 * max(n, 1))()
        self._lib.kvp_bm_block_table(self._h, int(req), buf, n)
        return list(buf[:n])

    def num_tokens(self, req: int) -> int:
        return self._lib.kvp_bm_num_tokens(self._h, int(req))

    def ref_count(self, block: int) -> int:
        return self._lib.kvp_bm_ref_count(self._h, int(block))

    def stats(self) -> dict:
        s = kvp_bm_stats_t()
        self._lib.kvp_bm_stats(self._h, ctypes.byref(s))
        return {f: getattr(s, f) for f, _ in s._fields_}
