"""CPU oracle for the paged-KV-cache decode path -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``kvp_oracle.c`` (plain C, IEEE double; the INT8
quantiser in float32 as its listing fixes).  This module compiles it with gcc
and exposes numpy-level wrappers.  It shares no code with the CUDA library in
``pagedattention_decode_kvp_gb300`` and neither imports the other.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may load it; the product path never does.

Pages cited (title, section):
  * "ATB KV Cache management" -- "Paged KV Cache": 16-token blocks.
  * "KV Cache 优化与显存管理" -- 二: PagedAttention, GQA head groups, INT8;
    三: KVCacheQuantizer (per-channel abs-max / 127, round, clip).
  * "ATB PagedAttention" -- "ATB 的 PagedAttention 实现": page = pos / size,
    offset = pos % size; "PagedAttention 的 Attention 计算修改": score, exp,
    weight V; "踩坑三": copy-on-write copies a whole page.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
library routines, closed forms and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvp_oracle.so")

F16, BF16, I8, E4M3 = 0, 1, 2, 3
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kvp_oracle.c into a shared library (gcc, OpenMP if available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-frounding-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f64.restype = ctypes.c_double
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        lib.orc_num_threads.restype = I
        lib.orc_set_num_threads.argtypes = [I]
        lib.orc_attention_decode.argtypes = [P, P, I, P, I, P, P, I, P, P, P, I, P,
                                             I, I, I, I, I, I, ctypes.c_double]
        lib.orc_attention_decode.restype = I
        lib.orc_append.argtypes = [P, P, P, I, I, I, I, I, I]
        lib.orc_append.restype = I
        lib.orc_copy_blocks.argtypes = [P, P, I, ctypes.c_size_t, I]
        lib.orc_copy_blocks.restype = I
        lib.orc_quantize_int8.argtypes = [P, I, ctypes.c_longlong, I, P, P]
        lib.orc_quantize_int8.restype = None
        lib.orc_attention_prefill.argtypes = [P, P, I, P, I, P, P, I, P, I, P, P, I, I, I, I, I,
                                              I, ctypes.c_double]
        lib.orc_attention_prefill.restype = I
        lib.orc_quantize_int8_fixed.argtypes = [P, I, ctypes.c_longlong, ctypes.c_float, P]
        lib.orc_quantize_int8_fixed.restype = None
        lib.orc_quantize_fp8.argtypes = [P, I, ctypes.c_longlong, I, P, P]
        lib.orc_quantize_fp8.restype = None
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_to_f64.restype = ctypes.c_double
        lib.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
        _lib = lib
        return lib


# ---------------------------------------------------------------- marshalling
def _raw(x):
    """(contiguous numpy array of raw storage, kind) for torch or numpy input."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.float16:
                return x.view(torch.int16).numpy().view(np.uint16), F16
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.int8:
                return x.numpy(), I8
            if x.dtype == torch.float8_e4m3fn:
                return x.view(torch.uint8).numpy(), E4M3
            if x.dtype == torch.uint8:          # E4M3 bit patterns
                return x.numpy(), E4M3
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16), F16
    if x.dtype == np.int8:
        return x, I8
    if x.dtype == np.uint8:                     # E4M3 bit patterns
        return x, E4M3
    raise TypeError(f"unsupported element type {x.dtype}")


def _i32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _f32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


# ---------------------------------------------------------------- public API
def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def f16_to_f64(bits: int) -> float:
    return _load().orc_f16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return _load().orc_bf16_to_f64(int(bits))


def e4m3_to_f64(code: int) -> float:
    return _load().orc_e4m3_to_f64(int(code))


def f32_to_e4m3(x: float) -> int:
    return int(_load().orc_f32_to_e4m3(float(x)))


def attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                     *, k_scale=None, v_scale=None, rows=None):
    """softmax(q K^T * scale) V through block tables, in float64.

    q [B, Hq, D] f16/bf16; k_cache/v_cache [NB, Hkv, bs, D] f16/bf16/int8 (int8
    needs k_scale/v_scale [NB, Hkv, bs] float32); block_tables [B, MB] int32;
    context_lens [B].  rows: optional [(b, h), ...] to compute only those.
    Returns float64 [B, Hq, D], or [len(rows), D] when rows is given.
    """
    lib = _load()
    qa, qk = _raw(q)
    ka, kk = _raw(k_cache)
    va, vk = _raw(v_cache)
    if kk != vk:
        raise TypeError("k_cache and v_cache element types differ")
    B, Hq, D = qa.shape
    NB, Hkv, bs, D2 = ka.shape
    if D2 != D or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    bt = _i32(block_tables)
    cl = _i32(context_lens).reshape(-1)
    if bt.ndim != 2 or bt.shape[0] != B or cl.shape[0] != B:
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    quant = kk in (I8, E4M3)
    ks = _f32(k_scale) if quant else None
    vs = _f32(v_scale) if quant else None
    if quant and (ks is None or vs is None):
        raise ValueError("int8 / fp8 pools need k_scale and v_scale")
    if rows is None:
        ra, n_rows = None, B * Hq
        out = np.zeros((B, Hq, D), dtype=np.float64)
    else:
        ra = _i32(rows).reshape(-1, 2)
        n_rows = ra.shape[0]
        out = np.zeros((n_rows, D), dtype=np.float64)
    err = lib.orc_attention_decode(_ptr(out), _ptr(ra), n_rows, _ptr(qa), qk,
                                   _ptr(ka), _ptr(va), kk, _ptr(ks), _ptr(vs),
                                   _ptr(bt), bt.shape[1], _ptr(cl), B, Hq, Hkv, D, NB,
                                   bs, float(scale))
    if err != 0:
        raise ValueError(f"oracle attention_decode: bad block table or length ({err})")
    return out


def attention_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                      *, rows=None):
    """Causal multi-query paged attention in float64.  q [T, Hq, D] holds each
    request's chunk of queries (rows query_start[b] .. query_start[b+1]-1), the
    chunk being the last tokens of the request's context_lens[b]; query i of a
    chunk of length L attends to positions 0 .. n - L + i.  Returns float64
    [T, Hq, D] (or [len(rows), D] for the given (row, head) pairs)."""
    lib = _load()
    qa, qk = _raw(q)
    ka, kk = _raw(k_cache)
    va, _ = _raw(v_cache)
    T, Hq, D = qa.shape
    NB, Hkv, bs, _ = ka.shape
    bt = _i32(block_tables)
    cl = _i32(context_lens).reshape(-1)
    qs = _i32(query_start).reshape(-1)
    B = cl.shape[0]
    if qs.shape[0] != B + 1 or bt.shape[0] != B:
        raise ValueError("query_start must be [B+1], block_tables [B, MB]")
    if rows is None:
        ra = np.array([(t, h) for t in range(T) for h in range(Hq)], dtype=np.int32)
        out = np.zeros((T * Hq, D), dtype=np.float64)
    else:
        ra = _i32(rows).reshape(-1, 2)
        out = np.zeros((ra.shape[0], D), dtype=np.float64)
    err = lib.orc_attention_prefill(_ptr(out), _ptr(ra), ra.shape[0], _ptr(qa), qk, _ptr(ka),
                                    _ptr(va), kk, _ptr(bt), bt.shape[1], _ptr(cl), _ptr(qs), B, Hq,
                                    Hkv, D, NB, bs, float(scale))
    if err != 0:
        raise ValueError(f"oracle attention_prefill: bad table or lengths ({err})")
    return out.reshape(T, Hq, D) if rows is None else out


def _like(result, template):
    """Hand raw bytes back as a torch tensor of the template's dtype when the
    caller passed torch tensors (numpy otherwise)."""
    try:
        import torch
        if isinstance(template, torch.Tensor):
            t = torch.from_numpy(np.ascontiguousarray(result))
            if template.dtype in (torch.float16, torch.bfloat16):
                return t.view(torch.int16).view(template.dtype)
            return t.view(template.dtype)
    except ImportError:  # pragma: no cover
        pass
    return result


def append(cache, src, slot_mapping):
    """Return a copy of ``cache`` [NB, Hkv, bs, D] with rows of ``src`` [T, Hkv, D]
    scattered to their slots (negative slot = skipped).  Raw bytes are moved,
    so any element type works."""
    c = np.array(_raw(cache)[0], copy=True)
    s = _raw(src)[0]
    sm = _i32(slot_mapping)
    NB, Hkv, bs, D = c.shape
    if s.shape[1:] != (Hkv, D) or s.dtype.itemsize != c.dtype.itemsize:
        raise ValueError("shape mismatch")
    err = _load().orc_append(_ptr(c), _ptr(s), _ptr(sm), sm.shape[0], Hkv, D,
                             c.dtype.itemsize, NB, bs)
    if err != 0:
        raise ValueError("oracle append: slot out of range")
    return _like(c, cache)


def append_rows(pool, rows, slot_mapping):
    """Generic scatter for any [NB, Hkv, bs, ...] pool with rows [T, Hkv, ...]
    (used for the float32 scale pools): same rule as ``append``."""
    p = np.array(pool, copy=True)
    NB, Hkv, bs = p.shape[:3]
    inner = int(np.prod(p.shape[3:])) if p.ndim > 3 else 1
    r = np.ascontiguousarray(rows)
    sm = _i32(slot_mapping)
    err = _load().orc_append(_ptr(p), _ptr(r), _ptr(sm), sm.shape[0], Hkv, inner,
                             p.dtype.itemsize, NB, bs)
    if err != 0:
        raise ValueError("oracle append: slot out of range")
    return p


def copy_blocks(pool, pairs):
    """Return a copy of ``pool`` [NB, ...] with block src copied onto block dst for
    each (src, dst) in ``pairs``, in order."""
    if isinstance(pool, np.ndarray):
        p = np.array(pool, copy=True)
    else:
        try:
            import torch
            is_float = isinstance(pool, torch.Tensor) and pool.dtype == torch.float32
        except ImportError:  # pragma: no cover
            is_float = False
        p = np.array(_f32(pool) if is_float else _raw(pool)[0], copy=True)
    pr = _i32(pairs).reshape(-1, 2)
    NB = p.shape[0]
    block_bytes = p.nbytes // NB if NB else 0
    err = _load().orc_copy_blocks(_ptr(p), _ptr(pr), pr.shape[0], block_bytes, NB)
    if err != 0:
        raise ValueError("oracle copy_blocks: block id out of range")
    return _like(p, pool)


def quantize_int8(src):
    """Per-row (last axis) INT8 quantisation of f16/bf16 ``src`` [..., D].
    Returns (codes int8 [..., D], scales float32 [...])."""
    a, kind = _raw(src)
    if kind not in (F16, BF16):
        raise TypeError("quantize_int8 takes f16 or bf16 input")
    D = a.shape[-1]
    rows = a.size // D if D else 0
    q = np.empty(a.shape, dtype=np.int8)
    s = np.empty(a.shape[:-1], dtype=np.float32)
    _load().orc_quantize_int8(_ptr(a), kind, rows, D, _ptr(q), _ptr(s))
    return q, s


def quantize_int8_fixed(src, scale):
    """Per-tensor INT8 quantisation of f16/bf16 ``src`` with a given scale."""
    a, kind = _raw(src)
    if kind not in (F16, BF16):
        raise TypeError("quantize_int8_fixed takes f16 or bf16 input")
    q = np.empty(a.shape, dtype=np.int8)
    _load().orc_quantize_int8_fixed(_ptr(a), kind, a.size, float(scale), _ptr(q))
    return q


def quantize_fp8(src):
    """Per-row (last axis) E4M3 quantisation of f16/bf16 ``src`` [..., D].
    Returns (codes as uint8 bit patterns [..., D], scales float32 [...])."""
    a, kind = _raw(src)
    if kind not in (F16, BF16):
        raise TypeError("quantize_fp8 takes f16 or bf16 input")
    D = a.shape[-1]
    rows = a.size // D if D else 0
    q = np.empty(a.shape, dtype=np.uint8)
    s = np.empty(a.shape[:-1], dtype=np.float32)
    _load().orc_quantize_fp8(_ptr(a), kind, rows, D, _ptr(q), _ptr(s))
    return q, s


def append_fp8(k_codes, k_scales, src, slot_mapping):
    """As append_int8 with the FP8 (E4M3) quantiser; codes are uint8 bit patterns
    (or torch float8_e4m3fn tensors, returned as such)."""
    q, s = quantize_fp8(src)
    codes = append(k_codes, q.view(np.uint8), slot_mapping)
    scales = _like(append_rows(_f32(k_scales), s, slot_mapping), k_scales)
    return codes, scales


def append_int8_fixed(k_codes, k_scales, src, slot_mapping, scale):
    """Per-tensor INT8 append: codes with the given scale, which is also written
    to the scale pool at each slot."""
    q = quantize_int8_fixed(src, scale)
    codes = append(k_codes, q, slot_mapping)
    rows = np.full(q.shape[:-1], scale, dtype=np.float32)
    scales = _like(append_rows(_f32(k_scales), rows, slot_mapping), k_scales)
    return codes, scales


def append_int8(k_codes, k_scales, src, slot_mapping):
    """Quantise ``src`` [T, Hkv, D] per row, then scatter codes and scales into
    copies of the int8 pool [NB, Hkv, bs, D] and scale pool [NB, Hkv, bs]."""
    q, s = quantize_int8(src)
    codes = append(k_codes, q, slot_mapping)
    scales = _like(append_rows(_f32(k_scales), s, slot_mapping), k_scales)
    return codes, scales
