"""The C-ABI library builds, loads and exports every symbol include/kvp.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

import pagedattention_decode_kvp_gb300 as kvp
from pagedattention_decode_kvp_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kvp.load_library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(kvp_\w+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("kvp_append", "kvp_append_int8", "kvp_copy_blocks", "kvp_attention_decode",
                 "kvp_attention_decode_int8", "kvp_decode_workspace_bytes", "kvp_read_status",
                 "kvp_append_fp8", "kvp_attention_decode_fp8", "kvp_append_int8_fixed",
                 "kvp_append_attention_decode",
                 "kvp_bm_create", "kvp_bm_allocate", "kvp_bm_append_slot", "kvp_bm_free"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    # the binding types every declared symbol
    assert _declared() <= set(kvp.SIGNATURES)


def test_version_and_status_strings(lib):
    assert kvp.kvp_version() >= 100
    assert kvp.kvp_status_string(0) == "KVP_OK"
    assert kvp.kvp_status_string(kvp.KVP_ERR_REFCOUNT) == "KVP_ERR_REFCOUNT"


def _desc(nb=64, hkv=2, bs=16, d=64):
    return kvp.kvp_cache_desc(nb, hkv, bs, d)


def test_workspace_sizing_rules(lib):
    # single pass when the table fits one partition: no workspace
    assert kvp.kvp_decode_workspace_bytes(4, 8, _desc(), 16) == 0
    # 4096-token contexts, 32 x 32 heads: the automatic split, and its workspace
    d = _desc(10000, 32, 16, 128)
    pb = kvp.kvp_decode_partition_blocks(32, 32, d, 256)
    assert 16 <= pb < 256
    parts = -(-256 // pb)
    assert kvp.kvp_decode_workspace_bytes(32, 32, d, 256) == 32 * 32 * parts * (128 + 2) * 4
    # explicit partition size
    assert kvp.kvp_decode_workspace_bytes(32, 32, d, 256, 64) == 32 * 32 * 4 * (128 + 2) * 4
    assert kvp.kvp_decode_workspace_bytes(32, 32, d, 256, 256) == 0   # single pass
    # many short requests stay single pass; one very long one is split
    assert kvp.kvp_decode_workspace_bytes(128, 32, _desc(8192, 32, 16, 128), 97) == 0
    assert kvp.kvp_decode_partition_blocks(4, 64, _desc(40000, 8, 16, 128), 8192, 1) <= 1024
    # the FP8 decode (kv_8bit = 2) runs fewer, larger CTAs per SM than the INT8
    # one, so it cuts long contexts into fewer partitions; other kinds answer 0
    d8 = _desc(40000, 8, 16, 128)
    int8_pb = kvp.kvp_decode_partition_blocks(4, 64, d8, 8192, kv_int8=True)
    fp8_pb = kvp.kvp_decode_partition_blocks(4, 64, d8, 8192, kv_fp8=True)
    assert 16 <= int8_pb <= fp8_pb <= 1024
    assert lib.kvp_decode_workspace_bytes(4, 64, d8, 8192, 0, 3) == 0
    # invalid sizes answer 0
    assert kvp.kvp_decode_workspace_bytes(4, 6, _desc(hkv=4), 16) == 0      # 6 % 4 != 0
    assert kvp.kvp_decode_workspace_bytes(4, 8, _desc(d=96), 16) == 0       # head_dim 96


def test_invalid_arguments_fail_before_any_launch(lib):
    P = None
    # unsupported block size / head_dim
    assert lib.kvp_append(P, P, P, P, P, 1, _desc(bs=32), 0, P, P) == kvp.KVP_ERR_UNSUPPORTED
    assert lib.kvp_append(P, P, P, P, P, 1, _desc(d=80), 0, P, P) == kvp.KVP_ERR_UNSUPPORTED
    # null pointers with work to do
    assert lib.kvp_append(P, P, P, P, P, 1, _desc(), 0, P, P) == kvp.KVP_ERR_INVALID_ARG
    # zero tokens is a no-op even with null pointers
    assert lib.kvp_append(P, P, P, P, P, 0, _desc(), 0, P, P) == kvp.KVP_OK
    assert lib.kvp_copy_blocks(P, P, P, P, 2, P, 0, _desc(), P, P) == kvp.KVP_OK
    assert lib.kvp_copy_blocks(P, P, P, P, 3, P, 1, _desc(), P, P) == kvp.KVP_ERR_INVALID_ARG
    # decode: Hq not a multiple of Hkv, null buffers, bad phases, missing workspace
    args = lambda hq, phases, ws_bytes: (P, P, P, P, P, 16, P, 4, hq, 0.125, _desc(), 0, 0, P,
                                         ws_bytes, phases, P, P)
    assert lib.kvp_attention_decode(*args(7, 3, 0)) == kvp.KVP_ERR_INVALID_ARG
    assert lib.kvp_attention_decode(*args(8, 3, 0)) == kvp.KVP_ERR_INVALID_ARG
    assert lib.kvp_attention_decode(*args(8, 4, 0)) == kvp.KVP_ERR_INVALID_ARG
    # the run-merge flag alone names no phase; with a phase it passes the phase check
    merge = kvp.KVP_DECODE_MERGE_RUNS
    assert lib.kvp_attention_decode(*args(8, merge, 0)) == kvp.KVP_ERR_INVALID_ARG
    assert lib.kvp_attention_decode(*args(8, merge | 16, 0)) == kvp.KVP_ERR_INVALID_ARG
    zero_merge = (P, P, P, P, P, 16, P, 0, 8, 0.125, _desc(), 0, 0, P, 0, 3 | merge, P, P)
    assert lib.kvp_attention_decode(*zero_merge) == kvp.KVP_OK
    big = (P, P, P, P, P, 256, P, 4, 8, 0.125, _desc(), 0, 0, P, 0, 3, P, P)
    assert lib.kvp_attention_decode(*big) == kvp.KVP_ERR_INVALID_ARG  # needs workspace
    # batch 0 is a no-op
    zero = (P, P, P, P, P, 16, P, 0, 8, 0.125, _desc(), 0, 0, P, 0, 3, P, P)
    assert lib.kvp_attention_decode(*zero) == kvp.KVP_OK
    assert lib.kvp_read_status(P, P) == kvp.KVP_ERR_INVALID_ARG
    # the per-tensor INT8 scale must be finite and positive
    assert lib.kvp_append_int8_fixed(P, P, 0, P, P, P, P, 0.0, 1.0, P, 1, _desc(), P, P) == \
        kvp.KVP_ERR_INVALID_ARG
    assert lib.kvp_append_fp8(P, P, 0, P, P, P, P, P, 1, _desc(), P, P) == kvp.KVP_ERR_INVALID_ARG


def test_product_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(kvp, "_lib", None)
    monkeypatch.setattr(kvp, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        kvp.load_library()


def test_selftest_wait_checks_its_arguments_before_launch(lib):
    A = ctypes.c_void_p(1 << 20)
    assert lib.kvp_selftest_wait_timeout(None, 1_000_000, None) == kvp.KVP_ERR_INVALID_ARG
    assert lib.kvp_selftest_wait_timeout(A, 0, None) == kvp.KVP_ERR_INVALID_ARG
    assert lib.kvp_selftest_wait_timeout(A, 6_000_000_000, None) == kvp.KVP_ERR_INVALID_ARG


def test_prefill_invalid_arguments_fail_before_any_launch(lib):
    P = None
    inf = float("inf")

    def call(hq=8, d=None, T=64, batch=2, mql=32, scale=0.125, dtype=0, shared=0):
        desc = _desc() if d is None else d
        return lib.kvp_attention_prefill(P, P, P, P, P, 16, P, P, T, batch, hq, mql, shared,
                                         scale, desc, dtype, P, P)
    # group (Hq / Hkv) must divide the 128-row tile; Hq must be a multiple of Hkv
    assert call(hq=_desc().num_kv_heads * 3) == kvp.KVP_ERR_UNSUPPORTED
    assert call(hq=_desc().num_kv_heads + 1) == kvp.KVP_ERR_INVALID_ARG
    # unsupported head_dim / block size, bad dtype, non-finite scale, negative sizes
    assert call(d=_desc(d=80)) == kvp.KVP_ERR_UNSUPPORTED
    assert call(d=_desc(bs=32)) == kvp.KVP_ERR_UNSUPPORTED
    assert call(dtype=2) == kvp.KVP_ERR_INVALID_ARG
    assert call(scale=inf) == kvp.KVP_ERR_INVALID_ARG
    assert call(T=-1) == kvp.KVP_ERR_INVALID_ARG
    assert call(mql=-1) == kvp.KVP_ERR_INVALID_ARG
    # the shared prefix is a count of table entries: 0 .. max_blocks_per_seq
    assert call(shared=-1) == kvp.KVP_ERR_INVALID_ARG
    assert call(shared=17) == kvp.KVP_ERR_INVALID_ARG
    assert call(shared=16, batch=0) == kvp.KVP_OK
    # null buffers with work to do
    assert call() == kvp.KVP_ERR_INVALID_ARG
    # nothing to do: no-ops even with null buffers
    assert call(batch=0) == kvp.KVP_OK
    # a work list of 2^31 or more 128-row items is refused before any launch
    # (fake, aligned, never dereferenced buffer addresses)
    A = ctypes.c_void_p(1 << 20)
    big = lib.kvp_attention_prefill(A, A, A, A, A, 16, A, A, 64, 65535, _desc().num_kv_heads,
                                    0x7fffffff, 0, 0.125, _desc(), 0, A, P)
    assert big == kvp.KVP_ERR_UNSUPPORTED
    # dense tiles are counted from the query rows: 2^31 - 1 tokens of 128-head
    # groups are 2^31 - 1 tiles for each of 8 kv heads
    big = lib.kvp_attention_prefill(A, A, A, A, A, 16, A, A, 0x7fffffff, 4, 8 * 128, 16, 1,
                                    0.125, _desc(hkv=8), 0, A, P)
    assert big == kvp.KVP_ERR_UNSUPPORTED
    assert call(mql=0) == kvp.KVP_OK
    assert call(T=0) == kvp.KVP_OK


def test_shared_prefix_decode_sizing_and_validation(lib):
    d = _desc(8192, 32, 16, 128)
    # 64 shared blocks of a 97-block table: the prefix pass covers 64, the split
    # decode the remaining 33 (one partition): two partitions per row
    wsb = kvp.kvp_decode_shared_prefix_workspace_bytes(128, 32, d, 97, 64)
    assert wsb == 128 * 32 * 2 * (128 + 2) * 4
    # a prefix shorter than one 128-token chunk sizes the ordinary decode
    assert kvp.kvp_decode_shared_prefix_workspace_bytes(128, 32, d, 97, 7) == \
        kvp.kvp_decode_workspace_bytes(128, 32, d, 97)
    # invalid sizes answer 0
    assert kvp.kvp_decode_shared_prefix_workspace_bytes(128, 32, d, 97, 98) == 0
    assert kvp.kvp_decode_shared_prefix_workspace_bytes(128, 32, d, 97, -1) == 0
    P = None
    A = ctypes.c_void_p(1 << 20)

    def call(shared=64, dtype=0, ws_bytes=wsb, ws=A, batch=128, mb=97):
        return lib.kvp_attention_decode_shared_prefix(A, A, A, A, A, mb, A, batch, 32, 0.125, d,
                                                      dtype, shared, 0, ws, ws_bytes, P, P)
    assert call(dtype=2) == kvp.KVP_ERR_INVALID_ARG          # 8-bit codes: not this call
    assert call(shared=98) == kvp.KVP_ERR_INVALID_ARG        # more than the table
    assert call(ws_bytes=wsb - 16) == kvp.KVP_ERR_INVALID_ARG
    assert call(ws=P) == kvp.KVP_ERR_INVALID_ARG
    assert call(batch=0) == kvp.KVP_OK
