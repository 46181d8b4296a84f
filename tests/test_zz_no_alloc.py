"""kvp_attention_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a plugin whose host framework owns all device memory,
or a serving loop that has handed nearly all HBM to the KV pool and must not
risk a cudaMalloc mid-step).  It keeps its split-context partials in a scratch
array built into the library instead of a caller workspace.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
import pagedattention_decode_kvp_gb300 as kvp
from pagedattention_decode_kvp_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kvp.load_library()


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    err = np.abs(a - b)
    return bool(np.all((err <= 3e-3) | (err <= 1e-2 * np.abs(b))))


@pytest.mark.gpu
def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(lib):
    w = workloads.make_custom(B=4, Hq=16, Hkv=2, D=128, lens=[3000, 17, 1500, 800],
                              num_blocks=400, dtype=torch.bfloat16, seed=21)
    desc = kvp.cache_desc(w.k_pool)
    need = kvp.kvp_decode_workspace_bytes(w.B, w.Hq, desc, w.max_blocks)
    assert 0 < need <= kvp.NOALLOC_SCRATCH_BYTES  # this case really uses the scratch
    kp, vp = w.k_pool.cuda(), w.v_pool.cuda()
    q, bt, cl = w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda()
    ref = torch.empty_like(q)
    ws = torch.empty(need // 4 + 4, dtype=torch.float32, device="cuda")
    kvp.kvp_attention_decode(ref, q, kp, vp, bt, cl, w.scale, workspace=ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # every buffer the calls write is allocated up front, so nothing below
    # but the entry point itself could take device memory
    outs = [torch.full_like(q, float("nan")) for _ in range(3)]

    def call(out):
        st = lib.kvp_attention_decode_noalloc(
            out.data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(),
            w.max_blocks, cl.data_ptr(), w.B, w.Hq, ctypes.c_float(w.scale), desc,
            kvp.KVP_BF16, 0, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == kvp.KVP_OK
        torch.cuda.synchronize()
        assert kvp.kvp_read_status(status) == kvp.KVP_OK

    call(outs[0])  # the first call on this device looks up the scratch address
    free_before = torch.cuda.mem_get_info()[0]
    for out in outs[1:]:  # two more calls in a row
        call(out)
    assert torch.cuda.mem_get_info()[0] == free_before  # no device memory was taken
    for out in outs:
        assert torch.isfinite(out.float()).all()
        assert _close(out, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # 64 requests x 64 heads x 8192-block tables cut into 16-block partitions:
    # far more partials than the scratch array holds
    desc = kvp.kvp_cache_desc(40000, 8, 16, 128)
    assert kvp.kvp_decode_workspace_bytes(64, 64, desc, 8192, 16) > kvp.NOALLOC_SCRATCH_BYTES
    st = lib.kvp_attention_decode_noalloc(None, None, None, None, None, 8192, None, 64, 64,
                                          ctypes.c_float(0.1), desc, kvp.KVP_BF16, 16, None,
                                          None)
    assert st == kvp.KVP_ERR_SCRATCH_LIMIT
    assert kvp.kvp_status_string(st) == "KVP_ERR_SCRATCH_LIMIT"
