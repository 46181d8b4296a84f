"""Failure detection without a GPU fault: every pipeline wait of the library
goes through one bounded mbarrier wait.  Here it waits on a barrier nothing
arrives on, with a short limit, must give up, record KVP_ERR_TIMEOUT in the
status word and leave the context usable (a prefill afterwards still matches
the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
import pagedattention_decode_kvp_gb300 as kvp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pagedattention_decode_kvp_gb300 import _build
    _build.build()
    kvp.load_library()


def test_bounded_wait_gives_up_and_reports_timeout():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvp.kvp_selftest_wait_timeout(status, 20_000_000)  # 20 ms
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    # the second warp waits with the default 2 s limit but stops on the
    # abort flag the first one sets: the launch ends well before 2 s
    assert 0.015 < elapsed < 0.5, elapsed
    # the first error stays: a second timeout leaves the word as it is
    kvp.kvp_selftest_wait_timeout(status, 1_000_000)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_TIMEOUT

    # the context is still usable
    w = workloads.make_prefill(B=2, Hq=8, Hkv=2, D=64, lens=[200, 90], qlens=[150, 30],
                               num_blocks=24, dtype=torch.float16, seed=77, device="cuda")
    out = torch.empty((w.T, w.Hq, w.D), dtype=w.dtype, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvp.kvp_attention_prefill(out, w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                              w.query_start, w.max_query_len, w.scale, status=st2)
    assert kvp.kvp_read_status(st2) == kvp.KVP_OK
    ref = oracle.attention_prefill(w.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(),
                                   w.block_tables.cpu(), w.context_lens.cpu(),
                                   w.query_start.cpu(), w.scale)
    got = out.double().cpu().numpy().reshape(ref.shape)
    err = np.abs(got - ref)
    assert ((err <= 3e-3) | (err <= 1e-2 * np.abs(ref))).all()
