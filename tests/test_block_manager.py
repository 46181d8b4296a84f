"""Host block manager (kvp_bm_*): allocation, sharing, copy-on-write, refcounts,
statistics -- checked against the pages' stated semantics and invariants."""
import os
import random

import pytest

import pagedattention_decode_kvp_gb300 as kvp
from pagedattention_decode_kvp_gb300 import _build

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_manager.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=")
            vals[k.strip()] = int(v)
    return vals


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kvp.load_library()


def _invariants(bm, n_blocks, reqs):
    st = bm.stats()
    assert st["free_blocks"] + st["used_blocks"] == n_blocks
    held = [b for r in reqs for b in bm.block_table(r)]
    assert st["block_refs"] == len(held)                      # sum of counts = table refs
    for b in set(held):
        assert bm.ref_count(b) == held.count(b)
    assert st["used_blocks"] == len(set(held))


def test_block_counts_from_the_pages():
    g = _golden()
    bm = kvp.BlockManager(64)
    bm.allocate(1, 48)
    bm.allocate(2, 1)
    bm.allocate(3, 17)
    assert len(bm.block_table(1)) == g["tokens_48_blocks"]
    assert len(bm.block_table(2)) == g["tokens_1_blocks"]
    assert len(bm.block_table(3)) == g["tokens_17_blocks"]
    bm.allocate(4, 100, reserve_blocks=1)     # allocate_request reserves one page
    assert len(bm.block_table(4)) == g["prompt_100_pages_with_reserve"]
    _invariants(bm, 64, [1, 2, 3, 4])


def test_contiguous_first_from_largest_range():
    bm = kvp.BlockManager(32)
    bm.allocate(1, 16 * 4)        # 0..3
    bm.allocate(2, 16 * 2)        # 4..5
    bm.allocate(3, 16 * 10)       # 6..15
    bm.free(2)                    # free ranges: [4,6) len 2 and [16,32) len 16
    bm.allocate(4, 16 * 3)
    assert bm.block_table(4) == [16, 17, 18]   # the largest range holds it
    bm.allocate(5, 16 * 13)                    # 19..31 is the only range of 13
    assert bm.block_table(5) == list(range(19, 32))
    bm.allocate(6, 16 * 2)                     # fits the 2-block hole
    assert bm.block_table(6) == [4, 5]
    _invariants(bm, 32, [1, 3, 4, 5, 6])


def test_scattered_when_no_range_is_long_enough():
    bm = kvp.BlockManager(8)
    for r in range(8):
        bm.allocate(r, 16)
    for r in (1, 3, 6):
        bm.free(r)
    bm.allocate(10, 16 * 3)
    assert bm.block_table(10) == [1, 3, 6]


def test_oom_leaves_state_unchanged():
    bm = kvp.BlockManager(4)
    bm.allocate(1, 16 * 3)
    before = bm.stats()
    with pytest.raises(kvp.KvpError) as e:
        bm.allocate(2, 16 * 2)
    assert e.value.status == kvp.KVP_ERR_OOM
    assert bm.stats() == before
    assert bm.num_tokens(2) == -1


def test_append_takes_a_new_block_when_full_and_prefers_the_next_id():
    bm = kvp.BlockManager(16)
    bm.allocate(1, 16)
    (b0,) = bm.block_table(1)
    slot, cs, cd = bm.append_slot(1)           # token 16 needs a second block
    assert (cs, cd) == (-1, -1)
    t = bm.block_table(1)
    assert len(t) == 2 and t[1] == b0 + 1 and slot == t[1] * 16
    for i in range(15):
        slot, _, _ = bm.append_slot(1)
        assert slot == t[1] * 16 + 1 + i
    assert bm.num_tokens(1) == 32


def test_prefix_sharing_copy_on_write_and_refcounts():
    bm = kvp.BlockManager(128)
    bm.allocate(0, 1030)                     # 64 full blocks + 6 tokens
    shared = bm.block_table(0)
    for r in range(1, 4):
        bm.share_prefix(0, r, 1030)
    assert all(bm.ref_count(b) == 4 for b in shared)
    # appending into the shared partial block copies it first
    slot, cs, cd = bm.append_slot(1)
    assert cs == shared[64] and cd not in shared
    assert slot == cd * 16 + 6
    assert bm.ref_count(shared[64]) == 3 and bm.ref_count(cd) == 1
    slot, cs, cd2 = bm.append_slot(1)        # now private: no copy
    assert cs == -1 and slot == cd * 16 + 7
    # last sharer writes in place once the others moved away
    for r in (2, 3):
        _, cs, _ = bm.append_slot(r)
        assert cs == shared[64]
    _, cs, _ = bm.append_slot(0)
    assert cs == -1 and bm.ref_count(shared[64]) == 1
    _invariants(bm, 128, [0, 1, 2, 3])


def test_release_by_non_holder_is_a_refcount_error_and_frees_at_zero():
    bm = kvp.BlockManager(8)
    bm.allocate(1, 32)
    bm.share_prefix(1, 2, 16)
    b = bm.block_table(1)
    bm.allocate(3, 16)
    with pytest.raises(kvp.KvpError) as e:
        bm.release_block(3, b[0])
    assert e.value.status == kvp.KVP_ERR_REFCOUNT
    bm.release_block(2, b[0])                  # count 2 -> 1: stays allocated
    assert bm.ref_count(b[0]) == 1
    bm.free(1)
    assert bm.ref_count(b[0]) == 0 and bm.ref_count(b[1]) == 0
    with pytest.raises(kvp.KvpError) as e:
        bm.free(1)
    assert e.value.status == kvp.KVP_ERR_NOT_FOUND


def test_no_leak_after_random_workload():
    rng = random.Random(5)
    n = 256
    bm = kvp.BlockManager(n, 16, 262144)
    live = {}
    nxt = 0
    for step in range(3000):
        op = rng.random()
        if op < 0.3:
            try:
                bm.allocate(nxt, rng.randint(0, 200))
                live[nxt] = True
            except kvp.KvpError as e:
                assert e.status == kvp.KVP_ERR_OOM
            nxt += 1
        elif op < 0.4 and live:
            src = rng.choice(list(live))
            k = rng.randint(0, max(0, bm.num_tokens(src)))
            bm.share_prefix(src, nxt, k)
            live[nxt] = True
            nxt += 1
        elif op < 0.85 and live:
            r = rng.choice(list(live))
            try:
                bm.append_slot(r)
            except kvp.KvpError as e:
                assert e.status == kvp.KVP_ERR_OOM
        elif live:
            r = rng.choice(list(live))
            bm.free(r)
            del live[r]
        if step % 100 == 0:
            _invariants(bm, n, list(live))
    for r in list(live):
        bm.free(r)
    st = bm.stats()
    assert st["free_blocks"] == n and st["block_refs"] == 0 and st["active_requests"] == 0
    assert abs(st["total_memory_gb"] - n * 262144 / 1e9) < 1e-12
