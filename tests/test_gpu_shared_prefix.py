"""GPU parity of the decode over a shared prompt prefix
(kvp_attention_decode_shared_prefix), through the C ABI, against the fp64 CPU
oracle on the same seeded inputs ("ATB KV Cache management", "Prefix Caching":
every request's table names the same physical blocks for the cached prompt).

Bar: the decode's -- within 3e-3 absolute OR 1e-2 relative of the oracle,
element by element.  The prefix part (its whole 128-token chunks, on the tensor
cores, once per kv head) and the rest of each context (the split decode over the
remaining blocks) are merged by the reduce; cases cover prefixes of one to nine
chunks with ragged tails, suffixes from empty to several partitions, GQA groups
1 to 8, fp16 and bf16, D 64 and 128, NaN in every pool slot no request owns,
tables that disagree on the prefix, and lengths that do not cover it."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import pagedattention_decode_kvp_gb300 as kvp

pytestmark = pytest.mark.gpu

ATOL, RTOL = 3e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pagedattention_decode_kvp_gb300 import _build
    _build.build()
    kvp.load_library()


def assert_close(gpu_out, ref, what=""):
    g = gpu_out.detach().double().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    ok = (err <= ATOL) | (err <= RTOL * np.abs(ref))
    if not ok.all():
        i = np.unravel_index(np.argmax(np.where(ok, 0, err)), err.shape)
        raise AssertionError(f"{what}: {int((~ok).sum())} elements out of tolerance; worst at "
                             f"{i}: gpu {g[i]} ref {ref[i]} (max abs err {err.max():.3e})")


def shared_case(B, Hq, Hkv, D, S, suffix, dtype=torch.float16, seed=5):
    """B requests sharing S prefix blocks; request b holds S*16 + suffix[b] tokens
    (its last token is the decode query's position).  One query per request."""
    lens = [S * 16 + s for s in suffix]
    nb = S + sum(-(-(n - S * 16) // 16) for n in lens) + 8
    w = workloads.make_prefill(B=B, Hq=Hq, Hkv=Hkv, D=D, lens=lens, qlens=[1] * B,
                               num_blocks=nb, dtype=dtype, seed=seed, shared_blocks=S)
    return w


def run(w, S, status=None, partition_blocks=0, tables=None, lens=None):
    tables = (w.block_tables if tables is None else tables).cuda()
    lens = (w.context_lens if lens is None else lens).cuda()
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=w.dtype, device="cuda")
    wsb = kvp.kvp_decode_shared_prefix_workspace_bytes(
        w.B, w.Hq, kvp.cache_desc(w.k_pool), int(tables.shape[1]), S, partition_blocks)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    kvp.kvp_attention_decode_shared_prefix(out, w.q.cuda(), w.k_pool.cuda(), w.v_pool.cuda(),
                                           tables, lens, w.scale, S, workspace=ws,
                                           partition_blocks=partition_blocks, status=status)
    torch.cuda.synchronize()
    return out


def oracle_decode(w, tables=None, lens=None):
    return oracle.attention_decode(w.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(),
                                   (w.block_tables if tables is None else tables).cpu(),
                                   (w.context_lens if lens is None else lens).cpu(), w.scale)


CASES = [
    # B, Hq, Hkv, D, S (shared blocks), suffix lengths, dtype
    (6, 8, 8, 128, 8, [0, 1, 15, 16, 17, 300], torch.float16),      # one chunk; empty suffix
    (5, 16, 2, 64, 11, [1, 100, 255, 256, 700], torch.float16),     # ragged prefix (11 blocks)
    (9, 32, 4, 128, 64, [16, 37, 200, 511, 512, 3, 90, 128, 260], torch.bfloat16),
    (4, 8, 1, 128, 70, [5, 1000, 2048, 64], torch.float16),         # G = 8, long suffixes
    (130, 4, 4, 64, 16, list(range(1, 131)), torch.float16),        # > 128 rows per kv head
    (3, 12, 4, 128, 24, [50, 70, 90], torch.bfloat16),              # G = 3 (ordinary decode)
]


@pytest.mark.parametrize("B,Hq,Hkv,D,S,suffix,dtype", CASES)
def test_shared_prefix_decode_matches_oracle(B, Hq, Hkv, D, S, suffix, dtype):
    w = shared_case(B, Hq, Hkv, D, S, suffix, dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(w, S, status)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    assert_close(out, oracle_decode(w), f"B{B} Hq{Hq} Hkv{Hkv} D{D} S{S} {dtype}")


@pytest.mark.parametrize("pb", [16, 40])
def test_shared_prefix_decode_explicit_partitions(pb):
    w = shared_case(7, 16, 4, 128, 16, [1, 40, 300, 900, 1500, 64, 2000], torch.float16, seed=9)
    out = run(w, 16, partition_blocks=pb)
    assert_close(out, oracle_decode(w), f"pb {pb}")


def test_shared_prefix_decode_equals_ordinary_decode_within_bar():
    w = shared_case(12, 8, 8, 128, 32, [3, 60, 129, 400, 17, 1, 256, 300, 77, 500, 8, 200],
                    torch.float16, seed=13)
    out = run(w, 32)
    ref_gpu = torch.empty_like(out)
    wsb = kvp.kvp_decode_workspace_bytes(w.B, w.Hq, kvp.cache_desc(w.k_pool),
                                         int(w.block_tables.shape[1]))
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    kvp.kvp_attention_decode(ref_gpu, w.q.cuda(), w.k_pool.cuda(), w.v_pool.cuda(),
                             w.block_tables.cuda(), w.context_lens.cuda(), w.scale, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle_decode(w)
    assert_close(out, ref, "shared prefix")
    assert_close(ref_gpu, ref, "ordinary")


def test_prefix_tables_that_disagree_set_status_and_zero_rows():
    w = shared_case(4, 8, 8, 64, 16, [30, 40, 50, 60], torch.float16, seed=21)
    tables = w.block_tables.clone()
    tables[2, 5] = tables[2, int(w.context_lens[2]) // 16]  # another block of the request
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(w, 16, status, tables=tables)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    # rows of the tile that read the first request's prefix through a table a
    # member disagrees with are zeros; no NaN reaches any row
    g = out.double().cpu().numpy()
    assert np.isfinite(g).all()
    assert (g[2] == 0).all()


@pytest.mark.parametrize("bad_req", [1, 9, 33, 39])
def test_wide_tile_checks_find_a_disagreeing_table_or_short_length(bad_req):
    """A prefix tile of 40 requests (checked 32 requests per batch of loads):
    a disagreeing prefix entry, or a length that does not cover the prefix, in
    the first or a later batch sets the status; no NaN reaches any row."""
    w = shared_case(40, 4, 4, 64, 16, [5 + 3 * i for i in range(40)], torch.float16, seed=23)
    tables = w.block_tables.clone()
    tables[bad_req, 7] = tables[bad_req, int(w.context_lens[bad_req]) // 16]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(w, 16, status, tables=tables)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    g = out.double().cpu().numpy()
    assert np.isfinite(g).all()
    assert (g[bad_req] == 0).all()
    lens = w.context_lens.clone()
    lens[bad_req] = 16 * 16 - 3
    status.zero_()
    out = run(w, 16, status, lens=lens)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert np.isfinite(out.double().cpu().numpy()).all()


def test_lengths_that_do_not_cover_the_prefix_set_status():
    w = shared_case(3, 8, 8, 64, 16, [10, 20, 30], torch.float16, seed=22)
    lens = w.context_lens.clone()
    lens[1] = 16 * 16 - 5  # shorter than the shared prefix
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(w, 16, status, lens=lens)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert np.isfinite(out.double().cpu().numpy()).all()


def test_prefix_workload_full_size():
    """The bench's prefix-sharing decode: 128 requests sharing 64 blocks (1024
    tokens) plus a copied partial block and 16-512 private tokens; every (request,
    head) row checked."""
    w = workloads.make("prefix", device="cpu")
    # the step before the decode: copy-on-write of the shared partial block,
    # then the append of every private token (the pools the decode reads)
    pairs = w.cow_pairs.cpu()
    k = oracle.append(oracle.copy_blocks(w.k_pool, pairs), w.new_k, w.slot_mapping.cpu())
    v = oracle.append(oracle.copy_blocks(w.v_pool, pairs), w.new_v, w.slot_mapping.cpu())
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=w.dtype, device="cuda")
    wsb = kvp.kvp_decode_shared_prefix_workspace_bytes(
        w.B, w.Hq, kvp.cache_desc(w.k_pool), int(w.block_tables.shape[1]), 64)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvp.kvp_attention_decode_shared_prefix(out, w.q.cuda(), k.cuda(), v.cuda(),
                                           w.block_tables.cuda(), w.context_lens.cuda(),
                                           w.scale, 64, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    ref = oracle.attention_decode(w.q, k, v, w.block_tables, w.context_lens, w.scale)
    assert_close(out, ref, "prefix workload")
