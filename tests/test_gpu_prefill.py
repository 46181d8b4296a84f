"""GPU parity of the causal multi-query (prefill / chunked-prefill) kernel,
called through the C ABI, against the fp64 CPU oracle on the same seeded inputs.

Bar: within 3e-3 absolute OR 1e-2 relative of the oracle, element by element
(the same bar as the decode: fp16/bf16 inputs, fp32 accumulation, P rounded to
the input type -- bf16 P carried as a high part plus a bf16 residual).
Cases span several 128-row query tiles and 128-key chunks with ragged tails
(full tiles leave through a TMA store, partial ones through plain stores), a
whole-prompt prefill, chunks that start mid-context, single-token chunks, empty
chunks, NaN in every pool slot no request owns, a sparse work list longer than
one scan window per block, rows whose running maximum jumps between chunks (the
lazy rescale of O and the row sums), and the data errors the header documents.
With a shared prompt prefix the rows of all requests are packed into dense
tiles; that mode must equal the per-request tiles bit for bit."""
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


def run_gpu(w, status=None, max_query_len=None, out=None, q=None, shared=0):
    if out is None:
        out = torch.full((w.T, w.Hq, w.D), float("nan"), dtype=w.dtype, device="cuda")
    kvp.kvp_attention_prefill(out, (w.q if q is None else q).cuda(), w.k_pool.cuda(),
                              w.v_pool.cuda(),
                              w.block_tables.cuda(), w.context_lens.cuda(),
                              w.query_start.cuda(),
                              w.max_query_len if max_query_len is None else max_query_len,
                              w.scale, shared_prefix_blocks=shared, status=status)
    torch.cuda.synchronize()
    return out


# (context length, chunk length) per request: a whole prompt spanning several
# tiles, chunks starting mid-context and crossing tile / chunk boundaries, one
# token, an empty chunk, exact multiples of 64 and 128.
CASES = [(300, 300), (1030, 200), (17, 1), (50, 0), (64, 64), (129, 129), (200, 37),
         (16, 16), (1, 1), (520, 130)]
# (Hq, Hkv, D): groups G = 1, 4, 8 and the extremes 32 (4 tokens per 128-row
# tile) and 128 (one token with all its heads per tile)
SHAPES = [(4, 4, 128), (8, 2, 64), (16, 2, 128), (8, 1, 128), (32, 4, 64), (64, 2, 64),
          (128, 1, 64)]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv,D", SHAPES)
def test_prefill_parity(dtype, Hq, Hkv, D):
    lens = [c[0] for c in CASES]
    qlens = [c[1] for c in CASES]
    w = workloads.make_prefill(B=len(CASES), Hq=Hq, Hkv=Hkv, D=D, lens=lens, qlens=qlens,
                               num_blocks=200, dtype=dtype, seed=Hq * 13 + D + Hkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, status)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                   w.query_start, w.scale)
    assert_close(out, ref, f"prefill {dtype} {Hq}/{Hkv} D{D}")


def test_prefill_scattered_and_contiguous_tables():
    for p in (0.0, 1.0):
        w = workloads.make_prefill(B=4, Hq=8, Hkv=2, D=128, lens=[700, 333, 129, 64],
                                   qlens=[700, 100, 129, 3], num_blocks=120,
                                   dtype=torch.bfloat16, seed=5, contiguous_p=p)
        out = run_gpu(w)
        ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables,
                                       w.context_lens, w.query_start, w.scale)
        assert_close(out, ref, f"contiguity {p}")


def test_one_token_chunks_match_the_decode_definition():
    """A chunk of one query per request is a decode step: compare with the
    oracle's decode on the same pools."""
    lens = [1, 16, 17, 300, 1000]
    w = workloads.make_prefill(B=5, Hq=16, Hkv=2, D=128, lens=lens, qlens=[1] * 5,
                               num_blocks=120, dtype=torch.float16, seed=9)
    out = run_gpu(w)
    ref = oracle.attention_decode(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                  w.scale)
    assert_close(out, ref, "one-token chunks")


def test_long_prompt_sampled_rows():
    """A 4096-token prompt (32 query tiles for G = 1; 64 key chunks for the last
    tile), checked on sampled rows the oracle computes one by one."""
    w = workloads.make_prefill(B=2, Hq=8, Hkv=8, D=128, lens=[4096, 2500], qlens=[4096, 900],
                               num_blocks=450, dtype=torch.bfloat16, seed=21)
    out = run_gpu(w)
    rng = np.random.default_rng(3)
    t = rng.integers(0, w.T, size=96)
    t[:4] = [0, 4095, 4096, w.T - 1]
    h = rng.integers(0, w.Hq, size=96)
    rows = np.stack([t, h], axis=1).astype(np.int32)
    ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                   w.query_start, w.scale, rows=rows)
    got = out.cpu()[torch.from_numpy(t).long(), torch.from_numpy(h).long()]
    assert_close(got, ref, "long prompt sampled")


def test_prefill_is_deterministic():
    w = workloads.make_prefill(B=3, Hq=8, Hkv=2, D=64, lens=[400, 90, 33], qlens=[400, 90, 5],
                               num_blocks=60, dtype=torch.float16, seed=2)
    a = run_gpu(w)
    b = run_gpu(w)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _plant_score_jumps(w, amp=8.0, step=12.0, period=5):
    """Scores that jump between chunks: K's first component is step * (c % period)
    at the keys of chunk c (positions 128 c .. 128 c + 127, through each
    request's table), q's first component +amp for even heads and -amp for odd
    ones.  An even head's scores then rise by amp * step * scale = 8.5 (12.2 in
    log2 units, past the 2^8 the running maximum may lag by) at each chunk of a
    period, so O and the row sums are rescaled chunk after chunk; an odd head
    keeps its first chunk's maximum."""
    k = w.k_pool.clone()
    tables = w.block_tables.cpu()
    for b in range(w.B):
        pos = torch.arange(int(w.context_lens[b]))
        blk = tables[b, pos // 16].long()
        k[blk, :, pos % 16, 0] = (step * ((pos // 128) % period)).to(k.dtype)[:, None]
    q = w.q.clone()
    q[:, 0::2, 0] = amp
    q[:, 1::2, 0] = -amp
    w.k_pool, w.q = k, q


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D,shared", [(128, 0), (64, 0), (128, 16)])
def test_rows_whose_maximum_jumps_between_chunks(dtype, D, shared):
    lens, qlens = [1100, 900, 700, 300], [1100, 300, 64, 300]
    w = workloads.make_prefill(B=4, Hq=8, Hkv=2, D=D, lens=lens, qlens=qlens, num_blocks=220,
                               dtype=dtype, seed=41 + D + shared, shared_blocks=shared)
    _plant_score_jumps(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, status=status, shared=shared)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                   w.query_start, w.scale)
    assert_close(out, ref, f"max jumps {dtype} D{D} shared {shared}")


def test_chunk_longer_than_context_sets_status_and_zeroes_rows():
    w = workloads.make_prefill(B=2, Hq=8, Hkv=2, D=64, lens=[40, 100], qlens=[40, 60],
                               num_blocks=20, dtype=torch.float16, seed=4)
    w.context_lens = torch.tensor([40, 50], dtype=torch.int32)  # request 1: L = 60 > n = 50
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, status)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert torch.count_nonzero(out[40:].float()) == 0
    ref = oracle.attention_prefill(w.q[:40], w.k_pool, w.v_pool, w.block_tables[:1],
                                   w.context_lens[:1], w.query_start[:2], w.scale)
    assert_close(out[:40], ref, "healthy request beside a bad one")


def test_bad_block_id_sets_status_and_zeroes_rows():
    w = workloads.make_prefill(B=2, Hq=4, Hkv=4, D=128, lens=[70, 90], qlens=[70, 20],
                               num_blocks=20, dtype=torch.bfloat16, seed=6)
    w.block_tables[1, 2] = 20  # == num_blocks: out of range
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, status)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert torch.count_nonzero(out[70:].float()) == 0
    assert torch.isfinite(out[:70].float()).all()


def test_max_query_len_too_small_sets_status():
    w = workloads.make_prefill(B=1, Hq=8, Hkv=1, D=128, lens=[300], qlens=[300],
                               num_blocks=20, dtype=torch.float16, seed=8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, status, max_query_len=100)  # grid covers 112 tokens of 300
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK


def test_empty_prefill_calls_are_no_ops():
    w = workloads.make_prefill(B=2, Hq=8, Hkv=2, D=64, lens=[30, 20], qlens=[0, 0],
                               num_blocks=8, dtype=torch.float16, seed=1)
    out = torch.full((1, 8, 64), 7.0, dtype=torch.float16, device="cuda")
    q = torch.zeros((1, 8, 64), dtype=torch.float16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, status, out=out, q=q)  # max_query_len 0: nothing launched
    run_gpu(w, status, max_query_len=16, out=out, q=q)  # launched, every chunk empty
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    assert bool((out == 7.0).all())  # nothing written


def test_prefill_rejects_unsupported_groups():
    w = workloads.make_prefill(B=1, Hq=12, Hkv=4, D=64, lens=[20], qlens=[20],
                               num_blocks=4, dtype=torch.float16, seed=1)  # G = 3
    with pytest.raises(kvp.KvpError) as e:
        run_gpu(w)
    assert e.value.status == kvp.KVP_ERR_UNSUPPORTED


def test_prefix_prefill_workload_full_size_sampled():
    """The benchmarked prefix-cached prompt pass at full size (128 requests,
    33K query tokens, 1030-token shared prefix), through the same call the
    bench times: every head of each request's first and last query rows and a
    random sample of the rest, against the oracle."""
    w = workloads.make_prefill_named("prefix_prefill", device="cuda", nan_sentinel=True)
    out = torch.empty((w.T, w.Hq, w.D), dtype=w.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvp.kvp_attention_prefill(out, w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                              w.query_start, w.max_query_len, w.scale, status=status)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    # every head of each request's first and last query rows (the fewest and
    # the most attended keys, at both ends of every tile walk), plus a seeded
    # random sample of interior (row, head) pairs
    qs = w.query_start.cpu().numpy()
    ends = np.unique(np.concatenate([qs[:-1], qs[1:] - 1]))
    t = np.repeat(ends, w.Hq)
    h = np.tile(np.arange(w.Hq), len(ends))
    rng = np.random.default_rng(17)
    t = np.concatenate([t, rng.integers(0, w.T, size=2048)])
    h = np.concatenate([h, rng.integers(0, w.Hq, size=2048)])
    rows = np.stack([t, h], axis=1).astype(np.int32)
    ref = oracle.attention_prefill(w.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(),
                                   w.block_tables.cpu(), w.context_lens.cpu(),
                                   w.query_start.cpu(), w.scale, rows=rows)
    got = out.cpu()[torch.from_numpy(t).long(), torch.from_numpy(h).long()]
    assert_close(got, ref, "prefix_prefill sampled")


def test_context_beyond_the_staged_table():
    """A 17000-token context (1063 blocks) reaches past the 128 block ids the
    softmax warps load ahead for their range check (the rest are checked at
    the tile's end) and past any short table.  Sampled rows against the
    oracle."""
    w = workloads.make_prefill(B=2, Hq=8, Hkv=2, D=128, lens=[17000, 300], qlens=[150, 300],
                               num_blocks=1100, dtype=torch.float16, seed=31)
    out = run_gpu(w)
    rng = np.random.default_rng(5)
    t = rng.integers(0, w.T, size=64)
    t[:3] = [0, 149, 150]
    h = rng.integers(0, w.Hq, size=64)
    rows = np.stack([t, h], axis=1).astype(np.int32)
    ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                   w.query_start, w.scale, rows=rows)
    got = out.cpu()[torch.from_numpy(t).long(), torch.from_numpy(h).long()]
    assert_close(got, ref, "context beyond the staged table")


def test_rows_past_num_query_tokens_set_status_and_write_nothing():
    """query_start says request 1 owns rows 40..99 but q / out hold 60 rows:
    the request is skipped (status), request 0 is computed normally."""
    w = workloads.make_prefill(B=2, Hq=8, Hkv=2, D=128, lens=[40, 100], qlens=[40, 60],
                               num_blocks=20, dtype=torch.float16, seed=12)
    q = w.q[:60].clone()
    out = torch.full((60, w.Hq, w.D), 5.0, dtype=w.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, status, out=out, q=q)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert bool((out[40:] == 5.0).all())
    ref = oracle.attention_prefill(w.q[:40], w.k_pool, w.v_pool, w.block_tables[:1],
                                   w.context_lens[:1], w.query_start[:2], w.scale)
    assert_close(out[:40], ref, "request before the overflowing one")


def test_sparse_work_list_spans_several_windows():
    """100 requests with G = 8 and one 1024-token chunk among chunks of at most
    64 tokens: max_query_len makes 64 tiles per (request, kv head), 51 200 work
    items, so each persistent block scans more than one window of candidates
    and skips most of them.  Sampled rows (every request's first and last row
    among them) against the oracle."""
    rng = np.random.default_rng(41)
    qlens = [int(x) for x in rng.integers(1, 65, size=100)]
    qlens[37] = 1024
    lens = [q + int(p) for q, p in zip(qlens, rng.integers(0, 200, size=100))]
    nb = sum(-(-n // 16) for n in lens) + 8
    w = workloads.make_prefill(B=100, Hq=64, Hkv=8, D=64, lens=lens, qlens=qlens, num_blocks=nb,
                               dtype=torch.float16, seed=43)
    assert w.max_query_len == 1024
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, status)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    qs = w.query_start.cpu().numpy()
    t = list(rng.integers(0, w.T, size=128)) + [int(x) for x in qs[:-1]] + \
        [int(x) - 1 for x in qs[1:]]
    h = list(rng.integers(0, w.Hq, size=len(t)))
    rows = np.stack([np.array(t), np.array(h)], axis=1).astype(np.int32)
    ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                   w.query_start, w.scale, rows=rows)
    got = out.cpu()[torch.tensor(t).long(), torch.tensor(h).long()]
    assert_close(got, ref, "sparse work list")


# --------------------------------------------------------------- shared prefix (dense tiles)
def _same_bits(a, b):
    return torch.equal(a.cpu().view(torch.int16), b.cpu().view(torch.int16))


SHARED_CASES = [  # (context length, chunk length) with a 16-block (256-token) shared prefix
    [(300, 40), (1100, 200), (260, 4), (520, 130), (256, 0), (700, 1), (1000, 300)],
    # chunks that start inside the shared prefix (causal masking on shared chunks)
    [(300, 100), (257, 257), (400, 150), (290, 64)],
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 128), (16, 4, 64), (32, 4, 128), (8, 1, 64)])
@pytest.mark.parametrize("case", [0, 1])
def test_shared_prefix_dense_tiles_equal_per_request_tiles(dtype, Hq, Hkv, D, case):
    """Dense tiles (rows of several requests in one 128-row tile, the shared
    prefix's chunks read once per tile) against per-request tiles, bit for
    bit, and against the oracle."""
    lens = [n for n, _ in SHARED_CASES[case]]
    qlens = [q for _, q in SHARED_CASES[case]]
    w = workloads.make_prefill(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, lens=lens, qlens=qlens,
                               num_blocks=260, dtype=dtype, shared_blocks=16,
                               seed=D + Hq + case, contiguous_p=0.5)
    per_request = run_gpu(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dense = run_gpu(w, status=status, shared=16)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    assert _same_bits(dense, per_request), "dense tiles differ from per-request tiles"
    ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                   w.query_start, w.scale)
    assert_close(dense, ref, f"dense {dtype} {Hq}/{Hkv} D{D} case {case}")


def test_shared_prefix_disagreeing_table_sets_status_and_zeroes_its_tiles():
    lens, qlens = [300, 400, 280, 350], [60, 300, 50, 90]
    w = workloads.make_prefill(B=4, Hq=8, Hkv=2, D=64, lens=lens, qlens=qlens, num_blocks=120,
                               dtype=torch.float16, shared_blocks=12, seed=4)
    # request 2 names one of its private blocks inside the shared prefix
    w.block_tables[2, 5] = int(w.block_tables[2, 17])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, status=status, shared=12)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    qs = w.query_start.tolist()
    assert torch.count_nonzero(out[qs[2]:qs[3]].float()) == 0  # request 2's rows
    # request 0 shares no 128-row tile with request 2 (G = 4: 32 tokens a tile)
    ref = oracle.attention_prefill(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                   w.query_start, w.scale)
    assert_close(out[:qs[1]], ref[:qs[1]], "rows of a request in good tiles")


def test_shared_prefix_longer_than_a_context_sets_status():
    w = workloads.make_prefill(B=2, Hq=8, Hkv=2, D=64, lens=[300, 260], qlens=[30, 20],
                               num_blocks=60, dtype=torch.float16, shared_blocks=16, seed=6)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(w, status=status, shared=17)  # 17 blocks = 272 tokens > 260
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK


def test_prefix_prefill_workload_dense_tiles_full_size():
    """The benchmarked prompt pass with its 64 shared prefix blocks: dense
    tiles equal per-request tiles bit for bit at full size (33 098 query
    tokens of 128 requests), and every head of each request's first and last
    rows matches the oracle."""
    w = workloads.make_prefill_named("prefix_prefill", device="cuda", nan_sentinel=True)
    S = w.info["shared_blocks"]
    out_pr = torch.empty((w.T, w.Hq, w.D), dtype=w.dtype, device="cuda")
    out_dn = torch.empty_like(out_pr)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for out, shared in ((out_pr, 0), (out_dn, S)):
        kvp.kvp_attention_prefill(out, w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                                  w.query_start, w.max_query_len, w.scale,
                                  shared_prefix_blocks=shared, status=status)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    assert _same_bits(out_dn, out_pr)
    qs = w.query_start.cpu().numpy()
    ends = np.unique(np.concatenate([qs[:-1], qs[1:] - 1]))
    rows = np.stack([np.repeat(ends, w.Hq), np.tile(np.arange(w.Hq), len(ends))],
                    axis=1).astype(np.int32)
    ref = oracle.attention_prefill(w.q.cpu(), w.k_pool.cpu(), w.v_pool.cpu(),
                                   w.block_tables.cpu(), w.context_lens.cpu(),
                                   w.query_start.cpu(), w.scale, rows=rows)
    got = out_dn.cpu()[torch.from_numpy(rows[:, 0]).long(), torch.from_numpy(rows[:, 1]).long()]
    assert_close(got, ref, "prefix_prefill dense tiles")
