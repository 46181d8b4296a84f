"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle
on the same seeded inputs.

Bars: append, copy_blocks and INT8 quantisation bit-exact; attention outputs
(fp32 accumulation, fp16/bf16 out) within 3e-3 absolute OR 1e-2 relative of the
fp64 oracle, element by element.  Inputs given to the oracle never come from
the GPU: the oracle applies its own copy/append/quantise to the host pools.
"""
import math

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


def assert_attn_close(gpu_out, ref, what=""):
    g = gpu_out.detach().double().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    ok = (err <= ATOL) | (err <= RTOL * np.abs(ref))
    if not ok.all():
        i = np.unravel_index(np.argmax(np.where(ok, 0, err)), err.shape)
        raise AssertionError(f"{what}: {int((~ok).sum())} elements out of tolerance; worst at "
                             f"{i}: gpu {g[i]} ref {ref[i]} (max abs err {err.max():.3e})")


def workspace_for(w, partition_blocks=0, fp8=False):
    d = kvp.kvp_cache_desc(w.num_blocks, w.Hkv, 16, w.D)
    nbytes = kvp.kvp_decode_workspace_bytes(w.B, w.Hq, d, w.max_blocks, partition_blocks,
                                            w.kv_int8 and not fp8, fp8)
    if nbytes == 0:
        return None
    return torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")


def gpu_decode_16(w, partition_blocks=0, status=None):
    """copy-on-write pairs, append, decode: the whole 16-bit step on the GPU."""
    kp = w.k_pool.cuda()
    vp = w.v_pool.cuda()
    if w.cow_pairs is not None:
        kvp.kvp_copy_blocks(kp, vp, w.cow_pairs.cuda(), status=status)
    kvp.kvp_append(w.new_k.cuda(), w.new_v.cuda(), kp, vp, w.slot_mapping.cuda(), status=status)
    out = torch.full_like(w.q, float("nan"), device="cuda")
    kvp.kvp_attention_decode(out, w.q.cuda(), kp, vp, w.block_tables.cuda(),
                             w.context_lens.cuda(), w.scale,
                             workspace=workspace_for(w, partition_blocks),
                             partition_blocks=partition_blocks, status=status)
    torch.cuda.synchronize()
    return out, kp, vp


def oracle_pools_16(w):
    kp, vp = w.k_pool, w.v_pool
    if w.cow_pairs is not None:
        kp = oracle.copy_blocks(kp, w.cow_pairs)
        vp = oracle.copy_blocks(vp, w.cow_pairs)
    kp = oracle.append(kp, w.new_k, w.slot_mapping)
    vp = oracle.append(vp, w.new_v, w.slot_mapping)
    return kp, vp


def same_bits(a, b):
    a = a.detach().cpu().contiguous()
    b = b.detach().cpu().contiguous()
    if a.dtype in (torch.float16, torch.bfloat16):
        a, b = a.view(torch.int16), b.view(torch.int16)
    elif a.dtype == torch.float32:
        a, b = a.view(torch.int32), b.view(torch.int32)
    return torch.equal(a, b)


# --------------------------------------------------------------- tiny workload
def test_tiny_workload_full_parity():
    w = workloads.make("tiny")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, kp, vp = gpu_decode_16(w, status=status)
    assert kvp.kvp_read_status(status) == kvp.KVP_OK
    okp, ovp = oracle_pools_16(w)
    assert same_bits(kp, okp) and same_bits(vp, ovp)  # append is a byte scatter
    ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
    assert_attn_close(out, ref, "tiny")
    # context_len 1 returns V_0 exactly
    blk = int(w.block_tables[0, 0])
    v0 = ovp[blk, :, 0, :]  # [Hkv, D]
    G = w.Hq // w.Hkv
    for h in range(w.Hq):
        assert same_bits(out[0, h].cpu(), v0[h // G])


# --------------------------------------------------------------- shape sweep
SWEEP = []
for dtype in (torch.float16, torch.bfloat16):
    for D in (64, 128):
        for Hq, Hkv in ((4, 4), (8, 4), (12, 4), (16, 2), (8, 1), (24, 2)):
            SWEEP.append((dtype, D, Hq, Hkv))


@pytest.mark.parametrize("dtype,D,Hq,Hkv", SWEEP)
@pytest.mark.parametrize("partition_blocks", [0, 8, 3])
def test_decode_shape_sweep(dtype, D, Hq, Hkv, partition_blocks):
    lens = [1, 15, 16, 17, 100, 257, 530, 0, 48]
    w = workloads.make_custom(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, lens=lens, num_blocks=160,
                              dtype=dtype, seed=hash((D, Hq, Hkv)) % 1000, max_blocks=40)
    out, kp, vp = gpu_decode_16(w, partition_blocks)
    okp, ovp = oracle_pools_16(w)
    assert same_bits(kp, okp) and same_bits(vp, ovp)
    ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
    assert_attn_close(out, ref, f"{dtype} D{D} {Hq}/{Hkv} pb{partition_blocks}")
    assert torch.count_nonzero(out[7]) == 0  # context 0 -> zero row


def test_scattered_vs_contiguous_tables_agree_with_oracle():
    lens = [700, 1500, 64]
    for p in (0.0, 0.85, 1.0):
        w = workloads.make_custom(B=3, Hq=8, Hkv=1, D=128, lens=lens, num_blocks=200,
                                  dtype=torch.bfloat16, contiguous_p=p, seed=3)
        out, _, _ = gpu_decode_16(w)
        okp, ovp = oracle_pools_16(w)
        ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
        assert_attn_close(out, ref, f"contiguity {p}")


def test_split_phases_equal_single_call():
    w = workloads.make_custom(B=3, Hq=16, Hkv=2, D=128, lens=[900, 33, 2000], num_blocks=300,
                              dtype=torch.float16, seed=4)
    out_all, kp, vp = gpu_decode_16(w, 16)
    out = torch.zeros_like(out_all)
    ws = workspace_for(w, 16)
    args = (out, w.q.cuda(), kp, vp, w.block_tables.cuda(), w.context_lens.cuda(), w.scale)
    kvp.kvp_attention_decode(*args, workspace=ws, partition_blocks=16,
                             phases=kvp.KVP_PHASE_PARTIAL)
    kvp.kvp_attention_decode(*args, workspace=ws, partition_blocks=16,
                             phases=kvp.KVP_PHASE_REDUCE)
    torch.cuda.synchronize()
    assert same_bits(out, out_all)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_warp_reduce_equals_cta_reduce(dtype, D):
    """Rows are merged by one warp each when no row can have more than 8
    partitions (max_blocks / partition_blocks <= 8), by a CTA each otherwise;
    both write the same bits, so the same workload with its table padded past
    8 partitions' width gives the same output."""
    lens = [1024, 1000, 513, 17, 129, 0, 777]
    w = workloads.make_custom(B=len(lens), Hq=16, Hkv=2, D=D, lens=lens, num_blocks=400,
                              dtype=dtype, seed=D + 13, max_blocks=64)
    out_warp, _, _ = gpu_decode_16(w, 8)
    w.block_tables = torch.cat([w.block_tables, torch.zeros((w.B, 8), dtype=torch.int32)], 1)
    assert w.max_blocks == 72
    out_cta, kp, vp = gpu_decode_16(w, 8)
    assert same_bits(out_warp, out_cta)
    okp, ovp = oracle_pools_16(w)
    ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
    assert_attn_close(out_warp, ref, f"warp reduce {dtype} D{D}")


def test_decode_is_deterministic():
    w = workloads.make_custom(B=4, Hq=8, Hkv=8, D=128, lens=[4000, 10, 2500, 1234],
                              num_blocks=700, dtype=torch.float16, seed=8)
    a, _, _ = gpu_decode_16(w)
    b, _, _ = gpu_decode_16(w)
    assert same_bits(a, b)


# --------------------------------------------------------------- copy_blocks
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.int8])
def test_copy_blocks_bit_exact(dtype):
    g = torch.Generator().manual_seed(2)
    NB, Hkv, D = 40, 4, 128
    if dtype == torch.int8:
        kp = torch.randint(-128, 128, (NB, Hkv, 16, D), generator=g, dtype=torch.int8)
        vp = torch.randint(-128, 128, (NB, Hkv, 16, D), generator=g, dtype=torch.int8)
        ks = torch.rand(NB, Hkv, 16, generator=g)
        vs = torch.rand(NB, Hkv, 16, generator=g)
    else:
        kp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
        vp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
        ks = vs = None
    pairs = torch.tensor([[3, 10], [3, 11], [7, 0], [5, 5], [39, 20]], dtype=torch.int32)
    gk, gv = kp.cuda(), vp.cuda()
    gks = ks.cuda() if ks is not None else None
    gvs = vs.cuda() if vs is not None else None
    kvp.kvp_copy_blocks(gk, gv, pairs.cuda(), k_scale=gks, v_scale=gvs)
    torch.cuda.synchronize()
    assert same_bits(gk, oracle.copy_blocks(kp, pairs))
    assert same_bits(gv, oracle.copy_blocks(vp, pairs))
    if ks is not None:
        assert same_bits(gks, oracle.copy_blocks(ks, pairs))
        assert same_bits(gvs, oracle.copy_blocks(vs, pairs))


# --------------------------------------------------------------- INT8
@pytest.mark.parametrize("src_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_append_int8_bit_exact(src_dtype, D):
    g = torch.Generator().manual_seed(31)
    NB, Hkv, T = 64, 4, 300
    key = (torch.randn(T, Hkv, D, generator=g) * torch.rand(T, Hkv, 1, generator=g) * 4)
    value = torch.randn(T, Hkv, D, generator=g)
    key[5] = 0.0                           # all-zero rows keep scale 1
    key[6, :, :3] = 2.5
    # abs-max 127 gives scale exactly 1, so x.5 entries are exact ties (-> even)
    ties = (torch.arange(D, dtype=torch.float32) - D / 2) + 0.5
    ties[0] = 127.0
    key[8] = ties
    value[9] = -ties
    key, value = key.to(src_dtype), value.to(src_dtype)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int32)
    slots[7] = -1                          # padding token
    kc = torch.zeros(NB, Hkv, 16, D, dtype=torch.int8)
    vc = torch.zeros_like(kc)
    ks = torch.full((NB, Hkv, 16), -7.0)
    vs = torch.full((NB, Hkv, 16), -7.0)
    gkc, gvc, gks, gvs = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    kvp.kvp_append_int8(key.cuda(), value.cuda(), gkc, gvc, gks, gvs, slots.cuda())
    torch.cuda.synchronize()
    okc, oks = oracle.append_int8(kc, ks, key, slots)
    ovc, ovs = oracle.append_int8(vc, vs, value, slots)
    assert same_bits(gkc, okc) and same_bits(gks, oks)
    assert same_bits(gvc, ovc) and same_bits(gvs, ovs)


def _tie_rows(src_dtype, D, n_rows, seed):
    """Rows that put many elements on or next to a half-integer of x / scale:
    (a) amax = 127 * 2^e, so scale = 2^e exactly and (k + 1/2) * 2^e are exact
    ties; (b) the same values moved by one unit in the last place either way;
    (c) arbitrary maxima with elements rounded from (k + 1/2) * amax / 127,
    which land within a few units in the last place of a tie."""
    g = torch.Generator().manual_seed(seed)
    rows = torch.empty(n_rows, D, dtype=torch.float32)
    for r in range(n_rows):
        kind = r % 3
        e = int(torch.randint(-10, 6, (1,), generator=g))
        k = torch.randint(-127, 127, (D,), generator=g).float()
        if kind < 2:
            x = ((k + 0.5) * 2.0 ** e).to(src_dtype)
            if kind == 1:  # one unit in the last place up or down
                bits = x.view(torch.int16)
                step = torch.randint(0, 2, (D,), generator=g, dtype=torch.int16) * 2 - 1
                x = (bits + step).view(src_dtype)
            x[0] = 127.0 * 2.0 ** e
        else:
            amax = float(torch.rand(1, generator=g)) * 30 + 0.01
            x = ((k + 0.5) * (amax / 127.0)).to(src_dtype)
            x[0] = -amax
        x = x.float()
        x = x[torch.randperm(D, generator=g)]  # the abs-max anywhere in the row
        rows[r] = x
    return rows.to(src_dtype)


@pytest.mark.parametrize("src_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_append_int8_ties_and_near_ties_bit_exact(src_dtype, D):
    """The quantiser's codes come from a rounded product on the fast path and
    from the IEEE quotient next to a half-integer; rows built on and around
    ties check both against the oracle's float32 division, bit for bit."""
    Hkv, NB = 2, 256
    x = _tie_rows(src_dtype, D, 2 * 1536, seed=D + (src_dtype == torch.bfloat16))
    key = x[:1536].view(768, Hkv, D)
    value = x[1536:].view(768, Hkv, D)
    T = key.shape[0]
    g = torch.Generator().manual_seed(5)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int32)
    kc = torch.zeros(NB, Hkv, 16, D, dtype=torch.int8)
    vc = torch.zeros_like(kc)
    ks = torch.zeros(NB, Hkv, 16)
    vs = torch.zeros(NB, Hkv, 16)
    gkc, gvc, gks, gvs = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    kvp.kvp_append_int8(key.cuda(), value.cuda(), gkc, gvc, gks, gvs, slots.cuda())
    torch.cuda.synchronize()
    okc, oks = oracle.append_int8(kc, ks, key, slots)
    ovc, ovs = oracle.append_int8(vc, vs, value, slots)
    assert same_bits(gks, oks) and same_bits(gvs, ovs)
    assert same_bits(gkc, okc) and same_bits(gvc, ovc)
    # the rows really exercise ties: many exact x.5 quotients among them
    q = key.float().view(-1, D) / torch.from_numpy(
        oracle.quantize_int8(key.view(-1, D))[1])[:, None]
    assert int(((q - q.floor()) == 0.5).sum()) > 1000


def int8_workload(B, Hq, Hkv, D, lens, NB, q_dtype, seed, max_blocks=None):
    w = workloads.make_custom(B=B, Hq=Hq, Hkv=Hkv, D=D, lens=lens, num_blocks=NB,
                              dtype=q_dtype, kv_int8=True, seed=seed, max_blocks=max_blocks)
    # the oracle quantises the fp16 source pools; unused scale slots hold NaN
    kc, ks = oracle.quantize_int8(w.k_pool)
    vc, vs = oracle.quantize_int8(w.v_pool)
    ks = torch.from_numpy(ks)
    vs = torch.from_numpy(vs)
    used = torch.zeros(NB, 16, dtype=torch.bool)
    for b, n in enumerate(lens):
        for i in range(n):
            used[int(w.block_tables[b, i // 16]), i % 16] = True
    ks[~used[:, None, :].expand_as(ks)] = float("nan")
    vs[~used[:, None, :].expand_as(vs)] = float("nan")
    return w, torch.from_numpy(kc), torch.from_numpy(vc), ks, vs


def gpu_decode_int8(w, kc, vc, ks, vs, partition_blocks=0):
    gkc, gvc, gks, gvs = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    kvp.kvp_append_int8(w.new_k.cuda(), w.new_v.cuda(), gkc, gvc, gks, gvs, w.slot_mapping.cuda())
    out = torch.full_like(w.q, float("nan"), device="cuda")
    kvp.kvp_attention_decode_int8(out, w.q.cuda(), gkc, gvc, gks, gvs, w.block_tables.cuda(),
                                  w.context_lens.cuda(), w.scale,
                                  workspace=workspace_for(w, partition_blocks),
                                  partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    return out, gkc, gvc, gks, gvs


@pytest.mark.parametrize("q_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (16, 2), (4, 4), (6, 2)])
@pytest.mark.parametrize("partition_blocks", [0, 8])
def test_decode_int8_parity(q_dtype, D, Hq, Hkv, partition_blocks):
    lens = [1, 17, 300, 16, 640, 0]
    w, kc, vc, ks, vs = int8_workload(len(lens), Hq, Hkv, D, lens, 120, q_dtype,
                                      seed=D + Hq, max_blocks=40)
    out, gkc, gvc, gks, gvs = gpu_decode_int8(w, kc, vc, ks, vs, partition_blocks)
    okc, oks = oracle.append_int8(kc, ks, w.new_k, w.slot_mapping)
    ovc, ovs = oracle.append_int8(vc, vs, w.new_v, w.slot_mapping)
    assert same_bits(gkc, okc) and same_bits(gvc, ovc)
    assert same_bits(gks, oks) and same_bits(gvs, ovs)
    ref = oracle.attention_decode(w.q, okc, ovc, w.block_tables, w.context_lens, w.scale,
                                  k_scale=oks, v_scale=ovs)
    assert_attn_close(out, ref, f"int8 {q_dtype} D{D} {Hq}/{Hkv} pb{partition_blocks}")


# --------------------------------------------------------------- device errors
def test_bad_block_id_sets_status_and_zeroes_rows():
    w = workloads.make_custom(B=3, Hq=8, Hkv=2, D=64, lens=[40, 300, 20], num_blocks=64,
                              dtype=torch.float16, seed=9)
    w.block_tables[1, 5] = 64        # out of range
    w.block_tables[2, 0] = -3
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _, _ = gpu_decode_16(w, 8, status=status)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert torch.count_nonzero(out[1]) == 0 and torch.count_nonzero(out[2]) == 0
    okp, ovp = oracle_pools_16(w)
    ref = oracle.attention_decode(w.q[:1], okp, ovp, w.block_tables[:1], w.context_lens[:1],
                                  w.scale)
    assert_attn_close(out[:1], ref, "healthy request next to bad ones")


def test_context_longer_than_table_sets_status():
    w = workloads.make_custom(B=2, Hq=4, Hkv=4, D=128, lens=[20, 30], num_blocks=16,
                              dtype=torch.float16, seed=10)
    lens = w.context_lens.clone()
    lens[1] = w.max_blocks * 16 + 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp, vp = w.k_pool.cuda(), w.v_pool.cuda()
    out = torch.full_like(w.q, 1.0, device="cuda")
    kvp.kvp_attention_decode(out, w.q.cuda(), kp, vp, w.block_tables.cuda(), lens.cuda(),
                             w.scale, workspace=workspace_for(w), status=status)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert torch.count_nonzero(out[1]) == 0


def test_append_slot_out_of_range_sets_status_and_skips():
    kp = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    vp = torch.zeros_like(kp)
    key = torch.ones(3, 2, 64, dtype=torch.float16, device="cuda")
    slots = torch.tensor([3, 64, -1], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvp.kvp_append(key, key, kp, vp, slots, status=status)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert torch.count_nonzero(kp) == 2 * 64 and bool((kp[0, :, 3] == 1).all())


def test_empty_inputs_are_no_ops():
    kp = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    key = torch.zeros(0, 2, 64, dtype=torch.float16, device="cuda")
    kvp.kvp_append(key, key, kp, kp.clone(), torch.zeros(0, dtype=torch.int32, device="cuda"))
    pairs = torch.zeros(0, 2, dtype=torch.int32, device="cuda")
    kvp.kvp_copy_blocks(kp, kp.clone(), pairs)
    q = torch.zeros(0, 8, 64, dtype=torch.float16, device="cuda")
    kvp.kvp_attention_decode(q.clone(), q, kp, kp, torch.zeros(0, 4, dtype=torch.int32,
                                                               device="cuda"),
                             torch.zeros(0, dtype=torch.int32, device="cuda"), 0.1)
    torch.cuda.synchronize()


# --------------------------------------------------------------- FP8 (E4M3) and per-tensor INT8
@pytest.mark.parametrize("src_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_append_fp8_bit_exact(src_dtype, D):
    g = torch.Generator().manual_seed(51)
    NB, Hkv, T = 64, 4, 300
    key = (torch.randn(T, Hkv, D, generator=g) * torch.rand(T, Hkv, 1, generator=g) * 4)
    value = torch.randn(T, Hkv, D, generator=g) * 0.01
    key[5] = 0.0
    key, value = key.to(src_dtype), value.to(src_dtype)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int32)
    slots[7] = -1
    kc = torch.zeros(NB, Hkv, 16, D, dtype=torch.uint8)
    vc = torch.zeros_like(kc)
    ks = torch.full((NB, Hkv, 16), -7.0)
    vs = torch.full((NB, Hkv, 16), -7.0)
    gkc, gvc, gks, gvs = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    kvp.kvp_append_fp8(key.cuda(), value.cuda(), gkc, gvc, gks, gvs, slots.cuda())
    torch.cuda.synchronize()
    okc, oks = oracle.append_fp8(kc.view(torch.float8_e4m3fn), ks, key, slots)
    ovc, ovs = oracle.append_fp8(vc.view(torch.float8_e4m3fn), vs, value, slots)
    assert torch.equal(gkc.cpu(), okc.view(torch.uint8)) and same_bits(gks, oks)
    assert torch.equal(gvc.cpu(), ovc.view(torch.uint8)) and same_bits(gvs, ovs)


@pytest.mark.parametrize("src_dtype", [torch.float16, torch.bfloat16])
def test_append_int8_fixed_scale_bit_exact(src_dtype):
    g = torch.Generator().manual_seed(52)
    NB, Hkv, D, T = 32, 2, 128, 200
    key = (torch.randn(T, Hkv, D, generator=g) * 3).to(src_dtype)
    key[0, 0, :4] = torch.tensor([1e4, -1e4, 6.0, -6.1])   # clip both ways
    value = (torch.randn(T, Hkv, D, generator=g)).to(src_dtype)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int32)
    kc = torch.zeros(NB, Hkv, 16, D, dtype=torch.int8)
    vc = torch.zeros_like(kc)
    ks = torch.zeros(NB, Hkv, 16)
    vs = torch.zeros(NB, Hkv, 16)
    gkc, gvc, gks, gvs = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    kvp.kvp_append_int8_fixed(key.cuda(), value.cuda(), gkc, gvc, gks, gvs, 0.05, 0.0125,
                              slots.cuda())
    torch.cuda.synchronize()
    okc, oks = oracle.append_int8_fixed(kc, ks, key, slots, 0.05)
    ovc, ovs = oracle.append_int8_fixed(vc, vs, value, slots, 0.0125)
    assert same_bits(gkc, okc) and same_bits(gks, oks)
    assert same_bits(gvc, ovc) and same_bits(gvs, ovs)
    assert int(gkc.cpu().view(-1).max()) == 127 and int(gkc.cpu().view(-1).min()) == -128


def fp8_workload(B, Hq, Hkv, D, lens, NB, q_dtype, seed, max_blocks=None):
    w = workloads.make_custom(B=B, Hq=Hq, Hkv=Hkv, D=D, lens=lens, num_blocks=NB,
                              dtype=q_dtype, kv_int8=True, seed=seed, max_blocks=max_blocks)
    kc, ks = oracle.quantize_fp8(w.k_pool)
    vc, vs = oracle.quantize_fp8(w.v_pool)
    ks, vs = torch.from_numpy(ks), torch.from_numpy(vs)
    used = torch.zeros(NB, 16, dtype=torch.bool)
    for b, n in enumerate(lens):
        for i in range(n):
            used[int(w.block_tables[b, i // 16]), i % 16] = True
    ks[~used[:, None, :].expand_as(ks)] = float("nan")
    vs[~used[:, None, :].expand_as(vs)] = float("nan")
    # unused slots hold E4M3 NaN codes (0x7f, 0xff): an over-read, or a V code
    # of a token past the context reaching the product, turns the output NaN
    kc, vc = torch.from_numpy(kc), torch.from_numpy(vc)
    unused = (~used)[:, None, :, None].expand_as(kc)
    nan_codes = torch.where(torch.arange(D) % 2 == 0, 0x7f, 0xff).to(torch.uint8)
    kc[unused] = nan_codes.expand_as(kc)[unused]
    vc[unused] = nan_codes.expand_as(vc)[unused]
    return w, kc, vc, ks, vs


@pytest.mark.parametrize("q_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (16, 2), (4, 4), (6, 2)])
@pytest.mark.parametrize("partition_blocks", [0, 8])
def test_decode_fp8_parity(q_dtype, D, Hq, Hkv, partition_blocks):
    lens = [1, 17, 300, 16, 640, 0]
    w, kc, vc, ks, vs = fp8_workload(len(lens), Hq, Hkv, D, lens, 120, q_dtype,
                                     seed=D + Hq + 5, max_blocks=40)
    gkc, gvc, gks, gvs = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
    kvp.kvp_append_fp8(w.new_k.cuda(), w.new_v.cuda(), gkc, gvc, gks, gvs, w.slot_mapping.cuda())
    out = torch.full_like(w.q, float("nan"), device="cuda")
    kvp.kvp_attention_decode_fp8(out, w.q.cuda(), gkc, gvc, gks, gvs, w.block_tables.cuda(),
                                 w.context_lens.cuda(), w.scale,
                                 workspace=workspace_for(w, partition_blocks, fp8=True),
                                 partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    okc, oks = oracle.append_fp8(kc.view(torch.float8_e4m3fn), ks, w.new_k, w.slot_mapping)
    ovc, ovs = oracle.append_fp8(vc.view(torch.float8_e4m3fn), vs, w.new_v, w.slot_mapping)
    assert torch.equal(gkc.cpu(), okc.view(torch.uint8))
    assert torch.equal(gvc.cpu(), ovc.view(torch.uint8))
    ref = oracle.attention_decode(w.q, okc, ovc, w.block_tables, w.context_lens, w.scale,
                                  k_scale=oks, v_scale=ovs)
    assert_attn_close(out, ref, f"fp8 {q_dtype} D{D} {Hq}/{Hkv} pb{partition_blocks}")


# --------------------------------------------------------------- fused append + decode
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 128), (16, 2, 64), (24, 2, 128), (8, 1, 128)])
@pytest.mark.parametrize("partition_blocks", [0, 8])
def test_fused_append_decode_equals_separate_calls(dtype, Hq, Hkv, D, partition_blocks):
    lens = [1, 16, 17, 300, 0, 530]
    w = workloads.make_custom(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, lens=lens, num_blocks=120,
                              dtype=dtype, seed=Hq * 7 + D, max_blocks=40)
    out_sep, kp_sep, vp_sep = gpu_decode_16(w, partition_blocks)
    # one new row per request (rows of requests with no context are ignored)
    key = torch.zeros(w.B, w.Hkv, w.D, dtype=dtype)
    val = torch.zeros_like(key)
    active = [b for b in range(w.B) if lens[b] > 0]
    key[active] = w.new_k
    val[active] = w.new_v
    kp, vp = w.k_pool.cuda(), w.v_pool.cuda()
    out = torch.full_like(w.q, float("nan"), device="cuda")
    kvp.kvp_append_attention_decode(key.cuda(), val.cuda(), out, w.q.cuda(), kp, vp,
                                    w.block_tables.cuda(), w.context_lens.cuda(), w.scale,
                                    workspace=workspace_for(w, partition_blocks),
                                    partition_blocks=partition_blocks)
    torch.cuda.synchronize()
    assert same_bits(kp, kp_sep) and same_bits(vp, vp_sep)
    assert same_bits(out, out_sep)
    okp, ovp = oracle_pools_16(w)
    ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
    assert_attn_close(out, ref, f"fused {dtype} {Hq}/{Hkv} D{D} pb{partition_blocks}")


# --------------------------------------------------------------- run-merged fetch
MERGE_CASES = [  # (kind, dtype, D, Hq, Hkv): every consumer of the decode
    ("16", torch.float16, 128, 4, 4),     # CUDA cores, one query head per kv head
    ("16", torch.bfloat16, 64, 16, 8),    # CUDA cores, two heads
    ("16", torch.bfloat16, 128, 16, 2),   # tensor cores, 8 heads
    ("16", torch.float16, 64, 24, 2),     # tensor cores, 12 heads (two query groups)
    ("int8", torch.float16, 128, 16, 2),
    ("int8", torch.bfloat16, 64, 8, 1),
    ("fp8", torch.float16, 128, 16, 2),
    ("fp8", torch.bfloat16, 64, 6, 2),
]


@pytest.mark.parametrize("kind,dtype,D,Hq,Hkv", MERGE_CASES)
@pytest.mark.parametrize("p_run", [0.0, 0.85, 1.0])
@pytest.mark.parametrize("partition_blocks", [0, 6])
def test_merged_run_fetch_equals_per_block_fetch(kind, dtype, D, Hq, Hkv, p_run,
                                                 partition_blocks):
    """KVP_DECODE_MERGE_RUNS fetches runs of up to 4 physically consecutive
    blocks with one copy each; every warp still consumes the same blocks in the
    same order, so the output must equal the per-block fetch bit for bit, and
    the oracle within tolerance.  Tables are scattered (no runs), 85% runs,
    and one run per request; lengths put partial groups and partial blocks at
    the ends of partitions."""
    lens = [1, 16, 17, 64, 65, 300, 530, 0, 611]
    w = workloads.make_custom(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, lens=lens, num_blocks=200,
                              dtype=dtype, kv_int8=kind != "16", contiguous_p=p_run,
                              seed=D + Hq + int(10 * p_run), max_blocks=48)
    ws = workspace_for(w, partition_blocks, fp8=kind == "fp8")
    outs = []
    if kind == "16":
        kp, vp = w.k_pool.cuda(), w.v_pool.cuda()
        kvp.kvp_append(w.new_k.cuda(), w.new_v.cuda(), kp, vp, w.slot_mapping.cuda())
        for flags in (0, kvp.KVP_DECODE_MERGE_RUNS):
            out = torch.full_like(w.q, float("nan"), device="cuda")
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            kvp.kvp_attention_decode(out, w.q.cuda(), kp, vp, w.block_tables.cuda(),
                                     w.context_lens.cuda(), w.scale, workspace=ws,
                                     partition_blocks=partition_blocks,
                                     phases=kvp.KVP_PHASE_ALL | flags, status=status)
            assert kvp.kvp_read_status(status) == kvp.KVP_OK
            outs.append(out)
        okp, ovp = oracle_pools_16(w)
        ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
    else:
        fp8 = kind == "fp8"
        quant = oracle.quantize_fp8 if fp8 else oracle.quantize_int8
        kc, ks = quant(w.k_pool)
        vc, vs = quant(w.v_pool)
        kc, vc = torch.from_numpy(kc), torch.from_numpy(vc)
        ks, vs = torch.from_numpy(ks), torch.from_numpy(vs)
        decode = kvp.kvp_attention_decode_fp8 if fp8 else kvp.kvp_attention_decode_int8
        gkc, gvc, gks, gvs = kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda()
        for flags in (0, kvp.KVP_DECODE_MERGE_RUNS):
            out = torch.full_like(w.q, float("nan"), device="cuda")
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            decode(out, w.q.cuda(), gkc, gvc, gks, gvs, w.block_tables.cuda(),
                   w.context_lens.cuda(), w.scale, workspace=ws,
                   partition_blocks=partition_blocks, phases=kvp.KVP_PHASE_ALL | flags,
                   status=status)
            assert kvp.kvp_read_status(status) == kvp.KVP_OK
            outs.append(out)
        if fp8:
            kc, vc = kc.view(torch.float8_e4m3fn), vc.view(torch.float8_e4m3fn)
        ref = oracle.attention_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                      k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert same_bits(outs[0], outs[1]), "run-merged fetch differs from per-block fetch"
    assert_attn_close(outs[1], ref, f"merged {kind} {dtype} D{D} {Hq}/{Hkv} p{p_run}")
    assert torch.count_nonzero(outs[1][7]) == 0  # context 0 -> zero row


def test_merged_run_fetch_bad_block_id_sets_status():
    w = workloads.make_custom(B=2, Hq=8, Hkv=2, D=128, lens=[300, 200], num_blocks=64,
                              dtype=torch.float16, contiguous_p=1.0, seed=12)
    kp, vp = w.k_pool.cuda(), w.v_pool.cuda()
    kvp.kvp_append(w.new_k.cuda(), w.new_v.cuda(), kp, vp, w.slot_mapping.cuda())
    okp, ovp = oracle_pools_16(w)
    w.block_tables[1, 3] = 64  # out of range, inside a run (after the appends)
    out = torch.full_like(w.q, float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvp.kvp_attention_decode(out, w.q.cuda(), kp, vp, w.block_tables.cuda(),
                             w.context_lens.cuda(), w.scale,
                             phases=kvp.KVP_PHASE_ALL | kvp.KVP_DECODE_MERGE_RUNS, status=status)
    assert kvp.kvp_read_status(status) == kvp.KVP_ERR_BAD_BLOCK
    assert torch.count_nonzero(out[1]) == 0
    ref = oracle.attention_decode(w.q[:1], okp, ovp, w.block_tables[:1], w.context_lens[:1],
                                  w.scale)
    assert_attn_close(out[:1], ref, "merged fetch, request with good ids")
