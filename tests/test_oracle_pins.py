"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: an exhaustive
enumeration, a library routine (torch float64 softmax / matmul, NumPy indexing),
a closed form, or the quantiser's definition written out in exact rational
arithmetic (plus properties any correct abs-max quantiser has).  A plausible slip in the oracle (wrong head group, dropped scale,
transposed operand, wrong slot arithmetic, wrong rounding) fails at least one.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

BS = 16


# ------------------------------------------------------------ 16-bit widening
def test_f16_widening_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    assert np.array_equal(np.signbit(ref[~np.isnan(ref)]), np.signbit(got[~np.isnan(got)]))


def test_bf16_widening_exhaustive():
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b) & 0xFFFF) for b in bits.tolist()])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


# ------------------------------------------------------------ attention helpers
def _paged_from_dense(K, V, lens, num_blocks, seed, fill=float("nan")):
    """Place dense per-request K/V [B, Hkv, n, D] into a pool through a random
    block table using NumPy-style indexing (independent of the oracle)."""
    B, Hkv, nmax, D = K.shape
    g = torch.Generator().manual_seed(seed)
    nblk = [-(-n // BS) for n in lens]
    perm = torch.randperm(num_blocks, generator=g)
    mb = max(1, max(nblk))
    tables = torch.full((B, mb), -1, dtype=torch.int32)
    kp = torch.full((num_blocks, Hkv, BS, D), fill, dtype=K.dtype)
    vp = torch.full((num_blocks, Hkv, BS, D), fill, dtype=V.dtype)
    at = 0
    for b in range(B):
        blocks = perm[at:at + nblk[b]]
        at += nblk[b]
        tables[b, :nblk[b]] = blocks.to(torch.int32)
        for i in range(lens[b]):
            kp[blocks[i // BS], :, i % BS, :] = K[b, :, i, :]
            vp[blocks[i // BS], :, i % BS, :] = V[b, :, i, :]
    return kp, vp, tables


def _dense_reference(q, K, V, lens, scale):
    """torch float64: softmax(q K^T scale) V per request, K/V heads repeated
    for the query-head groups (library routines only)."""
    B, Hq, D = q.shape
    Hkv = K.shape[1]
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        n = lens[b]
        if n == 0:
            continue
        k = K[b, :, :n].double().repeat_interleave(Hq // Hkv, dim=0)  # [Hq, n, D]
        v = V[b, :, :n].double().repeat_interleave(Hq // Hkv, dim=0)
        s = torch.einsum("hd,hnd->hn", q[b].double(), k) * scale
        p = torch.softmax(s, dim=-1)
        out[b] = torch.einsum("hn,hnd->hd", p, v)
    return out


CASES = [
    # B, Hq, Hkv, D, lens, dtype
    (3, 4, 4, 64, [1, 16, 37], torch.float16),
    (2, 8, 2, 64, [33, 100], torch.float16),
    (2, 8, 1, 128, [17, 64], torch.bfloat16),
    (1, 16, 2, 128, [250], torch.float16),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,dtype", CASES)
def test_dense_equivalence(B, Hq, Hkv, D, lens, dtype):
    g = torch.Generator().manual_seed(11)
    nmax = max(lens)
    q = torch.randn(B, Hq, D, generator=g).to(dtype)
    K = torch.randn(B, Hkv, nmax, D, generator=g).to(dtype)
    V = torch.randn(B, Hkv, nmax, D, generator=g).to(dtype)
    kp, vp, tables = _paged_from_dense(K, V, lens, num_blocks=64, seed=3)
    scale = 1.0 / math.sqrt(D)
    got = oracle.attention_decode(q, kp, vp, tables, lens, scale)
    ref = _dense_reference(q, K, V, lens, scale).numpy()
    assert np.isfinite(got).all()  # NaN sentinels in unused slots never read
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_rows_subset_matches_full():
    g = torch.Generator().manual_seed(5)
    q = torch.randn(2, 4, 64, generator=g).half()
    K = torch.randn(2, 2, 40, 64, generator=g).half()
    V = torch.randn(2, 2, 40, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, [40, 23], 16, seed=1)
    full = oracle.attention_decode(q, kp, vp, tables, [40, 23], 0.125)
    rows = [(1, 3), (0, 0), (1, 1)]
    sub = oracle.attention_decode(q, kp, vp, tables, [40, 23], 0.125, rows=rows)
    for i, (b, h) in enumerate(rows):
        assert np.array_equal(sub[i], full[b, h])


def test_block_permutation_invariance():
    g = torch.Generator().manual_seed(21)
    lens = [50, 7, 128]
    q = torch.randn(3, 4, 64, generator=g).half()
    K = torch.randn(3, 2, 128, 64, generator=g).half()
    V = torch.randn(3, 2, 128, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, lens, 32, seed=2)
    a = oracle.attention_decode(q, kp, vp, tables, lens, 0.125)
    pi = torch.randperm(32, generator=g)
    kp2 = torch.empty_like(kp)
    vp2 = torch.empty_like(vp)
    kp2[pi] = kp
    vp2[pi] = vp
    t2 = torch.where(tables >= 0, pi[tables.clamp(min=0).long()].to(torch.int32), tables)
    b = oracle.attention_decode(q, kp2, vp2, t2, lens, 0.125)
    assert np.array_equal(a, b)


def test_single_token_returns_v0_exactly():
    g = torch.Generator().manual_seed(4)
    q = torch.randn(2, 4, 64, generator=g).half()
    K = torch.randn(2, 2, 1, 64, generator=g).half()
    V = torch.randn(2, 2, 1, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, [1, 1], 8, seed=9)
    got = oracle.attention_decode(q, kp, vp, tables, [1, 1], 0.125)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(got[b, h], V[b, h // 2, 0].double().numpy())


def test_identical_keys_give_mean_of_v():
    g = torch.Generator().manual_seed(8)
    n = 45
    q = torch.randn(1, 2, 64, generator=g).half()
    k_one = torch.randn(64, generator=g).half()
    K = k_one.expand(1, 1, n, 64).clone()
    V = torch.randn(1, 1, n, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, [n], 8, seed=1)
    got = oracle.attention_decode(q, kp, vp, tables, [n], 0.3)
    mean = V[0, 0].double().mean(dim=0).numpy()
    np.testing.assert_allclose(got[0, 0], mean, rtol=0, atol=1e-14)
    np.testing.assert_allclose(got[0, 1], mean, rtol=0, atol=1e-14)


def test_scale_zero_gives_mean_of_v():
    g = torch.Generator().manual_seed(9)
    n = 70
    q = torch.randn(1, 1, 64, generator=g).half()
    K = torch.randn(1, 1, n, 64, generator=g).half()
    V = torch.randn(1, 1, n, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, [n], 8, seed=1)
    got = oracle.attention_decode(q, kp, vp, tables, [n], 0.0)
    np.testing.assert_allclose(got[0, 0], V[0, 0].double().mean(0).numpy(), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    g = torch.Generator().manual_seed(10)
    n = 40
    q = torch.randn(1, 1, 64, generator=g).half()
    K = torch.randn(1, 1, n, 64, generator=g).half()
    V = torch.randn(1, 1, n, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, [n], 8, seed=1)
    s = (K[0, 0].double() @ q[0, 0].double()).numpy()
    j = int(np.argmax(s))
    gap = np.sort(s)[-1] - np.sort(s)[-2]
    scale = 800.0 / max(gap, 1e-3)  # next-best weight <= e^-800: underflows
    got = oracle.attention_decode(q, kp, vp, tables, [n], scale)
    assert np.array_equal(got[0, 0], V[0, 0, j].double().numpy())


def test_two_tokens_closed_form():
    g = torch.Generator().manual_seed(12)
    q = torch.randn(1, 1, 64, generator=g).half()
    K = torch.randn(1, 1, 2, 64, generator=g).half()
    V = torch.randn(1, 1, 2, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, [2], 8, seed=1)
    sc = 0.2
    got = oracle.attention_decode(q, kp, vp, tables, [2], sc)[0, 0]
    qd = q[0, 0].double().numpy()
    s1 = sc * float(np.dot(qd, K[0, 0, 0].double().numpy()))
    s2 = sc * float(np.dot(qd, K[0, 0, 1].double().numpy()))
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))  # logistic form of the 2-way softmax
    ref = w1 * V[0, 0, 0].double().numpy() + (1.0 - w1) * V[0, 0, 1].double().numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_query_group_maps_to_kv_head_by_division():
    # Hq = 6, Hkv = 3: heads 0,1 -> kv 0; 2,3 -> kv 1; 4,5 -> kv 2.
    g = torch.Generator().manual_seed(13)
    n = 20
    q = torch.randn(1, 6, 64, generator=g).half()
    K = torch.randn(1, 3, n, 64, generator=g).half()
    V = torch.empty(1, 3, n, 64, dtype=torch.float16)
    for kv in range(3):
        V[0, kv] = float(kv + 1)  # constant value per kv head
    kp, vp, tables = _paged_from_dense(K, V, [n], 8, seed=1)
    got = oracle.attention_decode(q, kp, vp, tables, [n], 0.1)
    for h in range(6):
        np.testing.assert_allclose(got[0, h], float(h // 2 + 1), rtol=1e-14)


def test_zero_length_gives_zero_row_and_bad_block_raises():
    q = torch.ones(2, 1, 64, dtype=torch.float16)
    kp = torch.ones(4, 1, BS, 64, dtype=torch.float16)
    tables = torch.tensor([[0], [5]], dtype=torch.int32)
    got = oracle.attention_decode(q[:1], kp, kp, tables[:1], [0], 1.0)
    assert np.array_equal(got, np.zeros((1, 1, 64)))
    with pytest.raises(ValueError):
        oracle.attention_decode(q, kp, kp, tables, [0, 3], 1.0)   # block 5 >= 4
    with pytest.raises(ValueError):
        oracle.attention_decode(q[:1], kp, kp, tables[:1], [17], 1.0)  # 17 > 1 block


def test_int8_decode_equals_dense_on_dequantised_values():
    g = torch.Generator().manual_seed(14)
    lens = [33, 90]
    q = torch.randn(2, 8, 64, generator=g).half()
    Kc = torch.randint(-127, 128, (2, 2, 90, 64), generator=g, dtype=torch.int8)
    Vc = torch.randint(-127, 128, (2, 2, 90, 64), generator=g, dtype=torch.int8)
    Ks = torch.rand(2, 2, 90, generator=g) * 0.05 + 0.001
    Vs = torch.rand(2, 2, 90, generator=g) * 0.05 + 0.001
    kp, vp, tables = _paged_from_dense(Kc, Vc, lens, 16, seed=4, fill=0)
    ksp, vsp, _ = _paged_from_dense(Ks[..., None], Vs[..., None], lens, 16, seed=4, fill=0)
    got = oracle.attention_decode(q, kp, vp, tables, lens, 0.125,
                                  k_scale=ksp[..., 0], v_scale=vsp[..., 0])
    Kd = Kc.double() * Ks.double()[..., None]
    Vd = Vc.double() * Vs.double()[..., None]
    ref = _dense_reference(q, Kd, Vd, lens, 0.125).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ INT8 quantiser
def _f32(v: float) -> float:
    """The float32 nearest to the double v (ties to even)."""
    return struct.unpack("f", struct.pack("f", v))[0]


def _quantise_rows_by_definition(x, qmax=127, fixed_scale=None):
    """The INT8 rule written out from its definition ("KV Cache 优化与显存管理",
    三: scale = abs-max / 127 per token and head, zero scale -> 1, codes =
    x / scale rounded half to even, clipped to [-128, 127]) with exact
    rational arithmetic instead of float32 arrays: every float32 quotient is
    the exact quotient rounded once to double and once to float32, which
    equals rounding it directly to float32 because a double carries more than
    2 * 24 + 2 bits (Figueroa, "When is double rounding innocuous?", 1995).
    Python's round() is half-to-even.  Returns (codes [rows, D] int8, scales
    [rows] float32)."""
    rows = [[float(v) for v in r] for r in np.asarray(x, dtype=np.float64)]
    codes = np.zeros((len(rows), len(rows[0]) if rows else 0), dtype=np.int8)
    scales = np.zeros(len(rows), dtype=np.float32)
    for i, r in enumerate(rows):
        if fixed_scale is None:
            amax = max(abs(v) for v in r)
            s = _f32(float(Fraction(amax) / qmax))
            s = s if s > 0 else 1.0
        else:
            s = _f32(fixed_scale)
        for j, v in enumerate(r):
            q = round(_f32(float(Fraction(v) / Fraction(s))))
            codes[i, j] = min(127, max(-128, q))
        scales[i] = s
    return codes, scales


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_quantiser_matches_its_definition(dtype):
    g = torch.Generator().manual_seed(15)
    x = (torch.randn(160, 128, generator=g) * torch.rand(160, 1, generator=g) * 3).to(dtype)
    x[3] = 0
    x[4, :7] = 0
    x[5] = 1e-3
    codes, scales = oracle.quantize_int8(x)
    ref_codes, ref_scales = _quantise_rows_by_definition(x.float().numpy())
    assert np.array_equal(codes, ref_codes)
    assert np.array_equal(scales.view(np.uint32), ref_scales.view(np.uint32))


def test_quantiser_properties():
    """Properties any correct per-row abs-max quantiser has, independent of
    how it is written: each code times its scale is within half a scale of the
    source value, the abs-max element maps to +-127, the scale is the float32
    nearest to abs-max / 127 (its neighbours are farther), and codes stay in
    [-127, 127]."""
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(300, 64, generator=g) * torch.rand(300, 1, generator=g) * 10).half()
    codes, scales = oracle.quantize_int8(x)
    xf = x.double().numpy()
    sc = scales.astype(np.float64)[:, None]
    assert np.all(np.abs(codes * sc - xf) <= sc * (0.5 + 2.0 ** -20))
    amax_at = np.argmax(np.abs(xf), axis=1)
    assert np.all(np.abs(codes[np.arange(len(xf)), amax_at]) == 127)
    for i in range(len(xf)):
        exact = Fraction(float(np.abs(xf[i]).max())) / 127
        s = np.float32(scales[i])
        d = abs(Fraction(float(s)) - exact)
        for nb in (np.nextafter(s, np.float32(0)), np.nextafter(s, np.float32(np.inf))):
            assert d <= abs(Fraction(float(nb)) - exact)
    assert codes.min() >= -127 and codes.max() <= 127


def test_quantiser_special_rows():
    x = torch.zeros(4, 8, dtype=torch.float16)
    # row 1: amax 127 -> scale exactly 1.0; x.5 values are ties -> even
    x[1] = torch.tensor([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5])
    # row 2: the abs-max element maps to +-127
    x[2] = torch.tensor([0.1, -3.0, 2.0, 0.0, 1.0, -1.0, 0.25, 2.9])
    x[3] = torch.tensor([4.0, 1.0, -1.0, 0.0, 0.5, 2.0, -4.0, 3.0])
    codes, scales = oracle.quantize_int8(x)
    assert codes[0].tolist() == [0] * 8 and scales[0] == 1.0
    assert scales[1] == 1.0
    assert codes[1].tolist() == [127, 2, 4, -2, -4, 0, 0, 2]
    assert codes[2, 1] == -127 and np.abs(codes[2]).max() == 127
    assert codes[3, 0] == 127 and codes[3, 6] == -127


def test_quantiser_never_reaches_minus_128():
    g = torch.Generator().manual_seed(16)
    x = torch.randn(20000, 64, generator=g).half()
    codes, _ = oracle.quantize_int8(x)
    assert codes.min() >= -127 and codes.max() <= 127
    assert (np.abs(codes).max(axis=1) == 127).all()


# ------------------------------------------------------------ append / copy
def test_append_matches_numpy_indexing():
    g = torch.Generator().manual_seed(17)
    NB, Hkv, D = 6, 3, 64
    pool = torch.randn(NB, Hkv, BS, D, generator=g).half()
    src = torch.randn(5, Hkv, D, generator=g).half()
    slots = torch.tensor([0, 17, -1, 95, 40], dtype=torch.int32)
    got = oracle.append(pool, src, slots)
    ref = pool.clone().numpy()
    for t, s in enumerate(slots.tolist()):
        if s >= 0:
            ref[s // BS, :, s % BS, :] = src[t].numpy()
    assert np.array_equal(got.numpy(), ref)
    with pytest.raises(ValueError):
        oracle.append(pool, src[:1], torch.tensor([NB * BS], dtype=torch.int32))


def test_copy_blocks_matches_numpy_and_self_copy_is_identity():
    g = torch.Generator().manual_seed(18)
    pool = torch.randn(8, 2, BS, 64, generator=g).half()
    pairs = torch.tensor([[1, 5], [2, 2], [7, 0]], dtype=torch.int32)
    got = oracle.copy_blocks(pool, pairs).numpy()
    ref = pool.clone().numpy()
    ref[5] = ref[1]
    ref[0] = pool.numpy()[7]
    assert np.array_equal(got, ref)
    with pytest.raises(ValueError):
        oracle.copy_blocks(pool, torch.tensor([[0, 8]], dtype=torch.int32))


def test_append_int8_matches_quantise_then_scatter():
    g = torch.Generator().manual_seed(19)
    NB, Hkv, D = 4, 2, 64
    codes = torch.zeros(NB, Hkv, BS, D, dtype=torch.int8)
    scales = torch.zeros(NB, Hkv, BS)
    src = torch.randn(3, Hkv, D, generator=g).half()
    slots = torch.tensor([5, -1, 63], dtype=torch.int32)
    c, s = oracle.append_int8(codes, scales, src, slots)
    c, s = c.numpy(), s.numpy()
    qc, qs = _quantise_rows_by_definition(src.float().numpy().reshape(-1, D))
    qc, qs = qc.reshape(3, Hkv, D), qs.reshape(3, Hkv)
    assert np.array_equal(c[0, :, 5], qc[0]) and np.array_equal(c[3, :, 15], qc[2])
    assert np.array_equal(s[0, :, 5], qs[0]) and np.array_equal(s[3, :, 15], qs[2])
    assert int(np.count_nonzero(s)) == 2 * Hkv


# ------------------------------------------------------------ FP8 (E4M3) and per-tensor INT8
def test_e4m3_widening_exhaustive():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes.tolist()])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


def test_e4m3_rounding_matches_library_and_ties_go_even():
    g = torch.Generator().manual_seed(40)
    x = torch.cat([torch.randn(20000, generator=g) * 30,
                   torch.rand(5000, generator=g) * 896 - 448,
                   torch.randn(5000, generator=g) * 0.01])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(float(v)) for v in x.tolist()], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # exact midpoints between neighbouring codes round to the even code
    vals = [oracle.e4m3_to_f64(c) for c in range(0x7f)]
    for c in range(0x7e):
        mid = (vals[c] + vals[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle.f32_to_e4m3(mid) == want
        assert oracle.f32_to_e4m3(-mid) == 0x80 | want
    assert oracle.f32_to_e4m3(1e6) == 0x7e and oracle.f32_to_e4m3(-500.0) == 0xfe  # saturate


def test_fp8_quantiser_matches_library_restatement():
    g = torch.Generator().manual_seed(41)
    x = (torch.randn(300, 128, generator=g) * torch.rand(300, 1, generator=g) * 5).half()
    x[3] = 0
    codes, scales = oracle.quantize_fp8(x)
    xf = x.float()
    amax = xf.abs().amax(dim=-1, keepdim=True)
    sc = amax / 448.0
    sc = torch.where(sc > 0, sc, torch.ones_like(sc))
    ref = (xf / sc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    assert np.array_equal(scales.view(np.uint32), sc[:, 0].numpy().view(np.uint32))
    assert codes[3].tolist() == [0] * 128 and scales[3] == 1.0


def test_fixed_scale_int8_matches_its_definition():
    g = torch.Generator().manual_seed(42)
    x = (torch.randn(64, 128, generator=g) * 3).half()
    s = 0.0375
    got = oracle.quantize_int8_fixed(x, s)
    ref, _ = _quantise_rows_by_definition(x.float().numpy(), fixed_scale=s)
    assert np.array_equal(got, ref)
    big = torch.full((1, 8), 60000.0, dtype=torch.float16)
    assert oracle.quantize_int8_fixed(big, 1.0).tolist() == [[127] * 8]   # clip


def test_fp8_decode_equals_dense_on_dequantised_values():
    g = torch.Generator().manual_seed(43)
    lens = [21, 77]
    q = torch.randn(2, 8, 64, generator=g).half()
    src_k = torch.randn(2, 2, 77, 64, generator=g).half()
    src_v = torch.randn(2, 2, 77, 64, generator=g).half()
    ck, sk = oracle.quantize_fp8(src_k)
    cv, sv = oracle.quantize_fp8(src_v)
    Kc = torch.from_numpy(ck).view(torch.float8_e4m3fn)
    Vc = torch.from_numpy(cv).view(torch.float8_e4m3fn)
    kp, vp, tables = _paged_from_dense(Kc.view(torch.uint8), Vc.view(torch.uint8), lens, 16,
                                       seed=4, fill=0)
    ksp, vsp, _ = _paged_from_dense(torch.from_numpy(sk)[..., None],
                                    torch.from_numpy(sv)[..., None], lens, 16, seed=4, fill=0)
    got = oracle.attention_decode(q, kp.view(torch.float8_e4m3fn), vp.view(torch.float8_e4m3fn),
                                  tables, lens, 0.125, k_scale=ksp[..., 0], v_scale=vsp[..., 0])
    Kd = Kc.to(torch.float64) * torch.from_numpy(sk).double()[..., None]
    Vd = Vc.to(torch.float64) * torch.from_numpy(sv).double()[..., None]
    ref = _dense_reference(q, Kd, Vd, lens, 0.125).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_append_fp8_matches_quantise_then_scatter():
    g = torch.Generator().manual_seed(44)
    NB, Hkv, D = 4, 2, 64
    codes = torch.zeros(NB, Hkv, BS, D, dtype=torch.uint8).view(torch.float8_e4m3fn)
    scales = torch.zeros(NB, Hkv, BS)
    src = torch.randn(3, Hkv, D, generator=g).half()
    slots = torch.tensor([5, -1, 63], dtype=torch.int32)
    c, s = oracle.append_fp8(codes, scales, src, slots)
    assert c.dtype == torch.float8_e4m3fn
    qc, qs = oracle.quantize_fp8(src)
    assert np.array_equal(c.view(torch.uint8)[0, :, 5].numpy(), qc[0])
    assert np.array_equal(c.view(torch.uint8)[3, :, 15].numpy(), qc[2])
    assert np.array_equal(s[0, :, 5].numpy(), qs[0]) and np.array_equal(s[3, :, 15].numpy(), qs[2])


# ------------------------------------------------------------ multi-query (prefill) attention
def _causal_reference(q, K, V, starts, lens, scale):
    """torch float64 scaled_dot_product_attention with an explicit causal mask
    for queries that are the last L of n cached tokens."""
    import torch.nn.functional as F
    T, Hq, D = q.shape
    Hkv = K.shape[1]
    out = torch.zeros(T, Hq, D, dtype=torch.float64)
    for b in range(len(lens)):
        n, L = lens[b], starts[b + 1] - starts[b]
        k = K[b, :, :n].double().repeat_interleave(Hq // Hkv, dim=0)   # [Hq, n, D]
        v = V[b, :, :n].double().repeat_interleave(Hq // Hkv, dim=0)
        qq = q[starts[b]:starts[b + 1]].double().transpose(0, 1)        # [Hq, L, D]
        pos = torch.arange(n - L, n)
        mask = torch.arange(n)[None, :] <= pos[:, None]                 # [L, n]
        o = F.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=scale)
        out[starts[b]:starts[b + 1]] = o.transpose(0, 1)
    return out


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 4, 64), (8, 2, 64), (8, 1, 128)])
def test_prefill_equals_causal_sdpa(Hq, Hkv, D):
    g = torch.Generator().manual_seed(60)
    lens = [40, 100, 17]
    qlens = [40, 7, 1]          # full prefill, a chunk, a single token
    starts = [0]
    for L in qlens:
        starts.append(starts[-1] + L)
    q = torch.randn(starts[-1], Hq, D, generator=g).half()
    K = torch.randn(3, Hkv, 100, D, generator=g).half()
    V = torch.randn(3, Hkv, 100, D, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, lens, 32, seed=5)
    got = oracle.attention_prefill(q, kp, vp, tables, lens, starts, 1 / math.sqrt(D))
    ref = _causal_reference(q, K, V, starts, lens, 1 / math.sqrt(D)).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_prefill_single_token_chunks_equal_decode():
    g = torch.Generator().manual_seed(61)
    lens = [33, 80]
    q = torch.randn(2, 8, 64, generator=g).half()
    K = torch.randn(2, 2, 80, 64, generator=g).half()
    V = torch.randn(2, 2, 80, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, lens, 16, seed=6)
    pre = oracle.attention_prefill(q, kp, vp, tables, lens, [0, 1, 2], 0.2)
    dec = oracle.attention_decode(q, kp, vp, tables, lens, 0.2)
    np.testing.assert_allclose(pre, dec, rtol=1e-13, atol=1e-14)


def test_prefill_first_query_of_a_prompt_returns_v0():
    """A whole-prompt prefill's first query sits at position 0 and attends to
    key 0 alone: its output is V[0] exactly (widened), whatever q and K hold."""
    g = torch.Generator().manual_seed(62)
    lens = [37]
    q = torch.randn(37, 4, 64, generator=g).half()
    K = torch.randn(1, 2, 37, 64, generator=g).half()
    V = torch.randn(1, 2, 37, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, lens, 8, seed=7)
    out = oracle.attention_prefill(q, kp, vp, tables, lens, [0, 37], 0.125)
    for h in range(4):  # query heads 0, 1 read kv head 0; 2, 3 read kv head 1
        assert np.array_equal(out[0, h], V[0, h // 2, 0].double().numpy())


def test_prefill_never_reads_keys_after_the_query():
    """Causality: changing K/V at positions past a query's own leaves its row
    bit-identical, and changes the rows that can see them."""
    g = torch.Generator().manual_seed(63)
    lens, L = [50], 20              # queries at positions 30 .. 49
    q = torch.randn(L, 4, 64, generator=g).half()
    K = torch.randn(1, 2, 50, 64, generator=g).half()
    V = torch.randn(1, 2, 50, 64, generator=g).half()
    kp, vp, tables = _paged_from_dense(K, V, lens, 8, seed=8)
    base = oracle.attention_prefill(q, kp, vp, tables, lens, [0, L], 0.125)
    K2, V2 = K.clone(), V.clone()
    K2[:, :, 40:] = torch.randn(1, 2, 10, 64, generator=g).half()
    V2[:, :, 40:] = torch.randn(1, 2, 10, 64, generator=g).half()
    kp2, vp2, _ = _paged_from_dense(K2, V2, lens, 8, seed=8)
    moved = oracle.attention_prefill(q, kp2, vp2, tables, lens, [0, L], 0.125)
    assert np.array_equal(base[:10], moved[:10])       # positions 30 .. 39
    assert not np.allclose(base[10:], moved[10:])      # positions 40 .. 49 see the change
