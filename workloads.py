"""Seeded synthetic inputs for the paged-KV-cache decode path.

This module only *draws* inputs: random query / key / value values, block
tables, context lengths, slot mappings and copy-on-write pairs.  It holds none
of the method's arithmetic (no attention, no quantisation, no copying of cache
blocks) and imports neither the CUDA library nor the oracle; both of those are
fed the tensors made here.

Workloads (shapes follow the pages' examples; values are N(0, 1)):
  tiny      B=4, Hq=8, Hkv=2, D=64, fp16, 64-block pool, lens {1,17,100,255},
            tables from a seeded permutation, scale 1/8, 1 appended token/request.
  llama7b   Llama2-7B-shaped layer ("ATB KV Cache management", "KV Cache 的显存需求":
            32 kv heads x 128, fp16, 4096 tokens): B=32, Hq=Hkv=32, D=128,
            10000-block pool, every context 4096, tables shuffled through the pool,
            32 appended tokens (one per request, at position 4095).
  gqa70b    GQA 70B-shaped layer: B=64, Hq=64, Hkv=8, D=128, bf16, lens uniform
            in [512, 8192], 40000-block pool; tables are contiguous runs with
            probability 0.85 per block and a random free block otherwise
            ("ATB KV Cache management", "显存碎片问题": 80-90% contiguous).
  prefix    prefix sharing: B=128, 32/32 heads, D=128, fp16, 8192-block pool;
            a 1030-token prefix (64 full blocks + 6 tokens) in shared physical
            blocks, private suffixes uniform in [16, 512]; the step first copies
            the shared partial block for every request but the last (copy-on-write,
            "ATB PagedAttention", "踩坑三"), then appends every suffix token.
  int8long  long-context INT8: B=4, context 131072, Hq=64, Hkv=8, D=128, fp16
            source pools to be quantised per token and head, 40000-block pool,
            fully scattered tables, 1 appended token/request.
  fp8long   the same shapes with FP8 (E4M3) codes ("KV Cache 优化与显存管理", 二:
            INT8 or FP8).

Seeds: workload i (in the order above) uses base seed 1000 + i; each draw has
its own generator seeded base * 100 + k with k = 0 q, 1 K pool, 2 V pool,
3 new K, 4 new V, 5 tables, 6 lengths.  Pool slots that no table covers before
the append, and the tail slots of each partial last block, hold NaN in 16-bit
pools (a sentinel that any over-read turns into a NaN output).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BLOCK_SIZE = 16
WORKLOAD_NAMES = ("tiny", "llama7b", "gqa70b", "prefix", "int8long", "fp8long")


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    num_blocks: int
    dtype: torch.dtype          # q, new K/V and 16-bit pools
    kv_int8: bool               # pools hold 8-bit codes + float32 scales
    scale: float
    q: torch.Tensor             # [B, Hq, D]
    k_pool: torch.Tensor        # [NB, Hkv, bs, D] (int8 workloads: fp16 source values)
    v_pool: torch.Tensor
    block_tables: torch.Tensor  # [B, MB] int32, -1 past each request's blocks
    context_lens: torch.Tensor  # [B] int32, after the step's append
    new_k: torch.Tensor         # [T, Hkv, D]
    new_v: torch.Tensor
    slot_mapping: torch.Tensor  # [T] int32
    cow_pairs: Optional[torch.Tensor] = None  # [P, 2] int32 (src, dst)
    info: dict = field(default_factory=dict)
    kv_fp8: bool = False        # the 8-bit codes are FP8 E4M3 (else INT8)

    @property
    def block_size(self) -> int:
        return BLOCK_SIZE

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    def to(self, device) -> "Workload":
        moved = {}
        for k, v in self.__dict__.items():
            moved[k] = v.to(device) if isinstance(v, torch.Tensor) else v
        return Workload(**moved)


# ------------------------------------------------------------------ helpers
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, dtype, seed, device, chunk_rows: int = 1 << 14) -> torch.Tensor:
    """N(0,1) float32 draws rounded to ``dtype``; drawn in chunks along dim 0 so
    host memory stays bounded for multi-GB pools (same values for any chunking
    on one device type because each chunk has its own derived generator)."""
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    for i, s in enumerate(range(0, n0, chunk_rows)):
        e = min(n0, s + chunk_rows)
        g = _gen(seed * 1000003 + i, device)
        out[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=g,
                               dtype=torch.float32, device=device).to(dtype)
    return out


def _tables_from_lists(lists, mb) -> torch.Tensor:
    t = torch.full((len(lists), mb), -1, dtype=torch.int32)
    for b, blocks in enumerate(lists):
        if blocks:
            t[b, :len(blocks)] = torch.tensor(blocks, dtype=torch.int32)
    return t


def _slot_of(tables: torch.Tensor, b: int, pos: int) -> int:
    return int(tables[b, pos // BLOCK_SIZE]) * BLOCK_SIZE + pos % BLOCK_SIZE


def _nan_unfilled(pool: torch.Tensor, tables: torch.Tensor, filled_lens) -> None:
    """Set every pool slot not covered by positions [0, filled_lens[b]) of some
    request to NaN (16-bit pools only)."""
    NB = pool.shape[0]
    valid = torch.zeros(NB, BLOCK_SIZE, dtype=torch.bool)
    for b in range(tables.shape[0]):
        n = int(filled_lens[b])
        if n <= 0:
            continue
        nfull, rem = divmod(n, BLOCK_SIZE)
        full = tables[b, :nfull].long()
        valid[full] = True
        if rem:
            valid[int(tables[b, nfull]), :rem] = True
    mask = (~valid).to(pool.device)[:, None, :, None].expand_as(pool)
    pool.masked_fill_(mask, float("nan"))


def contiguous_share(tables: torch.Tensor, lens) -> float:
    """Share of logical blocks i > 0 stored right after block i - 1."""
    hit = tot = 0
    for b in range(tables.shape[0]):
        nb = -(-int(lens[b]) // BLOCK_SIZE)
        row = tables[b, :nb].tolist()
        for i in range(1, nb):
            tot += 1
            hit += row[i] == row[i - 1] + 1
    return hit / tot if tot else 1.0


# ------------------------------------------------------------------ builders
def make_custom(*, B, Hq, Hkv, D, lens, num_blocks, dtype=torch.float16, kv_int8=False,
                scale=None, seed=7, contiguous_p=0.0, max_blocks=None, device="cpu",
                name="custom", nan_sentinel=True) -> Workload:
    """A general workload: 1 appended token per request with lens[b] > 0 (the
    token at position lens[b]-1), tables drawn from the pool either scattered
    (contiguous_p = 0) or as runs (block i follows block i-1 with prob. p)."""
    lens = [int(x) for x in lens]
    nblk = [-(-n // BLOCK_SIZE) for n in lens]
    mb = max_blocks if max_blocks is not None else max(1, max(nblk) if nblk else 1)
    if sum(nblk) > num_blocks:
        raise ValueError("pool too small for the requested lengths")
    rng = np.random.default_rng(seed * 100 + 5)
    lists = _draw_tables(rng, nblk, num_blocks, contiguous_p)
    tables = _tables_from_lists(lists, mb)
    return _assemble(name, B, Hq, Hkv, D, num_blocks, dtype, kv_int8,
                     scale if scale is not None else 1.0 / math.sqrt(D),
                     lens, tables, seed, device, nan_sentinel)


def _draw_tables(rng, nblk, num_blocks, p, taken=()):
    free = np.ones(num_blocks, dtype=bool)
    free_list = list(range(num_blocks))
    pos = {b: i for i, b in enumerate(free_list)}

    def take(blk):
        free[blk] = False
        i = pos.pop(blk)
        last = free_list.pop()
        if last != blk:
            free_list[i] = last
            pos[last] = i

    for blk in taken:  # blocks already handed out elsewhere
        take(int(blk))
    lists = []
    for n in nblk:
        row = []
        for i in range(n):
            if i > 0 and p > 0 and rng.random() < p and row[-1] + 1 < num_blocks and free[row[-1] + 1]:
                blk = row[-1] + 1
            else:
                blk = free_list[int(rng.integers(len(free_list)))]
            take(blk)
            row.append(blk)
        lists.append(row)
    return lists


def _assemble(name, B, Hq, Hkv, D, NB, dtype, kv_int8, scale, lens, tables, seed, device,
              nan_sentinel=True, info=None) -> Workload:
    base = seed * 100
    pool_dtype = torch.float16 if kv_int8 else dtype
    q = _randn((B, Hq, D), dtype, base + 0, device)
    k_pool = _randn((NB, Hkv, BLOCK_SIZE, D), pool_dtype, base + 1, device)
    v_pool = _randn((NB, Hkv, BLOCK_SIZE, D), pool_dtype, base + 2, device)
    active = [b for b in range(B) if lens[b] > 0]
    T = len(active)
    new_k = _randn((max(T, 1), Hkv, D), pool_dtype, base + 3, device)[:T]
    new_v = _randn((max(T, 1), Hkv, D), pool_dtype, base + 4, device)[:T]
    slots = torch.tensor([_slot_of(tables, b, lens[b] - 1) for b in active], dtype=torch.int32)
    if nan_sentinel and not kv_int8:
        pre = [max(0, n - 1) for n in lens]
        _nan_unfilled(k_pool, tables, pre)
        _nan_unfilled(v_pool, tables, pre)
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, num_blocks=NB, dtype=dtype,
                    kv_int8=kv_int8, scale=scale, q=q, k_pool=k_pool, v_pool=v_pool,
                    block_tables=tables, context_lens=torch.tensor(lens, dtype=torch.int32),
                    new_k=new_k, new_v=new_v, slot_mapping=slots.to(device),
                    info=dict(info or {}))


def make(name: str, device="cpu", nan_sentinel=True, batch=None, contiguity=None) -> Workload:
    """Build one of the named workloads (see module docstring).  ``batch``
    shrinks llama7b / gqa70b / int8long to fewer requests with the pool scaled
    in proportion (same per-request shapes), e.g. for profiler captures.
    ``contiguity`` (llama7b, gqa70b) redraws the block tables so each block
    follows its predecessor with that probability (0 = fully scattered, 1 = one
    contiguous run per request)."""
    if contiguity is not None and name in ("llama7b", "gqa70b"):
        return _make_with_contiguity(name, float(contiguity), device, nan_sentinel, batch)
    idx = WORKLOAD_NAMES.index(name)
    seed = 1000 + idx
    base = seed * 100
    if name == "fp8long":
        w = make("int8long", device=device, nan_sentinel=nan_sentinel, batch=batch)
        w.name, w.kv_fp8 = "fp8long", True
        return w
    if batch is not None and name in ("llama7b", "gqa70b", "int8long"):
        return _make_scaled(name, int(batch), device, nan_sentinel, seed)
    if name == "tiny":
        lens = [1, 17, 100, 255]
        g = _gen(base + 5, "cpu")
        perm = torch.randperm(64, generator=g)[:26].tolist()
        lists, at = [], 0
        for n in lens:
            k = -(-n // BLOCK_SIZE)
            lists.append(perm[at:at + k])
            at += k
        tables = _tables_from_lists(lists, 16)
        return _assemble(name, 4, 8, 2, 64, 64, torch.float16, False, 1.0 / 8.0, lens,
                         tables, seed, device, nan_sentinel)
    if name == "llama7b":
        B, n, NB = 32, 4096, 10000
        g = _gen(base + 5, "cpu")
        perm = torch.randperm(NB, generator=g)[:B * 256].view(B, 256).to(torch.int32)
        return _assemble(name, B, 32, 32, 128, NB, torch.float16, False,
                         1.0 / math.sqrt(128), [n] * B, perm.contiguous(), seed, device,
                         nan_sentinel)
    if name == "gqa70b":
        B, NB = 64, 40000
        rng_len = np.random.default_rng(base + 6)
        lens = rng_len.integers(512, 8192, size=B, endpoint=True).tolist()
        rng_tab = np.random.default_rng(base + 5)
        lists = _draw_tables(rng_tab, [-(-n // BLOCK_SIZE) for n in lens], NB, 0.85)
        tables = _tables_from_lists(lists, 512)
        info = {"contiguous_share": contiguous_share(tables, lens)}
        return _assemble(name, B, 64, 8, 128, NB, torch.bfloat16, False,
                         1.0 / math.sqrt(128), lens, tables, seed, device, nan_sentinel, info)
    if name == "prefix":
        return _make_prefix(seed, device, nan_sentinel)
    if name == "int8long":
        B, n, NB = 4, 131072, 40000
        g = _gen(base + 5, "cpu")
        perm = torch.randperm(NB, generator=g)[:B * 8192].view(B, 8192).to(torch.int32)
        return _assemble(name, B, 64, 8, 128, NB, torch.float16, True,
                         1.0 / math.sqrt(128), [n] * B, perm.contiguous(), seed, device,
                         nan_sentinel)
    raise KeyError(name)


def _make_with_contiguity(name, p, device, nan_sentinel, batch) -> Workload:
    w = make(name, device="cpu", nan_sentinel=False, batch=batch)
    lens = [int(x) for x in w.context_lens]
    seed = 1000 + WORKLOAD_NAMES.index(name)
    lists = _draw_tables(np.random.default_rng(seed * 100 + 5), [-(-n // BLOCK_SIZE) for n in lens],
                         w.num_blocks, p)
    tables = _tables_from_lists(lists, w.max_blocks)
    info = {"contiguous_share": contiguous_share(tables, lens), "contiguity_p": p}
    return _assemble(name, w.B, w.Hq, w.Hkv, w.D, w.num_blocks, w.dtype, False, w.scale, lens,
                     tables, seed, device, nan_sentinel, info)


def _make_scaled(name, B, device, nan_sentinel, seed) -> Workload:
    base = seed * 100
    if name == "llama7b":
        NB = -(-10000 * B // 32)
        g = _gen(base + 5, "cpu")
        perm = torch.randperm(NB, generator=g)[:B * 256].view(B, 256).to(torch.int32)
        return _assemble(name, B, 32, 32, 128, NB, torch.float16, False, 1.0 / math.sqrt(128),
                         [4096] * B, perm.contiguous(), seed, device, nan_sentinel)
    if name == "gqa70b":
        NB = -(-40000 * B // 64)
        lens = np.random.default_rng(base + 6).integers(512, 8192, size=B, endpoint=True).tolist()
        lists = _draw_tables(np.random.default_rng(base + 5), [-(-n // BLOCK_SIZE) for n in lens],
                             NB, 0.85)
        tables = _tables_from_lists(lists, 512)
        info = {"contiguous_share": contiguous_share(tables, lens)}
        return _assemble(name, B, 64, 8, 128, NB, torch.bfloat16, False, 1.0 / math.sqrt(128),
                         lens, tables, seed, device, nan_sentinel, info)
    NB = -(-40000 * B // 4)
    g = _gen(base + 5, "cpu")
    perm = torch.randperm(NB, generator=g)[:B * 8192].view(B, 8192).to(torch.int32)
    return _assemble(name, B, 64, 8, 128, NB, torch.float16, True, 1.0 / math.sqrt(128),
                     [131072] * B, perm.contiguous(), seed, device, nan_sentinel)


def _make_prefix(seed, device, nan_sentinel) -> Workload:
    B, Hq, Hkv, D, NB = 128, 32, 32, 128, 8192
    prefix = 1030
    base = seed * 100
    rng_len = np.random.default_rng(base + 6)
    suffix = rng_len.integers(16, 512, size=B, endpoint=True).tolist()
    lens = [prefix + s for s in suffix]
    g = _gen(base + 5, "cpu")
    perm = torch.randperm(NB, generator=g).tolist()
    shared = perm[:65]               # 64 full prefix blocks + the partial one
    nxt = 65
    lists, cow = [], []
    for b in range(B):
        nb = -(-lens[b] // BLOCK_SIZE)
        row = shared[:64]
        if b < B - 1:                # every request but the last copies the
            dst = perm[nxt]          # shared partial block before writing to it
            nxt += 1
            cow.append((shared[64], dst))
            row = row + [dst]
        else:
            row = row + [shared[64]]
        extra = nb - 65
        row = row + perm[nxt:nxt + extra]
        nxt += extra
        lists.append(row)
    mb = -(-(prefix + 512) // BLOCK_SIZE)
    tables = _tables_from_lists(lists, mb)
    q = _randn((B, Hq, D), torch.float16, base + 0, device)
    k_pool = _randn((NB, Hkv, BLOCK_SIZE, D), torch.float16, base + 1, device)
    v_pool = _randn((NB, Hkv, BLOCK_SIZE, D), torch.float16, base + 2, device)
    T = sum(suffix)
    new_k = _randn((T, Hkv, D), torch.float16, base + 3, device)
    new_v = _randn((T, Hkv, D), torch.float16, base + 4, device)
    slots = [_slot_of(tables, b, pos) for b in range(B) for pos in range(prefix, lens[b])]
    if nan_sentinel:
        # before the step only the prefix is in the pool: its 65 shared blocks
        pre_tables = _tables_from_lists([shared], 65)
        _nan_unfilled(k_pool, pre_tables, [prefix])
        _nan_unfilled(v_pool, pre_tables, [prefix])
    return Workload(name="prefix", B=B, Hq=Hq, Hkv=Hkv, D=D, num_blocks=NB,
                    dtype=torch.float16, kv_int8=False, scale=1.0 / math.sqrt(D), q=q,
                    k_pool=k_pool, v_pool=v_pool, block_tables=tables,
                    context_lens=torch.tensor(lens, dtype=torch.int32), new_k=new_k,
                    new_v=new_v, slot_mapping=torch.tensor(slots, dtype=torch.int32).to(device),
                    cow_pairs=torch.tensor(cow, dtype=torch.int32).to(device),
                    info={"prefix_tokens": prefix, "shared_blocks": shared,
                          "suffix_tokens": T})



# ------------------------------------------------------------------ multi-query
@dataclass
class PrefillWorkload:
    """Inputs of one causal multi-query (prefill / chunked-prefill) call: the
    pools already hold every request's context_lens[b] tokens, the last
    qlens[b] of which are this call's query rows."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    num_blocks: int
    dtype: torch.dtype
    scale: float
    q: torch.Tensor             # [T, Hq, D], T = sum(qlens)
    k_pool: torch.Tensor        # [NB, Hkv, bs, D]
    v_pool: torch.Tensor
    block_tables: torch.Tensor  # [B, MB] int32, -1 past each request's blocks
    context_lens: torch.Tensor  # [B] int32
    query_start: torch.Tensor   # [B + 1] int32
    max_query_len: int
    info: dict = field(default_factory=dict)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def T(self) -> int:
        return int(self.q.shape[0])


def make_prefill(*, B, Hq, Hkv, D, lens, qlens, num_blocks, dtype=torch.float16, seed=11,
                 contiguous_p=0.0, max_blocks=None, device="cpu", name="prefill_custom",
                 nan_sentinel=True, shared_blocks=0) -> PrefillWorkload:
    """Request b: lens[b] cached tokens, its last qlens[b] are queries
    (qlens[b] <= lens[b]).  shared_blocks > 0: the first that many blocks of
    every request are the same physical blocks (a cached prompt prefix; each
    lens[b] must cover them).  Seeds base = seed * 100: k = 0 q, 1 K pool, 2 V
    pool, 5 tables.  Slots past every request's tokens hold NaN (16-bit)."""
    lens = [int(x) for x in lens]
    qlens = [int(x) for x in qlens]
    if len(lens) != B or len(qlens) != B:
        raise ValueError("lens and qlens need one entry per request")
    nblk = [-(-n // BLOCK_SIZE) for n in lens]
    mb = max_blocks if max_blocks is not None else max(1, max(nblk) if nblk else 1)
    S = int(shared_blocks)
    if S and any(n < S * BLOCK_SIZE for n in lens):
        raise ValueError("every request must hold the whole shared prefix")
    if S + sum(n - S for n in nblk) > num_blocks:
        raise ValueError("pool too small for the requested lengths")
    base = seed * 100
    rng = np.random.default_rng(base + 5)
    if S:
        shared = _draw_tables(rng, [S], num_blocks, contiguous_p)[0]
        rest = _draw_tables(rng, [n - S for n in nblk], num_blocks, contiguous_p,
                            taken=shared)
        lists = [shared + r for r in rest]
    else:
        lists = _draw_tables(rng, nblk, num_blocks, contiguous_p)
    tables = _tables_from_lists(lists, mb)
    T = sum(qlens)
    q = _randn((max(T, 1), Hq, D), dtype, base + 0, device)[:T]
    k_pool = _randn((num_blocks, Hkv, BLOCK_SIZE, D), dtype, base + 1, device)
    v_pool = _randn((num_blocks, Hkv, BLOCK_SIZE, D), dtype, base + 2, device)
    if nan_sentinel:
        _nan_unfilled(k_pool, tables, lens)
        _nan_unfilled(v_pool, tables, lens)
    qs = [0]
    for L in qlens:
        qs.append(qs[-1] + L)
    return PrefillWorkload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, num_blocks=num_blocks,
                           dtype=dtype, scale=1.0 / math.sqrt(D), q=q, k_pool=k_pool,
                           v_pool=v_pool, block_tables=tables.to(device),
                           context_lens=torch.tensor(lens, dtype=torch.int32).to(device),
                           query_start=torch.tensor(qs, dtype=torch.int32).to(device),
                           max_query_len=max(qlens) if qlens else 0)


PREFILL_NAMES = ("prefix_prefill",)


def make_prefill_named(name: str, device="cpu", nan_sentinel=True,
                       batch=None) -> PrefillWorkload:
    """prefix_prefill: the prefix-sharing workload's prompt pass with the prefix
    cached ("ATB KV Cache management", "Prefix Caching"): 128 requests (32/32
    heads, D 128, fp16, 8192-block pool) whose tables share the 1030-token
    prefix blocks; each request's private suffix (U[16, 512] tokens, already
    appended) is its chunk of queries, attending causally to prefix + suffix.
    Same tables and lengths as the `prefix` decode workload; q drawn with seed
    base + 0 as [T, Hq, D].  ``batch`` keeps the first requests only."""
    if name != "prefix_prefill":
        raise KeyError(name)
    seed = 1000 + WORKLOAD_NAMES.index("prefix")
    src = _make_prefix(seed, device, False)
    prefix = src.info["prefix_tokens"]
    lens = [int(x) for x in src.context_lens.cpu()]
    B = len(lens) if batch is None else min(int(batch), len(lens))
    lens = lens[:B]
    tables = src.block_tables[:B].cpu().clone()
    qlens = [n - prefix for n in lens]
    T = sum(qlens)
    base = seed * 100
    q = _randn((T, src.Hq, src.D), torch.float16, base + 0, device)
    k_pool, v_pool = src.k_pool.to(device), src.v_pool.to(device)
    if nan_sentinel:
        _nan_unfilled(k_pool, tables, lens)
        _nan_unfilled(v_pool, tables, lens)
    qs = [0]
    for L in qlens:
        qs.append(qs[-1] + L)
    return PrefillWorkload(name=name, B=B, Hq=src.Hq, Hkv=src.Hkv, D=src.D,
                           num_blocks=src.num_blocks, dtype=torch.float16, scale=src.scale,
                           q=q, k_pool=k_pool, v_pool=v_pool, block_tables=tables.to(device),
                           context_lens=torch.tensor(lens, dtype=torch.int32).to(device),
                           query_start=torch.tensor(qs, dtype=torch.int32).to(device),
                           max_query_len=max(qlens),
                           info={"prefix_tokens": prefix, "query_tokens": T,
                                 # the prefix's full blocks are shared physically; its
                                 # partial last block was copied per request on write
                                 "shared_blocks": prefix // BLOCK_SIZE})
