#!/usr/bin/env python3
"""Benchmark of the paged-KV decode step on GB300.

One step = the whole hot path over one batch: copy-on-write block copies (when
the workload has them), append of the step's new tokens (INT8-quantising for the
INT8 workload), paged decode attention (partition pass + reduce).  Inputs are
resident in HBM when the timed region starts; `value` is whole-job achieved HBM
GB/s over the step's algorithmic bytes, timed with CUDA events on the launching
stream around the K steps only; the dominant kernel's own time (the roofline
numerator) comes from a separate pass of the same steps with events around it.
Prints ONE JSON line (rank 0).

The default run (llama7b, the configuration the metric is quoted on) also
times, each in a timed region of its own, the GQA-70B, INT8 and FP8 long-context
and prefix-sharing decode workloads and the prefix-cached prompt pass
(prefix_prefill, TFLOP/s on the tensor roofline), under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

For N > 1 (torchrun) every rank runs an independent replica on its own GPU (the
decode has no exchange step): value = total bytes of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import shutil
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = ("paged-attention decode achieved HBM GB/s (% of peak) and attended KV tokens/s")
PREFILL_METRIC = ("paged-attention prefill of prefix-cached prompts: achieved tensor TFLOP/s "
                  "(causal attention FLOPs) and query tokens/s")
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["kvp_decode.cuh", "kvp_device.cuh", "kvp_decode_simt.cu", "kvp_decode_mma.cu",
                  "kvp_decode_int8.cu", "kvp_decode_fp8.cu", "kvp_decode_fp8_umma.cu",
                  "kvp_umma.cuh", "kvp_internal.h"]
PREFILL_SOURCES = ["kvp_prefill.cu", "kvp_umma.cuh", "kvp_device.cuh", "kvp_internal.h"]
# the shared-prefix decode runs the prefill kernel's prefix pass and the reduce too
SHARED_DECODE_SOURCES = KERNEL_SOURCES + ["kvp_prefill.cu", "kvp_reduce.cu"]


# ------------------------------------------------------------------ byte model
def kv_bytes_per_layer(Hkv: int, D: int, tokens: int, batch: int, elem_bytes: int) -> int:
    """2 (K and V) x kv heads x head_dim x tokens x batch x element bytes
    ("ATB KV Cache management", "KV Cache 的显存需求")."""
    return 2 * Hkv * D * tokens * batch * elem_bytes


def decode_bytes(w, lens) -> dict:
    """Algorithmic bytes of one decode call: K/V (and INT8 scales) of every
    attended token, the block-table entries read, q, out and context_lens."""
    elt = 1 if w.kv_int8 else 2
    qel = w.q.element_size()
    kv = sum(kv_bytes_per_layer(w.Hkv, w.D, n, 1, elt) for n in lens)
    scales = sum(2 * w.Hkv * n * 4 for n in lens) if w.kv_int8 else 0
    tables = sum(4 * (-(-n // 16)) for n in lens)
    q = w.B * w.Hq * w.D * qel
    return {"kv": kv, "scales": scales, "tables": tables, "q": q, "out": q, "lens": 4 * w.B,
            "partial_pass": kv + scales + tables + q + 4 * w.B,
            "call": kv + scales + tables + 2 * q + 4 * w.B}


def unique_kv_bytes(w, lens) -> int:
    """K/V (and INT8 scale) bytes of the distinct physical token slots a decode
    call reads: where requests share blocks (a cached prefix) each shared
    token counts once -- the least the call must move from HBM."""
    tab = w.block_tables.cpu()
    seen = set()
    for b, n in enumerate(lens):
        nfull, rem = divmod(n, 16)
        for i in range(nfull):
            seen.add((int(tab[b, i]), 16))
        if rem:
            seen.add((int(tab[b, nfull]), rem))
    # a block read with several lengths counts with its longest
    longest = {}
    for blk, k in seen:
        longest[blk] = max(longest.get(blk, 0), k)
    tokens = sum(longest.values())
    elt = 1 if w.kv_int8 else 2
    return tokens * (2 * w.Hkv * w.D * elt + (2 * w.Hkv * 4 if w.kv_int8 else 0))


def append_bytes(w) -> int:
    T, Hkv, D = int(w.slot_mapping.numel()), w.Hkv, w.D
    if w.kv_int8:  # read fp16 K and V, write int8 codes and fp32 scales
        return 2 * T * Hkv * D * 2 + 2 * T * Hkv * D + 2 * T * Hkv * 4 + 4 * T
    return 2 * 2 * T * Hkv * D * 2 + 4 * T


def copy_bytes(w) -> int:
    if w.cow_pairs is None:
        return 0
    P = int(w.cow_pairs.shape[0])
    block = w.Hkv * 16 * w.D * (1 if w.kv_int8 else 2)
    return P * 2 * block * 2 + 8 * P


# ------------------------------------------------------------------ helpers
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s)"


def measured_tensor_peak():
    """Dense 16-bit tensor peak in TFLOP/s (fp16 and bf16 run at one rate): the
    burst figure, for a kernel timed in steps of a few milliseconds."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback (1.9 PFLOP/s bf16 burst)"


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, "pagedattention_decode_kvp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, sources=None):
    """Per-launch DRAM bytes of the workload's dominant kernel from a committed
    ncu summary, valid only while the kernel sources are unchanged."""
    want = kernel_source_hash(sources)
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    pat = re.compile(r"traffic: workload=(\S+) kernel_src_sha=(\S+) bytes_per_launch=(\d+)")
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as fh:
            for m in pat.finditer(fh.read()):
                if m.group(1) == workload and m.group(2) == want:
                    return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        if shutil.which("nvidia-smi") is None:
            return self
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen(
            ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
             "--format=csv,noheader,nounits", "-lms", "100"],
            stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.send_signal(signal.SIGTERM)
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        sm = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "sm_mhz_min": min(sm), "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ the GPU arm
class Step:
    """Device buffers of one workload and the step through the public API."""

    def __init__(self, w, kvp, dev, partition_blocks=0, fused=False, merge_runs=False,
                 shared_prefix=0):
        self.w, self.kvp, self.dev = w, kvp, dev
        # > 0: the requests' first `shared_prefix` table entries are the same
        # physical blocks, decoded by kvp_attention_decode_shared_prefix
        self.shared = shared_prefix if not w.kv_int8 else 0
        # the run-merged fetch rides on the phases argument of every decode call
        self.flags = kvp.KVP_DECODE_MERGE_RUNS if merge_runs else 0
        # the fused step needs one new token per request at position n - 1
        self.fused = fused and not w.kv_int8 and w.cow_pairs is None and \
            int(w.slot_mapping.numel()) == w.B
        self.q = w.q.to(dev)
        self.tables = w.block_tables.to(dev)
        self.lens = w.context_lens.to(dev)
        self.slots = w.slot_mapping.to(dev)
        self.new_k = w.new_k.to(dev)
        self.new_v = w.new_v.to(dev)
        self.pairs = w.cow_pairs.to(dev) if w.cow_pairs is not None else None
        self.out = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        if w.kv_int8:
            self._init_int8()
        else:
            self.kp = w.k_pool.to(dev)
            self.vp = w.v_pool.to(dev)
        desc = kvp.cache_desc(self.kp)
        self.pb_arg = partition_blocks
        nb = kvp.kvp_decode_workspace_bytes(w.B, w.Hq, desc, w.max_blocks, partition_blocks,
                                            w.kv_int8 and not w.kv_fp8, w.kv_fp8)
        if self.shared:
            nb = kvp.kvp_decode_shared_prefix_workspace_bytes(w.B, w.Hq, desc, w.max_blocks,
                                                              self.shared, partition_blocks)
        self.ws = torch.empty(max(nb // 4, 1), dtype=torch.float32, device=dev) if nb else None
        self.split = nb > 0
        self.part_blocks = (min(partition_blocks, w.max_blocks) if partition_blocks else
                            kvp.kvp_decode_partition_blocks(w.B, w.Hq, desc, w.max_blocks,
                                                            w.kv_int8 and not w.kv_fp8,
                                                            w.kv_fp8))

    def _init_int8(self):
        """Quantise the fp16 source pools into the INT8 pools on the GPU: each
        row is independent, so the pool is appended to itself as
        NB*Hkv*16 single-head tokens (the long-context prefill)."""
        w, kvp = self.w, self.kvp
        NB, Hkv, D = w.num_blocks, w.Hkv, w.D
        ks, vs = w.k_pool.to(self.dev), w.v_pool.to(self.dev)
        code_dtype = torch.uint8 if w.kv_fp8 else torch.int8
        self.kp = torch.empty(NB, Hkv, 16, D, dtype=code_dtype, device=self.dev)
        self.vp = torch.empty_like(self.kp)
        self.ks = torch.empty(NB, Hkv, 16, dtype=torch.float32, device=self.dev)
        self.vs = torch.empty_like(self.ks)
        rows = NB * Hkv * 16
        slots = torch.arange(rows, dtype=torch.int32, device=self.dev)
        flat = lambda t: t.view(NB * Hkv, 1, 16, *t.shape[3:])  # noqa: E731
        append = kvp.kvp_append_fp8 if w.kv_fp8 else kvp.kvp_append_int8

        def quantise_all():
            append(ks.view(rows, 1, D), vs.view(rows, 1, D), flat(self.kp), flat(self.vp),
                   flat(self.ks), flat(self.vs), slots)

        quantise_all()  # warm-up (first launch of the kernel)
        reps = 3
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            quantise_all()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        moved = rows * D * 2 * 2 + rows * D * 2 + rows * 4 * 2
        self.prefill = {"rows": rows, "ms": round(ms, 5), "gbs": round(moved / ms / 1e6, 2),
                        "bytes": moved, "launches_timed": reps}
        del ks, vs

    def launches_per_step(self) -> int:
        append = 0 if self.fused else 1
        decode = 3 if self.shared else 1 + (1 if self.split else 0)  # (prefix pass, split, reduce)
        return (1 if self.pairs is not None else 0) + append + decode

    def run(self, ev=None):
        """One step; ev = (e_decode_start, e_partial_end) events to record."""
        kvp, w = self.kvp, self.w
        if self.fused:
            if ev is not None:
                ev[0].record()
            phases = [kvp.KVP_PHASE_PARTIAL, kvp.KVP_PHASE_REDUCE] if self.split else \
                [kvp.KVP_PHASE_ALL]
            for i, ph in enumerate(phases):
                kvp.kvp_append_attention_decode(self.new_k, self.new_v, self.out, self.q, self.kp,
                                                self.vp, self.tables, self.lens, w.scale,
                                                workspace=self.ws, phases=ph | self.flags,
                                                status=self.status,
                                                partition_blocks=self.pb_arg)
                if ev is not None and i == 0:
                    ev[1].record()
            return
        if self.pairs is not None:
            kvp.kvp_copy_blocks(self.kp, self.vp, self.pairs, status=self.status)
        if w.kv_int8:
            append = kvp.kvp_append_fp8 if w.kv_fp8 else kvp.kvp_append_int8
            append(self.new_k, self.new_v, self.kp, self.vp, self.ks, self.vs, self.slots,
                   status=self.status)
        else:
            kvp.kvp_append(self.new_k, self.new_v, self.kp, self.vp, self.slots,
                           status=self.status)
        if ev is not None:
            ev[0].record()
        if self.shared:
            kvp.kvp_attention_decode_shared_prefix(self.out, self.q, self.kp, self.vp, self.tables,
                                                   self.lens, w.scale, self.shared,
                                                   workspace=self.ws, status=self.status,
                                                   partition_blocks=self.pb_arg)
            if ev is not None:
                ev[1].record()
            return
        phases = [kvp.KVP_PHASE_PARTIAL, kvp.KVP_PHASE_REDUCE] if self.split else [kvp.KVP_PHASE_ALL]
        for i, ph in enumerate(phases):
            if w.kv_int8:
                decode = kvp.kvp_attention_decode_fp8 if w.kv_fp8 else \
                    kvp.kvp_attention_decode_int8
                decode(self.out, self.q, self.kp, self.vp, self.ks,
                       self.vs, self.tables, self.lens, w.scale, workspace=self.ws,
                       phases=ph | self.flags, status=self.status,
                       partition_blocks=self.pb_arg)
            else:
                kvp.kvp_attention_decode(self.out, self.q, self.kp, self.vp, self.tables,
                                         self.lens, w.scale, workspace=self.ws,
                                         phases=ph | self.flags, status=self.status,
                                         partition_blocks=self.pb_arg)
            if ev is not None and i == 0:
                ev[1].record()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_baseline(w, host_k, host_v, host_ks=None, host_vs=None, rows=None):
    """Time the CPU oracle (as it stands) on a sample of the decode."""
    import oracle
    lens = [int(x) for x in w.context_lens]
    if rows is None:
        rows = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    t0 = time.perf_counter()
    oracle.attention_decode(w.q, host_k, host_v, w.block_tables, w.context_lens, w.scale,
                            k_scale=host_ks, v_scale=host_vs, rows=rows)
    dt = time.perf_counter() - t0
    G = w.Hq // w.Hkv
    elt = 1 if w.kv_int8 else 2
    # bytes the sampled rows read: each (b, h) row reads its K/V once per query
    # head of the group, so count the sample as the fraction of the full call
    frac = len(rows) / (w.B * w.Hq)
    sampled_tokens = sum(lens[b] for b, _ in rows)
    full = decode_bytes(w, lens)["call"]
    return {"seconds": dt, "bytes": full * frac, "tokens": sampled_tokens / G,
            "rows": len(rows), "cores": oracle.num_threads(), "elt": elt}


def timed_region(run, steps, world, dev, local):
    """K steps bracketed by a barrier and a device synchronize on both sides,
    timed by two CUDA events on the launching stream (nothing else is recorded
    inside the region, so the kernels' programmatic launch overlap is kept);
    nvidia-smi clocks are sampled meanwhile.  Returns (max-over-ranks ms,
    clock summary)."""
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(steps):
            run()
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(start.elapsed_time(end), world, dev), clk.summary()


def kernel_pass(run_ev, steps) -> float:
    """Mean duration (ms) of the step's dominant kernel over a separate pass of
    K steps, from events recorded right before and right after it on the
    launching stream."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        run_ev(evs[i])
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)


def check_status(kvp, status, what):
    st = kvp.kvp_read_status(status)
    if st != kvp.KVP_OK:
        raise RuntimeError(f"{what}: device status {kvp.kvp_status_string(st)}")


def dtype_name(w) -> str:
    base = {torch.float16: "f16", torch.bfloat16: "bf16"}[w.dtype]
    if w.kv_int8:
        return base + (" (fp8 e4m3 KV)" if w.kv_fp8 else " (int8 KV)")
    return base


def measure_decode(name, args, kvp, world, dev, local, headline):
    """Build one decode workload on the device, warm up, time K steps (outer
    events only), then time its partition kernel in a separate pass.  Returns
    (workload, step, measurement dict)."""
    w = workloads.make(name, device=dev, nan_sentinel=False,
                       batch=args.batch if headline else None,
                       contiguity=args.contiguity if headline else None)
    # the prefix-sharing workload's first 64 table entries are the shared
    # prefix's full blocks (its partial last block is copied per request)
    shared = (w.info["prefix_tokens"] // 16 if w.cow_pairs is not None and
              not (headline and args.no_shared_prefix) else 0)
    step = Step(w, kvp, dev, args.partition_blocks if headline else 0, fused=not args.unfused,
                merge_runs=headline and args.merge_runs, shared_prefix=shared)
    lens = [int(x) for x in w.context_lens]
    dbytes = decode_bytes(w, lens)
    sbytes = dbytes["call"] + append_bytes(w) + copy_bytes(w)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    check_status(kvp, step.status, f"{name} after warm-up")
    elapsed_ms, clocks = timed_region(step.run, args.steps, world, dev, local)
    partial_ms = kernel_pass(step.run, args.steps)
    check_status(kvp, step.status, f"{name} after the timed steps")
    total_bytes = sum_over_ranks(sbytes * args.steps, world, dev)
    value = total_bytes / (elapsed_ms / 1e3) / 1e9
    tokens_per_s = sum_over_ranks(sum(lens) * args.steps, world, dev) / (elapsed_ms / 1e3)
    peak, peak_src = measured_peak()
    # the fused partition pass also moves the appended rows (read source, write slot)
    partial_bytes = dbytes["partial_pass"] + (append_bytes(w) if step.fused else 0)
    achieved = partial_bytes / (partial_ms / 1e3) / 1e9
    # the committed counters are for the full-size workloads only
    full_size = not (headline and (args.batch or args.contiguity is not None))
    traffic = (profiled_traffic(name, SHARED_DECODE_SOURCES if step.shared else None)
               if full_size else None)
    m = {
        "value": round(value, 2),
        "unit": "GB/s",
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "tokens_per_s": round(tokens_per_s, 1),
        "pct_of_peak": round(100 * value / peak, 2),
        "dtype": dtype_name(w),
        "config": {"workload": w.name + (f" (batch {w.B})" if headline and args.batch else ""),
                   "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D,
                   "block_size": 16, "num_blocks": w.num_blocks, "context_tokens": sum(lens),
                   "max_context": max(lens), "new_tokens": int(w.slot_mapping.numel()),
                   "cow_pairs": int(w.cow_pairs.shape[0]) if w.cow_pairs is not None else 0,
                   "partition_blocks": step.part_blocks,
                   "shared_prefix_blocks": step.shared,
                   "append": "fused into the decode" if step.fused else "separate kernel",
                   "fetch": "runs of consecutive blocks" if step.flags else "per block",
                   "l2": ("inputs larger than L2: {:.2f} GB of K/V per step vs 129 MB L2"
                          .format(dbytes["kv"] / 1e9)) if dbytes["kv"] > 4 * L2_BYTES else
                         "inputs partly L2-resident (L2 reuse is part of this workload)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "step_bytes": sbytes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("decode_fp8_umma_kernel" if w.kv_fp8 and w.D == 128 else
                                "prefix pass + decode_partial_kernel + reduce" if step.shared
                                else "decode_partial_kernel"), "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": partial_bytes,
                     "launch_ms": round(partial_ms, 5),
                     "timing": "kernel events in a separate pass of the same steps"},
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clocks,
    }
    if "contiguous_share" in w.info:
        m["config"]["contiguous_share"] = round(w.info["contiguous_share"], 4)
    if w.cow_pairs is not None:
        # shared prefix blocks: L2 serves every request after the first, so the
        # HBM roofline is taken on the distinct bytes; the logical figure
        # (every request's whole context) is kept beside it
        ubytes = unique_kv_bytes(w, lens)
        upartial = partial_bytes - dbytes["kv"] - dbytes["scales"] + ubytes
        r = m["roofline"]
        r["achieved_logical"] = r["achieved"]
        r["algorithmic_bytes_logical"] = partial_bytes
        r["achieved"] = round(upartial / (partial_ms / 1e3) / 1e9, 2)
        r["frac"] = round(r["achieved"] / peak, 4)
        r["algorithmic_bytes_per_launch"] = upartial
        r["bytes"] = "distinct physical K/V slots (shared prefix once)"
        m["value_unique"] = round((sbytes - dbytes["kv"] - dbytes["scales"] + ubytes)
                                  * args.steps / (elapsed_ms / 1e3) / 1e9, 2)
    if w.kv_int8:
        m["prefill_quantise"] = step.prefill
    return w, step, m, total_bytes


def decode_cpu_baseline(w, step, rows_all, rows_one):
    """The oracle as it stands on the host cores: `rows_all` (request, head)
    rows on every core (median of three runs) and `rows_one` rows on one core."""
    import oracle
    oracle.build()
    w_host = workloads.Workload(**{k: (v.cpu() if isinstance(v, torch.Tensor) else v)
                                   for k, v in w.__dict__.items()})
    hk, hv = step.kp.cpu(), step.vp.cpu()
    if w.kv_fp8:
        hk, hv = hk.view(torch.float8_e4m3fn), hv.view(torch.float8_e4m3fn)
    hks = step.ks.cpu() if w.kv_int8 else None
    hvs = step.vs.cpu() if w.kv_int8 else None
    rows = sample_rows(w, rows_all)
    runs = [cpu_oracle_baseline(w_host, hk, hv, hks, hvs, rows) for _ in range(3)]
    cb = sorted(runs, key=lambda r: r["seconds"])[1]
    res = {"value": round(cb["bytes"] / cb["seconds"] / 1e9, 4), "unit": "GB/s",
           "cores": cb["cores"], "kind": "oracle",
           "sample": f"{cb['rows']} of {w.B * w.Hq} (request, query head) rows of one decode "
                     f"call, median of 3 runs, {cb['seconds']:.2f} s each"}
    if rows_one:
        threads = oracle.num_threads()
        oracle.set_num_threads(1)
        try:
            c1 = cpu_oracle_baseline(w_host, hk, hv, hks, hvs, sample_rows(w, rows_one))
        finally:
            oracle.set_num_threads(threads)
        res["value_1core"] = round(c1["bytes"] / c1["seconds"] / 1e9, 4)
        res["sample_1core"] = (f"{c1['rows']} (request, query head) rows on 1 core, "
                               f"{c1['seconds']:.2f} s")
    return res


def run_e2e(step, host_keys, args, world, dev, unit_total, unit_scale, unit):
    """The same steps end to end through the public API, as a serving loop runs
    them: every step's inputs are copied in from pinned host memory and its
    output back into pinned host memory, on two copy streams beside the
    compute stream and double-buffered, so that step k+1's inputs travel while
    step k computes and step k's output returns while step k+1 computes.  The
    inputs sit in one pinned host buffer (each 256-byte aligned) and a step's
    device inputs are views of one device buffer, so they travel in one copy.
    The timed region ends when the last output has landed in host memory."""
    keys = [k for k in host_keys if getattr(step, k, None) is not None]
    offs, total = {}, 0
    for k in keys:
        t = getattr(step, k)
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.zeros(max(total, 256), dtype=torch.uint8).pin_memory()
    dev_bufs = [torch.empty(max(total, 256), dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [{}, {}]
    for k in keys:
        t = getattr(step, k).contiguous()
        nb = t.numel() * t.element_size()
        host_buf[offs[k]:offs[k] + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
        for i in range(2):
            views[i][k] = dev_bufs[i][offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    outs = [step.out, torch.empty_like(step.out)]
    out_hosts = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = int(host_buf.numel())
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    comp = torch.cuda.current_stream(dev)
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]   # buffer i's inputs landed
    done = [torch.cuda.Event() for _ in range(2)]       # the step on buffer i computed
    out_back = [torch.cuda.Event() for _ in range(2)]   # output i read back

    def e2e_step(k):
        i = k & 1
        with torch.cuda.stream(h2d_s):
            if k >= 2:
                h2d_s.wait_event(done[i])      # step k - 2 has read buffer i
            dev_bufs[i].copy_(host_buf, non_blocking=True)
            in_ready[i].record(h2d_s)
        comp.wait_event(in_ready[i])
        if k >= 2:
            comp.wait_event(out_back[i])       # step k - 2's output has left buffer i
        for key, v in views[i].items():
            setattr(step, key, v)
        step.out = outs[i]
        step.run()
        done[i].record(comp)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(done[i])
            out_hosts[i].copy_(outs[i], non_blocking=True)
            out_back[i].record(d2h_s)

    for k in range(args.warmup):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for k in range(args.steps):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    barrier(world)
    step.out = outs[0]
    return {"value": round(unit_total / e2e_s / unit_scale, 3), "unit": unit,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_s * 1e3 / args.steps, 4),
            "copies": "every step: inputs in, output back; two copy streams beside the compute "
                      "stream, double-buffered"}


EXTRA_DECODE = ("gqa70b", "int8long", "fp8long", "prefix")
EXTRA_PREFILL = ("prefix_prefill",)


def run_ours(args):
    import pagedattention_decode_kvp_gb300 as kvp
    from pagedattention_decode_kvp_gb300 import _build

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    kvp.load_library()

    w, step, m, total_bytes = measure_decode(args.workload, args, kvp, world, dev, local, True)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, ("q", "tables", "lens", "slots", "new_k", "new_v", "pairs"), args,
                      world, dev, total_bytes, 1e9, "GB/s")

    res = {"metric": METRIC, "value": m["value"], "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": m["dtype"],
           "data": "synthetic (seeded N(0,1), shapes of the pages' workloads)",
           "config": m["config"], "tokens_per_s": m["tokens_per_s"],
           "pct_of_peak": m["pct_of_peak"], "step_bytes": m["step_bytes"],
           "roofline": m["roofline"], "e2e": e2e, "gpu_launches": m["gpu_launches"],
           "clocks": m["clocks"]}
    if "prefill_quantise" in m:
        res["prefill_quantise"] = m["prefill_quantise"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = decode_cpu_baseline(w, step, args.cpu_rows, args.cpu_rows_1core)
    del step, w
    torch.cuda.empty_cache()

    # the other workloads of the same method, each timed the same way in this run
    extras = {}
    if args.extras:
        for name in EXTRA_DECODE:
            ew, estep, em, _ = measure_decode(name, args, kvp, world, dev, local, False)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                em["cpu_baseline"] = decode_cpu_baseline(ew, estep, 16 if ew.kv_int8 else 64, 0)
            extras[name] = em
            del estep, ew
            torch.cuda.empty_cache()
        for name in EXTRA_PREFILL:
            pw, pstep, pm, _ = measure_prefill(name, args, kvp, world, dev, local, False)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                pm["cpu_baseline"] = prefill_cpu_baseline(pw, pstep, 1024)
            extras[name] = pm
            del pstep, pw
            torch.cuda.empty_cache()
        res["workloads"] = extras

    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ prefill workloads
def prefill_work(w):
    """(FLOPs, attended (query row, key) pairs per head) of one causal
    multi-query call: row i of a chunk of L rows at context n attends to
    n - L + i + 1 keys; q.K and p.V cost 2 * D FLOPs per key each."""
    lens = [int(x) for x in w.context_lens.cpu()]
    qs = [int(x) for x in w.query_start.cpu()]
    pairs = 0
    for b, n in enumerate(lens):
        L = qs[b + 1] - qs[b]
        pairs += L * (n - L) + L * (L + 1) // 2
    return 4 * w.D * w.Hq * pairs, pairs


class PrefillStep:
    """One prompt pass through the public API: append the chunk's K/V into its
    slots (kvp_append), then causal multi-query attention
    (kvp_attention_prefill)."""

    def __init__(self, w, kvp, dev, shared_blocks=0):
        self.w, self.kvp = w, kvp
        self.shared = shared_blocks  # > 0: dense tiles over the shared prefix
        self.q = w.q.to(dev)
        self.kp, self.vp = w.k_pool.to(dev), w.v_pool.to(dev)
        self.tables = w.block_tables.to(dev)
        self.lens = w.context_lens.to(dev)
        self.qs = w.query_start.to(dev)
        lens = [int(x) for x in w.context_lens.cpu()]
        qs = [int(x) for x in w.query_start.cpu()]
        tab = w.block_tables.cpu()
        slots = [int(tab[b, p // 16]) * 16 + p % 16 for b, n in enumerate(lens)
                 for p in range(n - (qs[b + 1] - qs[b]), n)]
        self.slots = torch.tensor(slots, dtype=torch.int32, device=dev)
        blk, off = (self.slots // 16).long(), (self.slots % 16).long()
        # the chunk's K/V rows are the ones the pool already holds at those slots,
        # so every step's append rewrites them unchanged
        self.new_k = self.kp[blk, :, off, :].contiguous()
        self.new_v = self.vp[blk, :, off, :].contiguous()
        self.out = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def append_bytes(self) -> int:
        T = int(self.slots.numel())
        return 2 * 2 * T * self.w.Hkv * self.w.D * 2 + 4 * T

    def run(self, ev=None):
        kvp, w = self.kvp, self.w
        kvp.kvp_append(self.new_k, self.new_v, self.kp, self.vp, self.slots, status=self.status)
        if ev is not None:
            ev[0].record()
        kvp.kvp_attention_prefill(self.out, self.q, self.kp, self.vp, self.tables, self.lens,
                                  self.qs, w.max_query_len, w.scale,
                                  shared_prefix_blocks=self.shared, status=self.status)
        if ev is not None:
            ev[1].record()


def prefill_sample_rows(w, n):
    total = w.T * w.Hq
    n = min(n, total)
    stride = total / n
    return [(int(i * stride) // w.Hq, int(i * stride) % w.Hq) for i in range(n)]


def cpu_oracle_prefill(w, host_k, host_v, rows):
    """Time the CPU oracle (as it stands) on sampled (query row, head) pairs of
    one prefill call; FLOPs counted as the GPU's (4 * D per attended key)."""
    import oracle
    import numpy as np
    lens = [int(x) for x in w.context_lens.cpu()]
    qs = [int(x) for x in w.query_start.cpu()]
    starts = np.array(qs[:-1])
    keys = 0
    for t, _ in rows:
        b = int(np.searchsorted(starts, t, side="right")) - 1
        while qs[b + 1] == qs[b]:
            b += 1
        keys += lens[b] - (qs[b + 1] - qs[b]) + (t - qs[b]) + 1
    t0 = time.perf_counter()
    oracle.attention_prefill(w.q, host_k, host_v, w.block_tables, w.context_lens,
                             w.query_start, w.scale, rows=np.array(rows, dtype=np.int32))
    dt = time.perf_counter() - t0
    return {"seconds": dt, "flops": 4.0 * w.D * keys, "rows": len(rows), "keys": keys,
            "cores": oracle.num_threads()}


def measure_prefill(name, args, kvp, world, dev, local, headline):
    """Build a prefill workload on the device, warm up, time K steps (outer
    events only), then time the prefill kernel in a separate pass."""
    w = workloads.make_prefill_named(name, device=dev, nan_sentinel=False,
                                     batch=args.batch if headline else None)
    shared = 0 if (headline and args.per_request_tiles) else w.info.get("shared_blocks", 0)
    step = PrefillStep(w, kvp, dev, shared)
    flops, pairs = prefill_work(w)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    check_status(kvp, step.status, f"{name} after warm-up")
    elapsed_ms, clocks = timed_region(step.run, args.steps, world, dev, local)
    kernel_ms = kernel_pass(step.run, args.steps)
    check_status(kvp, step.status, f"{name} after the timed steps")
    total_flops = sum_over_ranks(flops * args.steps, world, dev)
    value = total_flops / (elapsed_ms / 1e3) / 1e12
    q_tokens_per_s = sum_over_ranks(w.T * args.steps, world, dev) / (elapsed_ms / 1e3)
    peak, peak_src = measured_tensor_peak()
    achieved = flops / (kernel_ms / 1e3) / 1e12
    full_size = not (headline and args.batch)
    m = {
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "query_tokens_per_s": round(q_tokens_per_s, 1),
        "dtype": {torch.float16: "f16", torch.bfloat16: "bf16"}[w.dtype],
        "config": {"workload": w.name + (f" (batch {w.B})" if headline and args.batch else ""),
                   "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D,
                   "block_size": 16, "num_blocks": w.num_blocks, "query_tokens": w.T,
                   "prefix_tokens": w.info.get("prefix_tokens"),
                   "tiles": (f"dense over all requests' rows ({shared} shared prefix blocks)"
                             if shared else "per request"),
                   "context_tokens": int(w.context_lens.sum()),
                   "attended_pairs_per_head": pairs,
                   "l2": "K/V of the shared prefix is L2-resident across requests (prefix "
                         "reuse is part of this workload); the chunk's append writes "
                         "{:.2f} GB per step".format(step.append_bytes() / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(name, PREFILL_SOURCES) if full_size else None,
                     "kernel": "prefill_kernel", "peak_source": peak_src,
                     "algorithmic_flops_per_launch": flops,
                     "launch_ms": round(kernel_ms, 5),
                     "timing": "kernel events in a separate pass of the same steps"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    return w, step, m, total_flops


def prefill_cpu_baseline(w, step, nrows):
    import oracle
    oracle.build()
    wh = workloads.PrefillWorkload(**{k: (v.cpu() if isinstance(v, torch.Tensor) else v)
                                      for k, v in w.__dict__.items()})
    cb = cpu_oracle_prefill(wh, step.kp.cpu(), step.vp.cpu(), prefill_sample_rows(wh, nrows))
    return {"value": round(cb["flops"] / cb["seconds"] / 1e12, 6), "unit": "TFLOP/s",
            "cores": cb["cores"], "kind": "oracle",
            "sample": f"{cb['rows']} of {w.T * w.Hq} (query row, head) pairs of one prefill "
                      f"call, {cb['seconds']:.2f} s"}


def run_prefill(args):
    import pagedattention_decode_kvp_gb300 as kvp
    from pagedattention_decode_kvp_gb300 import _build

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    kvp.load_library()

    w, step, m, total_flops = measure_prefill(args.workload, args, kvp, world, dev, local, True)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, ("q", "tables", "lens", "qs", "slots", "new_k", "new_v"), args,
                      world, dev, total_flops, 1e12, "TFLOP/s")
    res = {"metric": PREFILL_METRIC, "value": m["value"], "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": m["dtype"],
           "data": "synthetic (seeded N(0,1), shapes of the pages' prefix-sharing workload)",
           "config": m["config"], "query_tokens_per_s": m["query_tokens_per_s"],
           "roofline": m["roofline"], "e2e": e2e, "gpu_launches": m["gpu_launches"],
           "clocks": m["clocks"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = prefill_cpu_baseline(w, step, args.cpu_rows)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference_prefill(args):
    """The CPU oracle as the reference arm of a prefill workload (rank 0 only)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = workloads.make_prefill_named(args.workload, device="cpu", nan_sentinel=False,
                                     batch=args.batch)
    rows = prefill_sample_rows(w, args.cpu_rows)
    for _ in range(args.warmup):
        cpu_oracle_prefill(w, w.k_pool, w.v_pool, rows)
    secs = flops = 0.0
    for _ in range(args.steps):
        cb = cpu_oracle_prefill(w, w.k_pool, w.v_pool, rows)
        secs += cb["seconds"]
        flops += cb["flops"]
    value = flops / secs / 1e12
    sample = f"{cb['rows']} of {w.T * w.Hq} (query row, head) pairs of one prefill call per step"
    res = {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6),
           "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
           "data": "synthetic (seeded N(0,1))",
           "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
                      "head_dim": w.D, "query_tokens": w.T},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cb["cores"],
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def sample_rows(w, n):
    total = w.B * w.Hq
    if n <= 0 or n >= total:
        return None
    stride = total / n
    return [(int(i * stride) // w.Hq, int(i * stride) % w.Hq) for i in range(n)]


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The CPU oracle as the reference arm, on the host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = workloads.make(args.workload, device=dev, nan_sentinel=False, batch=args.batch)
    w = workloads.Workload(**{k: (v.cpu() if isinstance(v, torch.Tensor) else v)
                              for k, v in w.__dict__.items()})
    kp, vp, ks, vs = w.k_pool, w.v_pool, None, None
    if w.kv_int8:
        quant = oracle.quantize_fp8 if w.kv_fp8 else oracle.quantize_int8
        kc, ksn = quant(kp)
        vc, vsn = quant(vp)
        kp, vp = torch.from_numpy(kc), torch.from_numpy(vc)
        if w.kv_fp8:
            kp, vp = kp.view(torch.float8_e4m3fn), vp.view(torch.float8_e4m3fn)
        ks, vs = torch.from_numpy(ksn), torch.from_numpy(vsn)
    rows = sample_rows(w, args.cpu_rows)
    for _ in range(args.warmup):
        cpu_oracle_baseline(w, kp, vp, ks, vs, rows)
    secs, nbytes, toks = 0.0, 0.0, 0.0
    for _ in range(args.steps):
        cb = cpu_oracle_baseline(w, kp, vp, ks, vs, rows)
        secs += cb["seconds"]
        nbytes += cb["bytes"]
        toks += cb["tokens"]
    value = nbytes / secs / 1e9
    sample = (f"{cb['rows']} of {w.B * w.Hq} (request, query head) rows of one decode call "
              "per step")
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None,
           "dtype": "f64 (oracle)", "data": "synthetic (seeded N(0,1))",
           "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
                      "head_dim": w.D},
           "tokens_per_s": round(toks / secs, 1),
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cb["cores"],
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama7b",
                    choices=workloads.WORKLOAD_NAMES + workloads.PREFILL_NAMES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="(request, head) rows the CPU oracle times (0 = default sample)")
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer requests (pool scaled in proportion), for profiler captures")
    ap.add_argument("--partition-blocks", type=int, default=0,
                    help="split-context partition size in blocks (0 = the library's choice)")
    ap.add_argument("--contiguity", type=float, default=None,
                    help="redraw llama7b/gqa70b block tables as runs with this probability")
    ap.add_argument("--unfused", action="store_true",
                    help="append with kvp_append, then decode (default: the fused entry point "
                         "where every request appends one token at its last position)")
    ap.add_argument("--merge-runs", action="store_true",
                    help="decode with the run-merged fetch (one copy per run of up to 4 "
                         "physically consecutive blocks)")
    ap.add_argument("--per-request-tiles", action="store_true",
                    help="prefill: 128-row tiles per request (default for prefix_prefill: "
                         "dense tiles over the shared prefix)")
    ap.add_argument("--cpu-rows-1core", type=int, default=128,
                    help="(request, head) rows the CPU oracle times on one core (0 = skip)")
    ap.add_argument("--no-extras", action="store_true",
                    help="time only the named workload (default for llama7b: also gqa70b, "
                         "int8long, fp8long, prefix and prefix_prefill, each in its own "
                         "timed region, reported under \"workloads\")")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="decode the prefix-sharing workload per request instead of with its "
                         "shared prefix attended once per kv head")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    prefill = args.workload in workloads.PREFILL_NAMES
    if args.cpu_rows == 0:
        if prefill:
            args.cpu_rows = 8192 if args.impl == "ours" else 2048
        else:
            args.cpu_rows = 1024 if args.impl == "ours" else 64
    args.extras = (not args.no_extras and args.workload == "llama7b" and args.batch is None
                   and args.contiguity is None and args.partition_blocks == 0
                   and not args.unfused and not args.merge_runs)
    if args.impl == "reference":
        (run_reference_prefill if prefill else run_reference)(args)
    else:
        (run_prefill if prefill else run_ours)(args)


if __name__ == "__main__":
    main()
