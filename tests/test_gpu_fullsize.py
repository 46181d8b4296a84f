"""GPU parity at the benchmarked sizes, through the exact step bench.py times.

Each decode workload (llama7b, gqa70b, prefix, int8long, fp8long) is drawn on
the host, run once through ``bench.Step`` (same entry points, fused or not,
same automatic split-context partitions), and checked against the oracle fed
the same host inputs: the appended slots, copy-on-write blocks and 8-bit codes
/ scales bit-exact; the attention output of every (request, head) row, element
by element, within 3e-3 absolute OR 1e-2 relative of the fp64 oracle.  Inputs
given to the oracle never come from the GPU.
"""
import numpy as np
import pytest
import torch

import bench
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


def assert_close(got, ref, what):
    g = got.detach().double().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    ok = (err <= ATOL) | (err <= RTOL * np.abs(ref))
    if not ok.all():
        i = np.unravel_index(np.argmax(np.where(ok, 0, err)), err.shape)
        raise AssertionError(f"{what}: {int((~ok).sum())} elements out of tolerance; worst at "
                             f"{i}: gpu {g[i]} ref {ref[i]} (max abs err {err.max():.3e})")


def slot_rows(pool, slots):
    """Pool rows [T, Hkv, ...] at the given slots (block * 16 + offset)."""
    s = slots.long().cpu()
    return pool[s // 16, :, s % 16]


def run_step(name, merge_runs=False):
    w = workloads.make(name, device="cpu")
    step = bench.Step(w, kvp, torch.device("cuda"), 0, fused=True, merge_runs=merge_runs)
    step.run()
    torch.cuda.synchronize()
    assert kvp.kvp_read_status(step.status) == kvp.KVP_OK
    return w, step


@pytest.mark.parametrize("name", ["llama7b", "gqa70b", "prefix"])
def test_16bit_workload_full_size(name):
    w, step = run_step(name)
    okp, ovp = w.k_pool, w.v_pool
    if w.cow_pairs is not None:  # copy-on-write first, as the step does
        okp = oracle.copy_blocks(okp, w.cow_pairs)
        ovp = oracle.copy_blocks(ovp, w.cow_pairs)
    okp = oracle.append(okp, w.new_k, w.slot_mapping)
    ovp = oracle.append(ovp, w.new_v, w.slot_mapping)
    if w.cow_pairs is not None:  # the copied blocks, after the step's appends into them
        dst = w.cow_pairs[:, 1].long()
        assert torch.equal(step.kp[dst.cuda()].cpu().view(torch.int16), okp[dst].view(torch.int16))
        assert torch.equal(step.vp[dst.cuda()].cpu().view(torch.int16), ovp[dst].view(torch.int16))
    # the appended rows, bit for bit
    gk = slot_rows(step.kp.cpu(), w.slot_mapping)
    gv = slot_rows(step.vp.cpu(), w.slot_mapping)
    assert torch.equal(gk.view(torch.int16), slot_rows(okp, w.slot_mapping).view(torch.int16))
    assert torch.equal(gv.view(torch.int16), slot_rows(ovp, w.slot_mapping).view(torch.int16))
    ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
    assert_close(step.out, ref, f"{name} full size, every row")


@pytest.mark.parametrize("name", ["int8long", "fp8long"])
def test_8bit_workload_full_size(name):
    w, step = run_step(name)
    fp8 = name == "fp8long"
    quant = oracle.quantize_fp8 if fp8 else oracle.quantize_int8
    kc, ks = quant(w.k_pool)
    vc, vs = quant(w.v_pool)
    kc, vc = torch.from_numpy(kc), torch.from_numpy(vc)
    ks, vs = torch.from_numpy(ks), torch.from_numpy(vs)
    if fp8:
        kc, vc = kc.view(torch.float8_e4m3fn), vc.view(torch.float8_e4m3fn)
        okc, oks = oracle.append_fp8(kc, ks, w.new_k, w.slot_mapping)
        ovc, ovs = oracle.append_fp8(vc, vs, w.new_v, w.slot_mapping)
        raw = lambda t: t.view(torch.uint8)  # noqa: E731
    else:
        okc, oks = oracle.append_int8(kc, ks, w.new_k, w.slot_mapping)
        ovc, ovs = oracle.append_int8(vc, vs, w.new_v, w.slot_mapping)
        raw = lambda t: t  # noqa: E731
    # codes and scales of the appended rows and of a sample of quantised pool rows
    g = torch.Generator().manual_seed(3)
    probe = torch.cat([w.slot_mapping.cpu().to(torch.int64),
                       torch.randint(0, w.num_blocks * 16, (4096,), generator=g)])
    for gpu, ref in ((step.kp, okc), (step.vp, ovc)):
        assert torch.equal(slot_rows(raw(gpu.cpu()), probe), slot_rows(raw(ref), probe))
    for gpu, ref in ((step.ks, oks), (step.vs, ovs)):
        assert torch.equal(slot_rows(gpu.cpu(), probe).view(torch.int32),
                           slot_rows(ref, probe).view(torch.int32))
    ref = oracle.attention_decode(w.q, okc, ovc, w.block_tables, w.context_lens, w.scale,
                                  k_scale=oks, v_scale=ovs)
    assert_close(step.out, ref, f"{name} full size, every row")


def test_gqa70b_full_size_run_merged_fetch():
    """The GQA workload's tables are 85% runs of consecutive blocks: the
    run-merged fetch at full size, every row against the oracle."""
    w, step = run_step("gqa70b", merge_runs=True)
    okp = oracle.append(w.k_pool, w.new_k, w.slot_mapping)
    ovp = oracle.append(w.v_pool, w.new_v, w.slot_mapping)
    ref = oracle.attention_decode(w.q, okp, ovp, w.block_tables, w.context_lens, w.scale)
    assert_close(step.out, ref, "gqa70b full size, run-merged fetch")
