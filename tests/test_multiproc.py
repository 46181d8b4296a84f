"""The N > 1 path of bench.py on CPU: two gloo ranks, each an independent
replica (the decode has no exchange step), time = max over ranks, volume = sum
over ranks; the reference arm does its work on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        t = bench.max_over_ranks(1.0 + rank, world, "cpu")      # per-rank elapsed
        s = bench.sum_over_ranks(10.0 * (rank + 1), world, "cpu")  # per-rank bytes
        bench.barrier(world)
        q.put((rank, t, s))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replica_reduction():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t, s in res:
        assert t == 2.0      # max over ranks
        assert s == 30.0     # sum over ranks


def test_reference_arm_is_rank0_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload = "tiny"
        warmup = 3
        steps = 1
        cpu_rows = 8

    # rank 1 returns immediately without building or generating anything
    assert bench.run_reference(A()) is None


def test_byte_model_matches_the_pages():
    sys.path.insert(0, ROOT)
    import bench
    vals = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "kv_bytes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=")
            vals[k.strip()] = int(v)
    one = bench.kv_bytes_per_layer(vals["per_layer_heads"], vals["per_layer_head_dim"],
                                   vals["per_layer_tokens"], 1, vals["per_layer_dtype_bytes"])
    assert one == vals["per_layer_bytes_per_request"]
    assert bench.kv_bytes_per_layer(32, 128, 4096, 32, 2) == vals["per_layer_bytes_batch32"]
    assert bench.kv_bytes_per_layer(32, 128, vals["block_tokens"], 1, 2) == \
        vals["block_bytes_kv"]
