"""The benchmark's multi-rank path on CPU: two gloo ranks, each with its own
batch (weak scaling), combine their step times with a max all-reduce and
report the job-wide value (no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each rank: its own seeded batch of the prefill workload's length draw
    from gqa_attention_cu_gb300 import workloads
    lq, lkv = workloads.draw_lengths(workloads.WORKLOADS["bf16_prefill"],
                                     torch.Generator().manual_seed(rank))
    w = {"lq": lq, "lkv": lkv, "is_causal": True, "num_heads": 32, "kv_num_heads": 8,
         "head_size": 128, "v_head_size": 128, "dtype": "bf16"}
    flops, _ = bench.work_units(w)
    local_ms = 1.0 + rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    total = bench.sum_over_ranks(flops, world, torch.device("cpu"))
    q.put((rank, ms, flops, total))
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, ms0, f0, t0), (_, ms1, f1, t1) = res
    assert ms0 == ms1 == 2.0                  # max over ranks
    assert t0 == t1 == f0 + f1                # job-wide work = sum of the ranks'
    assert f0 != f1                           # independent batches per rank
