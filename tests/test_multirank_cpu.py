"""The N>1 benchmark logic on CPU with gloo (world_size 2): ranks draw distinct
batches (weak scaling), the job time is the max over ranks, and the job value
counts every rank's tokens.  No GPU and no data-path collective involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 10.0 + 5.0 * rank
        g = bench.global_elapsed_ms(local, world)
        from sparse_mla_attention_03_gb300 import inputs
        wl = inputs.make_prefill("shard", T=4, H=8, ctx=256, topk=32, seed=bench.rank_seed(0, rank))
        q.put((rank, g, wl.indices.sum().item()))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_sharding():
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
    (r0, g0, s0), (r1, g1, s1) = res
    assert g0 == g1 == 15.0          # max over ranks
    assert s0 != s1                  # distinct batches per rank
    assert bench.job_throughput(1024, 10, 2, 15.0) == pytest.approx(1024 * 10 * 2 / 0.015)
    assert bench.global_elapsed_ms(3.0, 1) == 3.0
