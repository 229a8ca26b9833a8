"""The multi-GPU path of bench.py: independent replicas (each rank its own prompts), a
timing barrier and the max over ranks. Exercised here on CPU with two gloo ranks."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    w = synth.WORKLOADS["llama8b_l16"]
    batch = bench.workload_batch(w, rank)
    bench.replica_barrier(world)
    elapsed = 1.0 + rank               # rank 1 is the slow replica
    mx = bench.max_over_ranks(elapsed, world)
    total = bench.sum_over_ranks(int(batch.cu_seqlens[-1]), world)
    value = bench.whole_job_throughput(total, 10, mx)
    out[rank] = (mx, value, int(batch.cu_seqlens[-1]), batch.tokens[:8].tolist(), batch.lens.tolist())
    dist.destroy_process_group()


def test_two_gloo_replicas_time_by_the_slowest_and_prefill_their_own_prompts():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (mx0, v0, t0, tok0, lens0), (mx1, v1, t1, tok1, lens1) = out[0], out[1]
    assert mx0 == mx1 == 2.0                       # every rank sees the slowest rank's time
    assert v0 == v1 == pytest.approx((t0 + t1) * 10 / 2.0)   # all ranks' tokens / slowest time
    assert tok0 != tok1 or lens0 != lens1           # independent prompts per replica
    assert len(lens0) == len(lens1) == 16


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7, 1) == 7.0
    assert bench.whole_job_throughput(1000, 10, 2.0) == 5000.0
