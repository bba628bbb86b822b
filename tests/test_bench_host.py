"""Host-side logic of bench.py: pair counting and the multi-rank aggregation.

The aggregation is exercised with two gloo ranks on the CPU: each rank
reports its own timing, the job time is the maximum over ranks, and the job
throughput counts the work of every rank (weak scaling, no data exchange).
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from block_diffusion_masked_gb300 import inputs


@pytest.mark.parametrize("n,bs", [(64, 4), (1024, 16), (67, 3), (5, 9), (8192, 32)])
def test_pair_count_matches_oracle(n, bs):
    assert bench.visible_pairs_per_sample(n, bs) == oracle.visible_pairs(n, bs)


def test_flops_convention():
    w = inputs.WORKLOADS["small"]
    f, b = bench.flops(w)
    assert f == 4.0 * bench.visible_pairs_per_sample(w.n, w.block_size) * w.batch * w.heads * w.headdim
    assert b == 2.5 * f
    cf, _ = bench.causal_flops(w)
    assert cf == 4.0 * (2 * w.batch * w.n * (w.n + 1) // 2) * w.heads * w.headdim


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank])
        out[rank] = got
        out[world + rank] = bench.job_tflops(1e12, got[0], world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == [11.0, 5.0] and out[1] == [11.0, 5.0]
    # 2 ranks x 1 TFLOP each in 11 ms
    assert abs(out[2] - 2 * 1e12 / 11e-3 / 1e12) < 1e-9


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_tflops(2e12, 1000.0, 1) == 2.0
