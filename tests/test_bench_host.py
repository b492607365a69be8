"""Host logic of bench.py without a GPU: throughput aggregation over ranks (world size 2, gloo)."""
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


def _worker(rank, world, port, ms_values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = torch.tensor([ms_values[rank]])
    gathered = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(gathered, t)
    value, worst = bench.aggregate([float(v.item()) for v in gathered], 4096)
    out[rank] = (value, worst)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_single():
    v, w = bench.aggregate([2.0], 4096)
    assert w == 2.0 and abs(v - 4096 / 2e-3) < 1e-6


def test_aggregate_takes_slowest_rank_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, [1.5, 2.5], out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        value, worst = out[r]
        assert worst == 2.5
        assert abs(value - 2 * 4096 / 2.5e-3) < 1e-3


def test_flop_counts_match_the_stated_formulas():
    g = bench.mi_synth.GEOMETRIES["block_1024"]
    gemm, attn = bench.flops_of(g)
    assert abs(gemm / 1e9 - 935.4) < 0.5
    assert abs(attn / 1e9 - 209.6) < 0.5


def test_reference_arm_requires_warmup():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])
