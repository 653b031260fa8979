"""The multi-process host logic of bench.py on CPU: two gloo ranks on
127.0.0.1 (world size 2). The path runs as independent replicas, one per
GPU; what the ranks share is the timing (the slowest rank's time) and the
rule that the reference arm runs on rank 0 only."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = 1.5 + 2.0 * rank  # rank 1 is the slower one
        got = bench.max_over_ranks(torch, dist, mine, torch.device("cpu"))
        dist.barrier()
        out.put((rank, got, bench.reference_rank_runs(rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(got == 3.5 for _, got, _ in res)          # both ranks see the max
    assert [runs for _, _, runs in res] == [True, False]  # the reference arm: rank 0 only


def test_single_process_passes_values_through():
    assert bench.max_over_ranks(torch, None, 2.25, torch.device("cpu")) == 2.25
