"""The bench's multi-rank host logic on two gloo ranks (CPU, no GPU).

Each rank decodes its own batch (a different seed, same recipe), the timed
span is the maximum over the ranks, and the reported value is the whole job's
tokens per second.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from synth import TINY_QUEST_4K, make_quest_decode_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = bench.rank_workload(TINY_QUEST_4K.scaled(context_min=64, context_max=64), rank)
        x = make_quest_decode_inputs(wl, device="cpu")
        span_ms = [3.0, 7.5][rank]                       # each rank's own timed span
        worst = bench.max_over_ranks(span_ms, world)
        qs = [torch.zeros_like(x.q) for _ in range(world)]
        dist.all_gather(qs, x.q.contiguous())
        out[rank] = (wl.seed, worst, bool(torch.equal(qs[0], qs[1])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    (s0, w0, same0), (s1, w1, same1) = out[0], out[1]
    assert s0 != s1                                      # each replica has its own batch
    assert not same0 and not same1                       # ... and its own inputs
    assert w0 == w1 == 7.5                               # max over ranks, seen by every rank
    assert bench.job_throughput(32, world, 7.5) == pytest.approx(32 * 2 / 7.5e-3)


def test_single_rank_is_the_identity():
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.rank_workload(TINY_QUEST_4K, 0) is TINY_QUEST_4K
