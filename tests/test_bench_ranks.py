"""The bench's multi-rank logic on the CPU: two gloo ranks.

Under torchrun every rank runs an independent replica of the step (the rule
has no exchange between sequences or heads), the job's step time is the
slowest rank's, tokens/s counts every rank's tokens, and only rank 0 prints.
The reference arm runs on rank 0 alone."""

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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = bench.max_over_ranks([1.0 + rank, 10.0 * (rank + 1)], torch.device("cpu"))
        out[rank] = (r, w, local, ms[0], ms[1], bench.whole_job_tokens_per_s(w, ms[0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_tokens():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        r, w, local, ms, e2e, value = res[rank]
        assert (r, w, local) == (rank, world, rank)
        assert ms == 2.0 and e2e == 20.0  # every rank sees the slowest rank's times
        assert value == pytest.approx(world * bench.TOKENS_PER_STEP / 2.0e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    class Args:
        warmup, steps = 3, 1

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(Args()) is None  # no work and no line on other ranks


def test_whole_job_tokens_per_s_counts_every_rank():
    one = bench.whole_job_tokens_per_s(1, 0.5)
    assert one == pytest.approx(bench.TOKENS_PER_STEP / 0.5e-3)
    assert bench.whole_job_tokens_per_s(4, 0.5) == pytest.approx(4 * one)
