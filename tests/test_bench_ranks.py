"""bench.py's multi-rank path on CPU: two gloo ranks reduce their timings to
the maximum over ranks, and the whole-job value counts every rank's bytes
over the slowest rank's time; the reference arm runs on rank 0 only."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        med = {"gemv_m1": 10.0 + rank, "isq": 5.0 - rank, "other": 1.0}
        ms, m = bench.max_over_ranks(dist, 20.0 + 3 * rank, med, ["gemv_m1", "isq"],
                                     torch.device("cpu"))
        out[rank] = (ms, m["gemv_m1"], m["isq"], m["other"],
                     bench.whole_job_gbps(1e9, world, m["gemv_m1"]))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, gemv, isq, other, gbps = res[rank]
        assert ms == 23.0 and gemv == 11.0 and isq == 5.0  # maxima over both ranks
        assert other == 1.0                                # stages not reduced stay
        assert gbps == pytest.approx(2e9 / 11e-3 / 1e9)    # both ranks' bytes, slowest time


def test_reference_arm_only_on_rank_zero(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    # a non-zero rank returns before touching the oracle or printing anything
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0
