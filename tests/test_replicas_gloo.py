"""The multi-GPU path is replicas only: every rank runs its own batch, the
job's time is the slowest rank's, the job's units are all ranks' units.  Its
host logic, with two gloo ranks on the CPU (no GPU)."""

import os
import socket
import sys
from pathlib import Path

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402
from long_context_sparse_25_b300 import synth  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local = [3.5, 7.25][rank]  # this rank's measured time
        out[rank] = bench.max_over_ranks(local, dist, torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_time_is_the_slowest_rank_over_two_gloo_ranks():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 7.25, 1: 7.25}


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(2.5, None, torch.device("cpu")) == 2.5


def test_job_units_count_every_rank():
    wl = synth.WORKLOADS["csa_decode_1m"]
    assert bench.job_units(wl, 1) == 32
    assert bench.job_units(wl, 8) == 8 * 32
    pf = synth.WORKLOADS["csa_prefill_64k"]
    assert bench.job_units(pf, 2) == 2 * 65536


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    wl = synth.WORKLOADS["csa_decode_1m"]
    args = type("A", (), {"steps": 1, "warmup": 3, "gpus": 2})()
    bench.run_reference(args, wl)  # returns at once: no oracle work, no line
    assert capsys.readouterr().out == ""
