"""The benchmark's multi-process plumbing on CPU (gloo, world size 2): the
timed region's elapsed time is the slowest rank's on every rank, and the
reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], world, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    values = [3.25, 7.5]
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), values, out), nprocs=world, join=True)
    assert dict(out) == {0: 7.5, 1: 7.5}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    class A:
        workload = "decode_27b"
        steps = 1
        warmup = 3
        gpus = 2
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
