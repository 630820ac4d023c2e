"""The multi-rank parts of the benchmark on CPU: gloo ranks, world size 2 (one process per rank,
as torchrun starts them on a node)."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        w, r, _ = b.dist_env()
        assert (w, r) == (world, rank)
        # every rank learns the slowest rank's time
        got = b.slowest_over_ranks(1.0 + rank, torch.device("cpu"), w)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_slowest_over_ranks_gloo_world2():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        assert dict(out) == {0: 2.0, 1: 2.0}


def test_single_rank_is_its_own_time():
    assert _bench().slowest_over_ranks(3.5, torch.device("cpu"), 1) == 3.5


def test_reference_arm_runs_only_on_rank_zero(monkeypatch, capsys):
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, steps, warmup = "tiny", 1, 0

    b.run_reference(Args())  # returns at once: no work and no line on a non-zero rank
    assert capsys.readouterr().out == ""
