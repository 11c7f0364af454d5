"""The benchmark's multi-rank host logic on CPU: two gloo ranks.

With --gpus N each rank clips its own replica (no data-path collective); the
job's throughput is the units all ranks processed over the slowest rank's
time.  This runs that aggregation with world size 2 on the CPU.
"""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.rank_env()
        elapsed = [10.0, 14.0][rank]                  # rank 1 is the slowest
        value, t = bench.aggregate(elapsed, 1e9, w, bench.make_reduce_max(w, "cpu"))
        q.put((r, w, lr, value, t))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, value, t) in enumerate(out):
        assert (rank, world, local) == (r, 2, r)
        assert t == 14.0                              # max over ranks
        assert value == pytest.approx(2 * 1e9 / 14e-3)


def test_single_rank_needs_no_group():
    value, t = bench.aggregate(5.0, 1e9, 1, bench.make_reduce_max(1, "cpu"))
    assert t == 5.0 and value == pytest.approx(1e9 / 5e-3)


def test_reference_arm_on_a_non_zero_rank_exits_quietly(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_clock_summary_flags_throttling():
    text = ("0, 1400, 2070, 1300.0, 0x0, Not Active, Active, Not Active, Not Active\n"
            "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active\n")
    c = bench.summarize_clocks(text)
    assert c["samples"] == 2 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_algorithmic_bytes():
    assert bench.algorithmic_bytes(92_248_320, 4, "write") == 1_106_979_840
    assert bench.algorithmic_bytes(92_248_320, 2, "write") == 553_489_920
    assert bench.algorithmic_bytes(14_264_448, 4, "read") == 57_057_792
