"""Host-side logic of bench.py (not gpu): op counts, clock parsing, and the
multi-rank timing reduction over gloo with two CPU ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_algorithmic_op_counts_match_the_stated_figures():
    # two passes x 256 steps x (2^16 * 3 + 2^(16-K) * (2^K - 1) * 2)
    assert bench.alg_ops_per_tile(2) == 150_994_944      # 151.0 M
    assert bench.alg_ops_per_tile(3) == 159_383_552      # 159.4 M
    assert bench.alg_ops_per_tile(4) == 163_577_856      # 163.6 M


def test_parse_clock_csv():
    text = ("1965, 2070, 900.1 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "2070, 2070, 1001.0 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "2000, 2070, 950.0 W, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            "garbage line\n")
    r = bench.parse_clock_csv(text)
    assert r["sm_mhz"] == 2000 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"] and r["samples"] == 3
    assert bench.parse_clock_csv("") is None


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world, None)
        m = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        q.put((rank, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25
