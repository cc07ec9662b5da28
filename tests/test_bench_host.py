"""Host-side pieces of bench.py: multi-rank aggregation over gloo, per-rank request ids, byte accounting."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench
import synthetic as S


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, units, e2e_ms, e2e_units = bench.reduce_across_ranks(10.0 + rank, 100.0 * (rank + 1), 20.0 - rank, 7.0)
        w = S.workload(4).replace(B=3, steps=2)
        trees, paths = bench.rank_plan_trees(w, rank)
        q.put((rank, ms, units, e2e_ms, e2e_units, [t.tolist() for t in trees[0]]))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    world, port = 2, _free_port()
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, units, e2e_ms, e2e_units, _ in out:
        assert ms == 11.0 and units == 300.0          # max time, summed units
        assert e2e_ms == 20.0 and e2e_units == 14.0
    assert out[0][5] != out[1][5]                     # ranks serve different requests


def test_single_process_passthrough():
    assert bench.reduce_across_ranks(3.0, 5.0, 4.0, 6.0) == (3.0, 5.0, 4.0, 6.0)


def test_algorithmic_bytes_by_hand():
    # 1 request, 1 layer, Hk=Hv=1, d=32, K=4, conv on, bf16 inputs; n=3 nodes, nb=1 boundary, L=2 pending
    w = S.workload(1).replace(B=1, layers=1, Hk=1, Hv=1, dk=32, dv=32, K=4, in_dtype=S.DTYPE_BF16)
    C = 2 * 32 + 32
    tile = 32 * 32 * 4
    expect = tile + tile + 1 * tile                      # state read, committed write, one boundary
    expect += 3 * (C * 2 + 2 * 1 * 2)                    # x, beta, log_g (bf16)
    expect += 3 * 32 * 4                                 # o
    expect += 3 * (32 + 32 + 1 + C) * 4                  # bank k, u, a, x
    expect += 3 * C * 4 * 2 + 2 * C * 4                  # conv window read + write, two pending raw rows
    expect += 2 * (32 + 32 + 1) * 4                      # pending k, u, a
    expect += C * 4 * 4                                  # conv weights
    assert bench.algorithmic_bytes(w, [3], [1], [2]) == expect
