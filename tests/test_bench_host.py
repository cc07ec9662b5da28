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


def test_algorithmic_fma_by_hand():
    # 2 requests, 1 layer, Hv=2, d=4: n=3 with 1 tile update and L=1; n=1 with none and L=0
    w = S.workload(1).replace(B=2, layers=1, Hk=1, Hv=2, dk=4, dv=4)
    per_elem = (2 * 3 + 1 + 1) + (2 * 1 + 0 + 0)
    assert bench.algorithmic_fma(w, [3, 1], [1, 0], [1, 0]) == per_elem * 2 * 4 * 4
    assert abs(bench.fp32_peak_tflops(152, 2070.0) - 80.55) < 0.01


def test_hbm_stashes_counts_spilled_pushes():
    # a perfect binary tree of 15 nodes: the third stash level (light depth two) spills to HBM
    from gated_deltanet_tree_gb300.build import build
    build()
    from gated_deltanet_tree_gb300 import _native as N
    parent = np.array([-1] + [(i - 1) // 2 for i in range(1, 15)], dtype=np.int32)
    n_max = 16
    P = np.full((1, n_max), -1, dtype=np.int32)
    P[0, :len(parent)] = parent
    words, _ = N.gdn_pack_schedules(P, np.array([len(parent)], dtype=np.int32))
    ops = words[0, 5 + 3 * n_max:5 + 3 * n_max + len(parent)]
    spilled = int((((ops >> 12) & 3) == 3).sum())
    assert spilled >= 1 and words[0, 4] == 2
    assert bench.hbm_stashes(words, n_max) == [spilled]
    assert bench.hbm_stashes(N.gdn_pack_schedules_per_node(P, np.array([len(parent)], dtype=np.int32))[0],
                             n_max) == [int((np.bincount(parent[1:], minlength=len(parent)) > 0).sum())]


def test_tensor_core_flops_follow_the_issued_mmas():
    """One head, one layer: the tf32 FLOPs reported are those of the MMAs the persistent kernel issues (one
    N = 4 NB and one N = 2 NB product per K step of 8), and the kernel applies where the dispatch sends
    batches to it."""
    import bench
    w = S.workload(2).replace(Hk=1, Hv=1, layers=1, B=1)
    shapes = bench.tc_mma_shapes(w, 22)
    assert len(shapes) == 2 * 128 // 8
    assert sorted({n for _, n, _ in shapes}) == [48, 96]   # 2 NB, 4 NB for NB = 24
    assert bench.tensor_flops(w, [22]) == 16 * 2 * 128 * 8 * (96 + 48)
    assert bench.tc_applies(w) and not bench.tc_applies(w.replace(n_max=64)) and not bench.tc_applies(w.replace(dv=64))


def test_traffic_record_roundtrip(tmp_path, monkeypatch):
    """The traffic record written from ncu CSV logs scales per (request, layer) block and is dropped as soon
    as one measured kernel's sources differ from those the capture was taken with."""
    import bench
    csv = tmp_path / "t.csv"
    hdr = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",' \
          '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'
    rows = []
    for i, (k, rd, wr) in enumerate([("ut_tcp_verify_kernel<128, bf16, 2>", 900, 700), ("conv_window_kernel<bf16, 4>", 300, 100)]):
        for m, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr)):
            rows.append(f'"{i}","1","p","h","{k}","1","7","(1,1,1)","(1,1,1)","0","10.3","s","{m}","byte","{v:,}"\n')
    csv.write_text("==PROF== noise\n" + hdr + "".join(rows))
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(tmp_path / "rec.txt"))
    bench.record_traffic([str(csv)], blocks=4, command="ncu ...")
    assert bench.measured_traffic(8) == (1600 + 400) / 4 * 8
    src = dict(bench.KERNEL_SOURCES)
    monkeypatch.setattr(bench, "KERNEL_SOURCES", dict(src, conv_window_kernel=["gdn_commit.cu"]))
    assert bench.measured_traffic(8) is None


def test_zero_copy_acceptances():
    import bench
    r = bench.zero_copy_acceptances([[0, 1, 2], [0, 2], [], [0], [0, 1, 3]])
    assert r == {"fraction": 0.6, "paths": 5, "zero_copy": 3, "mean_length": 1.8}
    # the batched workload's cycle: 32 requests x 8 steps, some but not all paths in slot order
    w = bench.S.workload(4)
    r = bench.zero_copy_acceptances([p for step in bench.rank_plan_trees(w, 0)[1] for p in step])
    assert r["paths"] == w.B * w.steps and 0 < r["fraction"] < 1


def test_bench_line_contract_with_a_stand_in_gpu_leg(monkeypatch, capsys):
    # main() assembles the JSON line from the GPU leg's figures; a stand-in for that leg (no device here) checks
    # the line's keys and the arithmetic between them
    w = S.workload(4)
    steps = 3
    fake = dict(ms=15.0, units=3.0e6, verify_ms=[4.8, 4.9, 5.0], finish_ms=1.5, clocks={"sm_mhz": 2070.0},
                ab=None, walk=None, simt=None, tc1=None, bout=None, avg_tflops=5.0e11, achieved=3000.0,
                peak=6781.8, peak_kind="measured", avg_bytes=1.44e10, e2e_ms=16.0, avg_flops=8.0e9,
                alu_peak=80.5, avg_verify_s=4.9e-3, e2e_units=3.0e6,
                e2e=dict(ms=16.0, units=3.0e6, steps=steps, h2d=100, d2h=200, step_ms_median=5.3,
                         step_ms_max=6.0, stalled_steps=0),
                nb_cap=0, walked=False, gpu_launches=3 * steps)
    monkeypatch.setattr(bench, "run_gpu", lambda args, w_, rank, world: fake)
    monkeypatch.setattr("sys.argv", ["bench.py", "--no-cpu-baseline", "--no-per-config", "--steps", str(steps),
                                     "--warmup", "3"])
    bench.main()
    line = __import__("json").loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["metric"] == bench.METRIC and line["unit"] == "nodes/s" and line["n_gpus"] == 1
    assert line["value"] == pytest.approx(3.0e6 / 15.0e-3)
    assert line["ms_per_step"] == pytest.approx(5.0)
    r = line["roofline"]
    assert r["frac"] == pytest.approx(3000.0 / 6781.8) and r["bound"] in ("hbm", "alu")
    assert r["avg_launch_ms"] == pytest.approx(4.9) and r["median_launch_ms"] == pytest.approx(4.9)
    assert line["e2e"]["value"] == pytest.approx(3.0e6 / 16.0e-3)
    assert line["e2e"]["h2d_bytes_per_step"] == 100 and line["e2e"]["d2h_bytes_per_step"] == 200
    assert line["gpu_launches"] == 9 and line["clocks"] == {"sm_mhz": 2070.0}
    assert line["config"]["requests_per_gpu"] == w.B and line["config"]["gdn_layers"] == w.layers
    assert line["zero_copy_acceptances"]["paths"] == w.B * w.steps
