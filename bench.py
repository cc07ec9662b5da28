"""Throughput of GDN tree verification with fused commit on one or more GPUs.

A step is one pass of the whole path over one batch: heavy-light schedules of
every request's tree on the host and their upload, the verify call (pending
commit folded into the conv window and the state tiles, every node solved in
the tree-masked UT form, o and factors written; boundary states as scratch)
and the commit of each request's accepted path.  The chain walk and the
per-node-state baseline run afterwards on the same inputs as A/B legs.  Default workload: 32 requests x 48 GDN layers of 48 v-heads
(d_k = d_v = 128, conv K = 4, bf16 inputs), a fresh 22-node top-4 DDTree per
request and step, alternating factor banks.  The metric is verified tree nodes
per second, one unit being one (request, GDN layer, v-head, node).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own batch of requests (weak scaling, no
collective on the data path); timing is the max over ranks.  --impl reference
times the CPU oracle on the host cores instead (a bounded sample).
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as S  # noqa: E402

METRIC = "verified tree-nodes/sec (GDN layer·head·node) and achieved HBM GB/s vs GB300 peak"
UNIT = "nodes/s"
UT_MAX_DEPTH = 24   # GDN_UT_MAX_DEPTH: deeper batches are verified by walking chains


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "traffic_gdn_tree_verify_batched32x48.txt")
# the files each measured kernel is built from: a record stays valid while their hashes do
KERNEL_SOURCES = {
    "ut_tcp_verify_kernel": ["gdn_verify_tcp.cu", "gdn_tile.cuh", "gdn_umma.cuh", "gdn_internal.h"],
    "conv_window_kernel": ["gdn_conv.cu", "gdn_internal.h"],
}


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "gated_deltanet_tree_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(units: int):
    """DRAM bytes of one verify call over `units` (request, layer) blocks, from the committed small-case
    capture of each kernel (bytes per block, scaled), or None once a kernel's sources changed since."""
    try:
        total = 0.0
        seen = set()
        for line in open(TRAFFIC_RECORD):
            parts = line.split()
            if not parts or parts[0] != "kernel":
                continue
            f = dict(zip(parts[2::2], parts[3::2]))
            name = parts[1]
            if f.get("sources_sha256") != kernel_source_hash(name):
                return None
            total += float(f["bytes_per_block"]) * units
            seen.add(name)
        return total if seen == set(KERNEL_SOURCES) else None
    except Exception:
        return None


def record_traffic(csv_paths, blocks: int, command: str):
    """Writes the traffic record from ncu CSV logs (dram__bytes_read.sum and dram__bytes_write.sum of the
    captured launches of each kernel) of a capture over `blocks` (request, layer) blocks."""
    import csv
    import subprocess as sp
    per = {}
    for path in csv_paths:
        with open(path) as fh:
            rows = [r for r in csv.reader(l for l in fh if l.startswith('"'))]
        hdr = rows[0]
        ki, mi, vi, ii = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value"), hdr.index("ID")
        for r in rows[1:]:
            name = next((k for k in KERNEL_SOURCES if k in r[ki]), None)
            if name is None or r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                continue
            per.setdefault(name, {}).setdefault(r[ii], {})[r[mi]] = float(r[vi].replace(",", ""))
    commit = sp.run(["git", "-C", ROOT, "rev-parse", "--short=12", "HEAD"], capture_output=True, text=True).stdout.strip()
    lines = ["# DRAM traffic of one gdn_tree_verify call per (request, layer) block, by kernel, from a capture over",
             f"# {blocks} blocks (a small case whose state is larger than L2), scaled by bench.py to the call's blocks",
             "# (traffic grows with the blocks: state, node rows and factors are per block; the conv weights, per",
             "# layer, are the only exception, under 0.1% of a call).  Captured at commit " + (commit or "?") + ".",
             "# Command (after the same bench command without ncu exited 0; one kernel per ncu call):",
             f"#   {command}",
             "# A kernel's line counts only while sources_sha256 equals the sha256 of its files (bench.py,",
             "# KERNEL_SOURCES); otherwise roofline.traffic is reported as null."]
    for name in KERNEL_SOURCES:
        launches = list(per.get(name, {}).values())
        if not launches:
            raise SystemExit(f"no launches of {name} in {csv_paths}")
        rd = statistics.mean(l["dram__bytes_read.sum"] for l in launches)
        wr = statistics.mean(l["dram__bytes_write.sum"] for l in launches)
        lines.append(f"kernel {name} sources_sha256 {kernel_source_hash(name)} bytes_per_block {(rd + wr) / blocks:.1f} "
                     f"read_per_launch {rd:.0f} write_per_launch {wr:.0f} launches {len(launches)}")
    with open(TRAFFIC_RECORD, "w") as fh:
        fh.write("\n".join(lines) + "\n")
    print("\n".join(lines))


def tf32_peak() -> float:
    """Dense tf32 tensor peak (TFLOP/s): the measured bf16 burst GEMM rate times the nominal tf32 : bf16
    ratio (1.1 : 2.25 PFLOP/s dense, taken as 1/2); the nominal 1.1 PFLOP/s if nothing was measured."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]) / 2
    except Exception:
        return 1100.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------
# algorithmic bytes of one verify call (compulsory traffic: every input read
# once, every output written once)
# ----------------------------------------------------------------------------

def hbm_stashes(words: np.ndarray, n_max: int):
    """Per request: the stashes a packed schedule writes to HBM (ops with the boundary-slot push bit);
    with boundary states as scratch, the others stay in tensor memory."""
    ops = words[:, 5 + 3 * n_max:5 + 4 * n_max]
    n = words[:, 0]
    return [int(((ops[b, :n[b]] >> 12) & 3 == 3).sum()) for b in range(words.shape[0])]


def algorithmic_bytes(w: S.Workload, n_per_req, nb_per_req, pend_len_per_req):
    """Compulsory bytes of one gdn_tree_verify call (conv window + chain verify); nb_per_req = the
    state tiles each request writes beside its committed state (stored boundary states or HBM stashes)."""
    ib = 2 if w.in_dtype == S.DTYPE_BF16 else 4
    tile = w.dk * w.dv * 4 * w.Hv                    # all v-heads of one (request, layer)
    C = w.C
    total = 0
    for n, nb, L in zip(n_per_req, nb_per_req, pend_len_per_req):
        per_bl = tile                                 # state read
        per_bl += tile if L > 0 else 0                # committed state written once
        per_bl += nb * tile                           # boundary states written
        per_bl += n * (C * ib + 2 * w.Hv * ib)        # x, beta, log_g read
        per_bl += n * w.Hv * w.dv * 4                 # o written
        per_bl += n * (w.Hk * w.dk + w.Hv * w.dv + w.Hv + (C if w.conv_mode else 0)) * 4   # factor bank written
        if w.conv_mode and w.K > 1:
            per_bl += (w.K - 1) * C * 4 * (2 if L > 0 else 1)   # conv window read (+ written when folded)
            per_bl += min(L, w.K - 1) * C * 4                    # pending raw rows read
        per_bl += L * (w.Hk * w.dk + w.Hv * w.dv + w.Hv) * 4     # pending factors read
        total += per_bl * w.layers
    if w.conv_mode:
        total += w.layers * C * w.K * 4               # conv weights
    return total


def tree_depth(parent) -> int:
    depth = [0] * len(parent)
    for i in range(1, len(parent)):
        depth[i] = depth[parent[i]] + 1
    return max(depth)


def algorithmic_fma(w: S.Workload, n_per_req, updates_per_req, pend_len_per_req):
    """FP32 multiply-adds of one verify call on the state tiles: per node T^T k and T^T q (2 per element),
    1 per element for every node whose update is applied to a tile (none in the tree-masked UT form; the
    non-leaf nodes when walking chains), 1 per element per folded node.  The per-node vector work (the
    ancestor-pair solve, normalisation, conv) is a few thousand operations per head and is left out."""
    per_elem = sum(2 * n + up + L for n, up, L in zip(n_per_req, updates_per_req, pend_len_per_req))
    return per_elem * w.layers * w.Hv * w.dk * w.dv


TC_MAX_NODES = 32   # the tensor-core UT kernels take d_v = 128 and n_max <= 32 (gdn_tree_verify's dispatch)
TC_WIDE_NODES, TC_WIDE_DEPTH = 64, 16   # ... and n_max <= 64 when no tree is deeper than 16


def tc_applies(w: S.Workload, depth_max: int = 0) -> bool:
    """Whether gdn_tree_verify's default dispatch solves the batch on the tensor cores (depth_max: the packers'
    deepest node of the batch, 0 when unknown)."""
    if not (w.dv == 128 and w.dk in (32, 64, 128)):
        return False
    return w.n_max <= TC_MAX_NODES or (w.n_max <= TC_WIDE_NODES and 1 <= depth_max <= TC_WIDE_DEPTH)


def tc_mma_shapes(w: S.Workload, n: int):
    """(M, N, K) of every tcgen05 MMA the persistent tensor-core kernel issues for one head and a tree of n
    nodes (NB = n rounded up to 8; K = 8 per instruction, d_k / 8 instructions each): T0^T_hi times all
    4 NB operand rows (high and low k, q), then T0^T_lo times the 2 NB high rows.  (Its Gram coefficients
    are formed on the CUDA cores, once per k-head.)"""
    nb = (n + 7) // 8 * 8
    per_step = [(w.dv, 4 * nb, 8), (w.dv, 2 * nb, 8)]
    return per_step * (w.dk // 8)


CHAIN_SEG = 16   # GDN_VERIFY_CHAINS: nodes per segment


def chain_tensor_flops(w: S.Workload, n_per_req):
    """tf32 FLOPs of the chain-segment MMAs in one call: per segment of m nodes, the tree kernel's two
    products for a tree of m nodes."""
    per_head = 0
    for n in n_per_req:
        for s0 in range(0, n, CHAIN_SEG):
            per_head += sum(2 * m * nn * k for m, nn, k in tc_mma_shapes(w, min(CHAIN_SEG, n - s0)))
    return per_head * w.layers * w.Hv


def tensor_flops(w: S.Workload, n_per_req):
    """tf32 FLOPs the tensor cores execute in one verify call (2 M N K per MMA)."""
    per_head = sum(sum(2 * m * nn * k for m, nn, k in tc_mma_shapes(w, n)) for n in n_per_req)
    return per_head * w.layers * w.Hv


def fp32_peak_tflops(sm_count: int, sm_mhz: float) -> float:
    """Dense FP32 FMA peak: 128 FP32 lanes per SM, 2 flops per FMA."""
    return sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"gdn_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# oracle baseline (CPU)
# ----------------------------------------------------------------------------

def _oracle_unit(args):
    """Oracle verify of one (request, layer) block at one step: every node's root path replayed from the
    block's initial state (the cost does not depend on the state's values, so no commit history is replayed)."""
    cfg_kw, b, l, step = args
    sys.path.insert(0, ROOT)
    import synthetic as S2
    from oracle import gdn_oracle as O
    w = S2.Workload(**cfg_kw)
    parent = S2.tree_for(w, b, step)
    n = len(parent)
    x, be, ag = S2.node_inputs(w, b, l, step)
    d = O.dims_of(w)
    T = S2.init_state(w, b, l).astype(np.float64)
    W = S2.init_conv_state(w, b, l).astype(np.float64)
    cw = S2.conv_weight(w, l).astype(np.float64) if w.conv_mode else None
    t0 = time.perf_counter()
    O.verify_tree(T, W, parent, O.as_f64(x[:n], w.in_dtype), O.as_f64(be[:n], w.in_dtype),
                  O.as_f64(ag[:n], w.in_dtype), cw, d)
    return n * w.Hv, time.perf_counter() - t0


def _warm_worker(_):
    sys.path.insert(0, ROOT)
    import synthetic  # noqa: F401
    from oracle import gdn_oracle  # noqa: F401
    return 0


def oracle_throughput(w: S.Workload, target_s: float = 15.0, cores=None, warmup: int = 0, steps: int = 0,
                      full: bool = False, all_steps: bool = False):
    """The oracle (one full root-path replay per node, fp64) on `cores` host processes (spawn pool, one BLAS
    thread each), on (request, layer) blocks of the workload.

    full: every block of step 0, once (the whole call).  Otherwise a seeded sample drawn from every block of
    step 0 (or, with all_steps, of every step of the cycle): `warmup` untimed and `steps` timed rounds of
    one block per process, or as many rounds as fit in about `target_s` seconds.
    """
    import dataclasses
    cores = cores or os.cpu_count() or 1
    kw = dataclasses.asdict(w)
    nsteps = w.steps if all_steps else 1
    units = [(kw, b, l, s) for s in range(nsteps) for l in range(w.layers) for b in range(w.B)]
    order = np.random.default_rng(0).permutation(len(units)) if not full else np.arange(len(units))
    os.environ["OPENBLAS_NUM_THREADS"] = "1"   # inherited by the spawned workers
    os.environ["OMP_NUM_THREADS"] = "1"
    ctx = mp.get_context("spawn")
    done_units, blocks, pos, timed_steps = 0, 0, 0, 0

    def next_batch():
        nonlocal pos
        take = min(cores, len(units) - pos) if full else cores
        batch = [units[order[(pos + i) % len(units)]] for i in range(take)]
        pos += take
        return batch

    with ctx.Pool(cores) as pool:
        pool.map(_warm_worker, range(cores))      # spawn and imports are not timed
        for _ in range(warmup):
            pool.map(_oracle_unit, next_batch())
        if full:
            pos = 0
        t0 = time.perf_counter()
        while True:
            batch = next_batch()
            for u, _ in pool.map(_oracle_unit, batch):
                done_units += u
                blocks += 1
            timed_steps += 1
            if full and pos >= len(units):
                break
            if not full and steps > 0 and timed_steps >= steps:
                break
            if not full and steps <= 0 and time.perf_counter() - t0 >= target_s:
                break
    dt = time.perf_counter() - t0
    total = w.B * w.layers * nsteps
    what = (f"one whole verify call ({total} (request, layer) block{'s' if total > 1 else ''})" if full else
            f"{blocks} of {total} (request, layer) blocks ({100.0 * blocks / total:.2f}%, seeded sample"
            + (f" over all {nsteps} steps of the cycle" if all_steps else " of step 0") + ")")
    return {"value": done_units / dt, "unit": UNIT, "cores": cores, "kind": "oracle", "steps": timed_steps,
            "ms_per_step": dt * 1e3 / timed_steps, "seconds": dt,
            "sample": f"{what}, all {w.Hv} v-heads and every node, {dt:.2f} s wall on {cores} host "
                      f"process{'es' if cores > 1 else ''} (spawn pool, one BLAS thread each)"}


def cpu_baselines(w: S.Workload, seconds: float):
    """The oracle on 1 thread and on all host cores: configs 1-3 in full (one verify call each), a sample of
    the headline workload across its whole cycle, and on all cores a sample of each stress configuration
    (64-node top-8 trees, 64-node chains) across its cycle.  Run before the first GPU call of the process."""
    ncores = os.cpu_count() or 1
    main_all = oracle_throughput(w, target_s=seconds, cores=ncores, all_steps=True)
    main_one = oracle_throughput(w, target_s=seconds * 0.6, cores=1, all_steps=True)
    per = {}
    for cfg in (1, 2, 3):
        wc = S.workload(cfg)
        one = oracle_throughput(wc, cores=1, full=True)
        allc = oracle_throughput(wc, cores=ncores, full=True)
        per[str(cfg)] = {"workload": wc.name, "one_thread": {k: one[k] for k in ("value", "seconds", "sample")},
                         "all_cores": {k: allc[k] for k in ("value", "seconds", "sample", "cores")}}
    for cfg, key in ((5, "5(i)"), (6, "5(ii)")):   # the stress configs: a seeded sample across their cycle
        wc = S.workload(cfg)
        allc = oracle_throughput(wc, target_s=seconds / 3, cores=ncores, all_steps=True)
        per[key] = {"workload": wc.name, "all_cores": {k: allc[k] for k in ("value", "seconds", "sample", "cores")}}
    out = dict(main_all)
    out["nproc"] = ncores
    out["one_thread"] = {k: main_one[k] for k in ("value", "seconds", "sample", "cores")}
    out["per_config"] = per
    return out


def reduce_across_ranks(ms: float, units: float, e2e_ms: float, e2e_units: float, device=None):
    """Whole-job figures: the slowest rank's time, the units of all ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, units, e2e_ms, e2e_units
    t = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([units, e2e_units], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t[0]), float(u[0]), float(t[1]), float(u[1])


def zero_copy_acceptances(paths) -> dict:
    """Accepted paths already in bank-slot order (path[i] == i for every i, the empty path included): the
    acceptances that a fold reading the bank in path order takes without a compaction copy.  This library's
    fold gathers the pending rows by node index, so no acceptance needs the copy; the fraction says how often
    one would without that."""
    paths = [list(p) for p in paths]
    zc = sum(all(int(v) == i for i, v in enumerate(p)) for p in paths)
    return {"fraction": zc / len(paths) if paths else None, "paths": len(paths), "zero_copy": zc,
            "mean_length": sum(len(p) for p in paths) / len(paths) if paths else None}


def rank_plan_trees(w: S.Workload, rank: int):
    """Every rank serves its own requests: request ids are offset by rank * B."""
    trees = [[S.tree_for(w, b + rank * w.B, s) for b in range(w.B)] for s in range(w.steps)]
    paths = [[S.path_for(w, trees[s][b], b + rank * w.B, s) for b in range(w.B)] for s in range(w.steps)]
    return trees, paths


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args, w: S.Workload, rank: int, world: int):
    import torch
    import torch.distributed as dist
    from gated_deltanet_tree_gb300 import _native as N
    from harness import GpuSession, WorkloadPlan
    from gated_deltanet_tree_gb300.runtime import paths_tensor

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    # every rank serves its own requests: request ids are offset by rank
    trees, paths_h = rank_plan_trees(w, rank)
    plan = WorkloadPlan(w, trees=trees, paths=paths_h)
    gs = GpuSession(w, plan, device=dev, preload_steps=range(w.steps))
    stream = torch.cuda.current_stream(dev)
    ver = gs.ver

    # pinned host buffers for each step's packed schedule words (filled by the host HLD inside the timed loop)
    words_dev = [torch.empty(w.B, N.gdn_schedule_words(w.n_max), dtype=torch.int32, device=dev)
                 for _ in range(w.steps)]
    words_host = [torch.empty(w.B, N.gdn_schedule_words(w.n_max), dtype=torch.int32).pin_memory()
                  for _ in range(w.steps)]
    parents_host = []
    for s in range(w.steps):
        P = np.full((w.B, w.n_max), -1, dtype=np.int32)
        n = np.zeros(w.B, dtype=np.int32)
        for b, p in enumerate(plan.trees[s]):
            P[b, :len(p)] = p
            n[b] = len(p)
        parents_host.append((P, n))
    paths = [gs.paths(s) for s in range(w.steps)]

    depth_of = [0] * w.steps   # the deepest node of each step's trees (it selects the verify kernel)

    def sched_struct(s):
        return N.gdn_batch_schedule(B=w.B, n_max=w.n_max, nb_max=gs.nb_cap, depth_max=depth_of[s],
                                    words=words_dev[s].data_ptr())

    def one_step(i, timing=None):
        s = i % w.steps
        P, n = parents_host[s]
        words, _, depth_of[s] = N.gdn_pack_schedules(P, n, with_depth=True)   # host heavy-light schedules
        words_host[s].numpy()[...] = words
        words_dev[s].copy_(words_host[s], non_blocking=True)
        X, BE, AG = gs.inputs[s]
        sc = sched_struct(s)
        if timing is not None:
            timing[0].record(stream)
        N.gdn_tree_verify(gs.dims, w.layers, sc, X, gs.conv_w, BE, AG, gs.state, gs.conv_state, gs.out_o,
                          gs.boundary, ver.banks, ver.workspace, ver.ws_bytes, N.GDN_VERIFY_BOUNDARY_SCRATCH, stream)
        if timing is not None:
            timing[1].record(stream)
        N.gdn_commit_fold(gs.dims, w.layers, sc, paths[s][0], paths[s][1], 0, ver.banks, stream)

    def barrier():
        if world > 1:
            dist.barrier()

    # bytes / units of each step (pending length of step s = accepted path length of step s-1)
    units_per_step, bytes_per_step, fma_per_step, tflops_per_step, walks = [], [], [], [], []
    for i in range(args.warmup + args.steps):
        s = i % w.steps
        n_req = [len(p) for p in plan.trees[s]]
        P, n = parents_host[s]
        nb_req = [0] * w.B   # the tree-masked UT form writes no state but the committed one
        prev = plan.paths[(i - 1) % w.steps] if i > 0 else [[] for _ in range(w.B)]
        L_req = [len(p) for p in prev]
        units_per_step.append(sum(n_req) * w.layers * w.Hv)
        bytes_per_step.append(algorithmic_bytes(w, n_req, nb_req, L_req))
        walk = max(tree_depth(p) for p in plan.trees[s]) > UT_MAX_DEPTH   # deep trees walk chains
        walks.append(walk)
        if walk:   # the chain walk updates the tile at every node with children
            ups = [int((np.bincount(p[1:], minlength=len(p)) > 0).sum()) if len(p) > 1 else 0 for p in plan.trees[s]]
        else:      # the tree-masked UT form applies no per-node update to the tile
            ups = [0] * w.B
        if not walk and tc_applies(w):   # T0^T k and T0^T q on the tensor cores: the fold stays on FP32
            fma_per_step.append(algorithmic_fma(w, [0] * w.B, ups, L_req))
            tflops_per_step.append(tensor_flops(w, n_req))
        else:
            fma_per_step.append(algorithmic_fma(w, n_req, ups, L_req))
            tflops_per_step.append(0)

    for i in range(args.warmup):
        one_step(i)
    torch.cuda.synchronize(dev)
    ver.check_error()

    clocks = ClockSampler(dev.index)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start.record(stream)
    for k in range(args.steps):
        one_step(args.warmup + k, ev[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    ver.check_error()
    ms = t_start.elapsed_time(t_end)
    verify_ms = [a.elapsed_time(b) for a, b in ev]

    timed_units = sum(units_per_step[args.warmup:])
    timed_bytes = bytes_per_step[args.warmup:]

    # finish (materialise the last pending path) timed on its own
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    ver.finish(gs.state, gs.conv_state, stream)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    finish_ms = f0.elapsed_time(f1)

    # end to end through the public API with host buffers: inputs H2D from pinned memory, outputs D2H
    # A/B: the same steps with per-node-state schedules (every node reloads its parent's stored state)
    ab = walk = simt = tc1 = bout = None
    if not args.no_ab:
        bout = run_walk_ab(args, w, gs, dev, stream, paths, parents_host, mode="boundary_out")
        if tc_applies(w) and not any(walks[args.warmup:]):
            tc1 = run_walk_ab(args, w, gs, dev, stream, paths, parents_host, mode="tc_per_head")
            simt = run_walk_ab(args, w, gs, dev, stream, paths, parents_host, mode="ut_simt")
        walk = run_walk_ab(args, w, gs, dev, stream, paths, parents_host, mode="walk")
        ab = run_walk_ab(args, w, gs, dev, stream, paths, parents_host, mode="per_node")

    if args.no_e2e:
        e2e = dict(ms=float("nan"), units=0, steps=0, h2d=0, d2h=0)
    else:
        e2e = run_e2e(args, w, gs, dev, stream, paths, parents_host, words_host, words_dev, sched_struct,
                      units_per_step, rank)

    ms, timed_units_all, e2e_ms, e2e_units_all = reduce_across_ranks(ms, timed_units, e2e["ms"], e2e["units"], dev)

    peak, peak_kind = peaks()
    avg_verify_s = statistics.mean(verify_ms) / 1e3
    avg_bytes = statistics.mean(timed_bytes)
    achieved = avg_bytes / avg_verify_s / 1e9
    avg_flops = 2 * statistics.mean(fma_per_step[args.warmup:])
    avg_tflops = statistics.mean(tflops_per_step[args.warmup:])
    alu_peak = fp32_peak_tflops(torch.cuda.get_device_properties(dev).multi_processor_count,
                                (clk or {}).get("sm_max_mhz") or 2070.0)
    return dict(ms=ms, units=timed_units_all, verify_ms=verify_ms, finish_ms=finish_ms, clocks=clk, ab=ab, walk=walk,
                simt=simt, tc1=tc1, bout=bout, avg_tflops=avg_tflops,
                achieved=achieved, peak=peak, peak_kind=peak_kind, avg_bytes=avg_bytes, e2e_ms=e2e_ms,
                avg_flops=avg_flops, alu_peak=alu_peak, avg_verify_s=avg_verify_s,
                e2e_units=e2e_units_all, e2e=e2e, nb_cap=gs.nb_cap, walked=any(walks[args.warmup:]),
                gpu_launches=args.steps * 3)


def run_walk_ab(args, w, gs, dev, stream, paths, parents_host, mode):
    """The same workload verified another way: "walk" walks the heavy-light chains (branch states in
    tensor memory); "per_node" walks the per-node-state baseline, whose schedule has no heavy edges so
    every node with children is stored to and reloaded from HBM (the snapshot-style traffic the
    heavy-light chains avoid); "ut_simt" solves the tree-masked UT form on the CUDA cores."""
    import torch
    from gated_deltanet_tree_gb300 import _native as N
    per_node = mode == "per_node"
    steps = max(2, min(args.steps, 10))
    packed, nb_cap, depth = [], 1, []
    for s in range(w.steps):
        P, n = parents_host[s]
        words, nb, dm = (N.gdn_pack_schedules_per_node if per_node else N.gdn_pack_schedules)(P, n, with_depth=True)
        packed.append(torch.from_numpy(words).to(dev))
        nb_cap = max(nb_cap, nb)
        depth.append(dm)
    if mode == "boundary_out":   # the default kernel, every boundary state stored (the ABI's default)
        flags = 0
    else:
        flags = N.GDN_VERIFY_BOUNDARY_SCRATCH | {"ut_simt": N.GDN_VERIFY_UT_SIMT,
                                                 "tc_per_head": N.GDN_VERIFY_TC_PER_HEAD}.get(mode, N.GDN_VERIFY_CHAIN_WALK)
    boundary = torch.empty(w.B, w.layers, nb_cap, w.Hv, w.dk, w.dv, dtype=torch.float32, device=dev)
    ver = gs.ver

    def one(i):
        s = i % w.steps
        sc = N.gdn_batch_schedule(B=w.B, n_max=w.n_max, nb_max=nb_cap, depth_max=depth[s], words=packed[s].data_ptr())
        X, BE, AG = gs.inputs[s]
        N.gdn_tree_verify(gs.dims, w.layers, sc, X, gs.conv_w, BE, AG, gs.state, gs.conv_state, gs.out_o,
                          boundary, ver.banks, ver.workspace, ver.ws_bytes, flags, stream)
        N.gdn_commit_fold(gs.dims, w.layers, sc, paths[s][0], paths[s][1], 0, ver.banks, stream)

    for i in range(3):
        one(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    units = 0
    for i in range(3, 3 + steps):
        one(i)
        units += int(parents_host[i % w.steps][1].sum()) * w.layers * w.Hv
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ver.check_error()
    ms = e0.elapsed_time(e1)
    del boundary
    torch.cuda.empty_cache()
    return {"schedule": {"per_node": "per-node states in HBM (no heavy edges)",
                         "walk": "heavy-light chain walk, branch states in tensor memory",
                         "ut_simt": "tree-masked UT form on the CUDA cores (ut_verify_kernel)",
                         "tc_per_head": "tree-masked UT form on the tensor cores, a CTA per v-head (ut_tc_verify_kernel)",
                         "boundary_out": "default kernel with every boundary state stored to HBM (flags 0)"}[mode],
            "steps": steps, "nb_max": nb_cap,
            "ms_per_step": ms / steps, "value": units / (ms / 1e3), "unit": UNIT}


def run_e2e(args, w, gs, dev, stream, paths, parents_host, words_host, words_dev, sched_struct, units_per_step,
            rank=0):
    """Same calls with host buffers: each step builds its trees from the draft's log-probabilities (the
    DDTree builder, for DDTree workloads), packs their schedules, copies its inputs from pinned host memory
    and reads its outputs back.  Copies run on their own streams, double-buffered, so step k+1's upload
    and step k-1's download overlap step k's compute; after W untimed steps through the same loop, the timed
    span runs from the first upload to the last download of K steps."""
    import torch
    from gated_deltanet_tree_gb300 import _native as N
    steps = max(1, args.steps)   # as many steps as the device-timed leg: the pipeline's fill and drain amortise
    warm = max(3, getattr(args, "warmup", 3))   # untimed first: the first transfers through fresh buffers are slow
    nsrc = min(2, w.steps)
    drafts = None
    if w.tree == "ddtree":   # draft tables of the requests served (the trees are rebuilt from them each step)
        drafts = [np.stack([S.draft_logp(w, b + rank * w.B, s) for b in range(w.B)]) for s in range(nsrc)]
    host_in = []
    for s in range(nsrc):
        X, BE, AG = gs.inputs[s]
        host_in.append(tuple(t.cpu().pin_memory() for t in (X, BE, AG)))
    dev_in = [tuple(torch.empty_like(t) for t in gs.inputs[0]) for _ in range(2)]
    out = [gs.out_o, torch.empty_like(gs.out_o)]
    o_host = [torch.empty(gs.out_o.shape, dtype=gs.out_o.dtype).pin_memory() for _ in range(2)]
    nwh = max(steps, warm)
    wh = [torch.empty_like(words_host[0]).pin_memory() for _ in range(nwh)]
    wd = [torch.empty_like(words_dev[0]) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0]) + wh[0].numel() * 4
    d2h = o_host[0].numel() * o_host[0].element_size()
    ver = gs.ver
    # three streams of their own: the default stream would serialise with the copy streams
    stream = torch.cuda.Stream(dev)
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def run(nsteps):
        h2d_done = [ev() for _ in range(nsteps)]
        cmp_done = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps)]   # (also the step clock)
        d2h_done = [ev() for _ in range(nsteps)]
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        units = 0
        e0.record(s_h2d)
        for k in range(nsteps):
            i, s = k % 2, k % nsrc
            if drafts is not None:
                P, n = N.gdn_ddtree_build_batch(drafts[s], w.budget, w.n_max)   # host DDTree construction
            else:
                P, n = parents_host[s]
            words, _, depth = N.gdn_pack_schedules(P, n, with_depth=True)   # host heavy-light schedules
            wh[k].numpy()[...] = words
            with torch.cuda.stream(s_h2d):
                if k >= 2:
                    s_h2d.wait_event(cmp_done[k - 2])        # buffers i no longer read by compute
                wd[i].copy_(wh[k], non_blocking=True)
                for dst, src in zip(dev_in[i], host_in[s]):
                    dst.copy_(src, non_blocking=True)
                h2d_done[k].record(s_h2d)
            stream.wait_event(h2d_done[k])
            if k >= 2:
                stream.wait_event(d2h_done[k - 2])           # output buffer i downloaded
            sc = N.gdn_batch_schedule(B=w.B, n_max=w.n_max, nb_max=gs.nb_cap, depth_max=depth, words=wd[i].data_ptr())
            X_d, BE_d, AG_d = dev_in[i]
            N.gdn_tree_verify(gs.dims, w.layers, sc, X_d, gs.conv_w, BE_d, AG_d, gs.state, gs.conv_state, out[i],
                              gs.boundary, ver.banks, ver.workspace, ver.ws_bytes, N.GDN_VERIFY_BOUNDARY_SCRATCH, stream)
            N.gdn_commit_fold(gs.dims, w.layers, sc, paths[s][0], paths[s][1], 0, ver.banks, stream)
            cmp_done[k].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(cmp_done[k])
                o_host[i].copy_(out[i], non_blocking=True)
                d2h_done[k].record(s_d2h)
            units += int(np.asarray(n).sum()) * w.layers * w.Hv
        s_d2h.wait_event(d2h_done[nsteps - 1])
        e1.record(s_d2h)
        torch.cuda.synchronize(dev)
        # the interval between consecutive steps' compute ends: the pipeline's period, step by step
        per = [cmp_done[k - 1].elapsed_time(cmp_done[k]) for k in range(1, nsteps)]
        return e0.elapsed_time(e1), units, per

    run(warm)
    ms, units, per = run(steps)
    med = statistics.median(per) if per else float("nan")
    return dict(ms=ms, units=units, steps=steps, h2d=h2d, d2h=d2h, step_ms_median=med,
                step_ms_max=max(per) if per else float("nan"),
                stalled_steps=sum(1 for x in per if x > 2.0 * med))


def device_inputs(w: S.Workload, dev, seed: int):
    """Seeded inputs generated on the device with the workload's value recipe (host generation of the
    128-request configurations would take minutes): x ~ N(0, 1), beta = sigmoid(N(0, 1)) and
    log g = -softplus(N(0, 1)) in the input dtype; returns (x, beta, log_g)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    dt = torch.bfloat16 if w.in_dtype == S.DTYPE_BF16 else torch.float32
    sh = (w.B, w.layers, w.n_max)
    x = torch.randn(*sh, w.C, generator=g, device=dev).to(dt)
    be = torch.sigmoid(torch.randn(*sh, w.Hv, generator=g, device=dev)).to(dt)
    ag = (-torch.nn.functional.softplus(torch.randn(*sh, w.Hv, generator=g, device=dev))).to(dt)
    return x, be, ag


def run_config(cfg: int, dev, steps: int = 6, warmup: int = 3):
    """One bench line per further configuration: the verify -> commit loop on seeded synthetic inputs of that
    configuration's shapes (trees and accepted paths from the host generators, activations and states
    generated on the device), boundary states as scratch, CUDA events around every verify call."""
    import torch
    from gated_deltanet_tree_gb300 import _native as N
    from gated_deltanet_tree_gb300.runtime import TreeVerifier, paths_tensor
    from harness import dims_for
    w = S.workload(cfg)
    dims = dims_for(w)
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + cfg)
    f32 = dict(dtype=torch.float32, device=dev)
    state = torch.randn(w.B, w.layers, w.Hv, w.dk, w.dv, generator=g, **f32).mul_(0.1)
    conv_state = torch.randn(w.B, w.layers, max(w.K - 1, 0), w.C, generator=g, **f32)
    conv_w = torch.randn(w.layers, w.C, w.K, generator=g, **f32).mul_(1.0 / math.sqrt(w.K))
    out_o = torch.empty(w.B, w.layers, w.n_max, w.Hv, w.dv, **f32)
    ver = TreeVerifier(dims, w.B, w.layers, w.n_max, dev)
    inputs = [device_inputs(w, dev, 77 * cfg + i) for i in range(2)]   # two activation sets, alternated
    trees = [[S.tree_for(w, b, s) for b in range(w.B)] for s in range(w.steps)]
    paths = [[S.path_for(w, trees[s][b], b, s) for b in range(w.B)] for s in range(w.steps)]
    words, depth, nreq = [], [], []
    for s in range(w.steps):
        P = np.full((w.B, w.n_max), -1, dtype=np.int32)
        n = np.zeros(w.B, dtype=np.int32)
        for b, p in enumerate(trees[s]):
            P[b, :len(p)] = p
            n[b] = len(p)
        wd, _, dm = N.gdn_pack_schedules(P, n, with_depth=True)
        words.append(torch.from_numpy(wd).to(dev))
        depth.append(dm)
        nreq.append([len(p) for p in trees[s]])
    pt = [paths_tensor(paths[s], w.n_max, dev) for s in range(w.steps)]
    # the tree-masked UT kernels store no state but the committed one with boundary states as scratch, and a
    # pure chain stashes nothing, so no boundary buffer is needed (nb_max = 0)
    dummy = torch.empty(16, **f32)
    chains = w.tree == "chain" and w.dv == 128   # every tree a chain: 16-node segments on the tensor cores
    flags = N.GDN_VERIFY_BOUNDARY_SCRATCH | (N.GDN_VERIFY_CHAINS if chains else 0)

    def one(i, ev=None):
        s = i % w.steps
        X, BE, AG = inputs[i % 2]
        sc = N.gdn_batch_schedule(B=w.B, n_max=w.n_max, nb_max=0, depth_max=depth[s], words=words[s].data_ptr())
        if ev is not None:
            ev[0].record()
        N.gdn_tree_verify(dims, w.layers, sc, X, conv_w, BE, AG, state, conv_state, out_o, dummy, ver.banks,
                          ver.workspace, ver.ws_bytes, flags, None)
        if ev is not None:
            ev[1].record()
        N.gdn_commit_fold(dims, w.layers, sc, pt[s][0], pt[s][1], 0, ver.banks, None)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize(dev)
    ver.check_error()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for k in range(steps):
        one(warmup + k, evs[k])
    t1.record()
    torch.cuda.synchronize(dev)
    ver.check_error()
    ms = t0.elapsed_time(t1)
    vms = [a.elapsed_time(b) for a, b in evs]
    units = sum(sum(nreq[(warmup + k) % w.steps]) for k in range(steps)) * w.layers * w.Hv
    byts, fmas, tflops, walked = [], [], [], False
    for k in range(steps):
        i = warmup + k
        s = i % w.steps
        prev = paths[(i - 1) % w.steps]
        L = [len(p) for p in prev]
        byts.append(algorithmic_bytes(w, nreq[s], [0] * w.B, L))
        if chains:   # the running state absorbs every segment but the last; the products run on the tensor cores
            fmas.append(algorithmic_fma(w, [0] * w.B, [n - ((n - 1) % CHAIN_SEG + 1) for n in nreq[s]], L))
            tflops.append(chain_tensor_flops(w, nreq[s]))
            continue
        tc = tc_applies(w, depth[s])
        walk = depth[s] > UT_MAX_DEPTH and not tc
        walked = walked or walk
        ups = ([int((np.bincount(p[1:], minlength=len(p)) > 0).sum()) if len(p) > 1 else 0 for p in trees[s]]
               if walk else [0] * w.B)
        fmas.append(algorithmic_fma(w, nreq[s] if (walk or not tc) else [0] * w.B, ups, L))
        tflops.append(tensor_flops(w, nreq[s]) if tc else 0)
    peak, peak_kind = peaks()
    avg_v = statistics.mean(vms) / 1e3
    alu_peak = fp32_peak_tflops(torch.cuda.get_device_properties(dev).multi_processor_count, 2070.0)
    gbs = statistics.mean(byts) / avg_v / 1e9
    tf = 2 * statistics.mean(fmas) / avg_v / 1e12
    kernel = ("ut_tcp_verify_kernel (chains in %d-node segments on the tensor cores)" % CHAIN_SEG if chains else
              "chain_verify_kernel (heavy-light chain walk: depth > %d)" % UT_MAX_DEPTH if walked else
              "ut_tcp_verify_kernel (tensor cores, persistent)" if tc_applies(w, max(depth)) else
              "ut_verify_kernel (tree-masked UT form, CUDA cores)")
    line = {"workload": w.name, "requests": w.B, "gdn_layers": w.layers, "tree": f"{w.budget}-node {w.tree}",
            "value": units / (ms / 1e3), "unit": UNIT, "steps": steps, "warmup": warmup,
            "ms_per_step": ms / steps, "verify_ms_per_call": statistics.mean(vms),
            "us_per_call": 1e3 * statistics.mean(vms), "kernel": kernel + " + conv_window_kernel",
            "algorithmic_bytes_per_call": statistics.mean(byts),
            "hbm": {"achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak, "peak_kind": peak_kind},
            "alu": {"achieved": tf, "peak": alu_peak, "unit": "TFLOP/s", "frac": tf / alu_peak,
                    "peak_kind": "derived: SMs x 128 FP32 lanes x 2 x 2070 MHz",
                    "algorithmic_flops_per_call": 2 * statistics.mean(fmas)},
            "tensor": None if not any(tflops) else {
                "achieved": statistics.mean(tflops) / avg_v / 1e12, "peak": tf32_peak(), "unit": "TFLOP/s",
                "frac": statistics.mean(tflops) / avg_v / 1e12 / tf32_peak(),
                "tf32_flops_per_call": statistics.mean(tflops)},
            "bound": "alu" if tf / alu_peak > gbs / peak else "hbm",
            "inputs": "trees and paths from the host generators; activations, states and conv weights seeded on "
                      "the device with the same distributions; two activation sets alternate"}
    del state, conv_state, conv_w, out_o, ver, inputs, words, pt
    torch.cuda.empty_cache()
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--requests", type=int, default=None, help="override requests per GPU (smaller profiling case)")
    ap.add_argument("--layers", type=int, default=None, help="override GDN layers (smaller profiling case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ab", action="store_true", help="skip the per-node-state A/B run")
    ap.add_argument("--no-per-config", action="store_true", help="skip the lines of configurations 2, 3, 5(i), 5(ii)")
    ap.add_argument("--record-traffic", nargs="+", default=None, metavar="CSV",
                    help="write the traffic record from ncu CSV logs of a capture (with --requests, --layers "
                         "giving its blocks and --traffic-command the command) and exit")
    ap.add_argument("--traffic-command", default="")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = S.workload(args.workload)
    if args.record_traffic:
        record_traffic(args.record_traffic, (args.requests or w.B) * (args.layers or w.layers), args.traffic_command)
        return
    if args.requests:
        w = w.replace(B=args.requests)
    if args.layers:
        w = w.replace(layers=args.layers)
    config = {"workload": w.name, "requests_per_gpu": w.B, "gdn_layers": w.layers, "Hk": w.Hk, "Hv": w.Hv,
              "dk": w.dk, "dv": w.dv, "conv_K": w.K, "tree": f"{w.budget}-node top-{w.top_k} DDTree" if
              w.tree == "ddtree" else f"{w.budget}-node {w.tree}", "steps_cycle": w.steps,
              "l2": "inputs larger than L2 (state alone is %.1f GB)" % (w.B * w.layers * w.Hv * w.dk * w.dv * 4 / 1e9),
              "parallelism": f"replicas x{args.gpus}",
              "boundary_states": "scratch (GDN_VERIFY_BOUNDARY_SCRATCH): the tree-masked UT form forms no boundary "
                                 "state, so none is stored; ab_boundary_output times the same steps with every "
                                 "boundary state stored to HBM (the call's default)"}

    if args.impl == "reference":
        if rank != 0:
            return
        base = oracle_throughput(w, warmup=args.warmup, steps=args.steps)
        line = {"impl": "reference", "metric": METRIC, "value": base["value"], "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": base["ms_per_step"],
                "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": base,
                "e2e": {"value": base["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    from gated_deltanet_tree_gb300.build import build
    if rank == 0:
        build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        build()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the spawn pools start before the first GPU call of this process
        cpu = cpu_baselines(w, args.cpu_seconds)

    r = run_gpu(args, w, rank, world)
    per_config = None
    if rank == 0 and world == 1 and not args.no_per_config and args.workload == 4 and not args.requests:
        import torch
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
        per_config = {}
        for cfg, key in ((2, "2_qwen_layer_B1"), (3, "3_48_layers_B1"), (5, "5i_128x48_ddtree64_top8"),
                         (6, "5ii_128x48_chain64")):
            per_config[key] = run_config(cfg, dev, steps=8 if cfg <= 3 else 4, warmup=3 if cfg <= 3 else 2)
    if rank != 0:
        return
    value = r["units"] / (r["ms"] / 1e3)
    e2e = r["e2e"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (bf16 inputs)", "data": "synthetic (seeded DDTree-shaped trees, "
        "random activations; no model weights)", "config": config,
        "roofline": {"bound": "hbm" if r["avg_bytes"] / (r["peak"] * 1e9) >= r["avg_flops"] / (r["alu_peak"] * 1e12)
                     else "alu",
                     "kernel": "gdn_tree_verify (conv_window_kernel + "
                               + ("chain_verify_kernel)" if r["walked"] else
                                  "ut_tcp_verify_kernel)" if tc_applies(w) else "ut_verify_kernel)"),
                     "achieved": r["achieved"], "peak": r["peak"], "unit": "GB/s",
                     "frac": r["achieved"] / r["peak"], "peak_kind": r["peak_kind"],
                     "algorithmic_bytes_per_launch": r["avg_bytes"],
                     "avg_launch_ms": statistics.mean(r["verify_ms"]),
                     # the call's spread over the K timed calls (each timed alone with CUDA events)
                     "median_launch_ms": statistics.median(r["verify_ms"]),
                     "min_launch_ms": min(r["verify_ms"]), "max_launch_ms": max(r["verify_ms"]),
                     "traffic": measured_traffic(w.B * w.layers),
                     "traffic_note": "DRAM bytes of the whole call (both kernels) per launch, scaled from the committed "
                                     "small-case capture (profiles/traffic_gdn_tree_verify_batched32x48.txt); null once a "
                                     "kernel changed since",
                     "alu": {"achieved": r["avg_flops"] / r["avg_verify_s"] / 1e12, "peak": r["alu_peak"],
                             "unit": "TFLOP/s", "frac": r["avg_flops"] / r["avg_verify_s"] / 1e12 / r["alu_peak"],
                             "peak_kind": "derived: SMs x 128 FP32 lanes x 2 x max SM clock",
                             "algorithmic_flops_per_launch": r["avg_flops"]},
                     "tensor": None if not r["avg_tflops"] else {
                             "achieved": r["avg_tflops"] / r["avg_verify_s"] / 1e12, "peak": tf32_peak(),
                             "unit": "TFLOP/s", "frac": r["avg_tflops"] / r["avg_verify_s"] / 1e12 / tf32_peak(),
                             "peak_kind": "measured bf16 burst x 1/2 (nominal tf32 : bf16)",
                             "tf32_flops_per_launch": r["avg_tflops"]}},
        "finish_ms": r["finish_ms"],
        "clocks": r["clocks"],
        "e2e": None if args.no_e2e else {
            "value": r["e2e_units"] / (r["e2e_ms"] / 1e3), "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
            "d2h_bytes_per_step": e2e["d2h"], "steps": e2e["steps"],
            "host_per_step": ("DDTree construction from the draft tables, " if w.tree == "ddtree" else "")
                             + "heavy-light schedules, packing",
            # rank 0's pipeline period step by step (uploads, compute and downloads overlap across steps):
            # the median is the steady state; a stalled step took over twice the median (host-link stalls of
            # tens of ms also hit plain pinned copies with no kernel running)
            "step_ms_median": e2e.get("step_ms_median"), "step_ms_max": e2e.get("step_ms_max"),
            "stalled_steps": e2e.get("stalled_steps")},
        "gpu_launches": r["gpu_launches"],
        "ab_boundary_output": None if r["bout"] is None else dict(
            r["bout"], cost_vs_scratch=r["bout"]["ms_per_step"] / (r["ms"] / args.steps)),
        "ab_tc_per_head": None if r["tc1"] is None else dict(
            r["tc1"], persistent_speedup=r["tc1"]["ms_per_step"] / (r["ms"] / args.steps)),
        "ab_ut_simt": None if r["simt"] is None else dict(
            r["simt"], tc_speedup=r["simt"]["ms_per_step"] / (r["ms"] / args.steps)),
        "ab_chain_walk": None if r["walk"] is None else dict(
            r["walk"], ut_speedup=r["walk"]["ms_per_step"] / (r["ms"] / args.steps)),
        "ab_per_node_states": None if r["ab"] is None else dict(
            r["ab"], hld_speedup=r["ab"]["ms_per_step"] / r["walk"]["ms_per_step"],
            ut_speedup=r["ab"]["ms_per_step"] / (r["ms"] / args.steps)),
        "per_config": per_config,
        "cpu_baseline": cpu,
        # rank 0's accepted paths over the workload's step cycle
        "zero_copy_acceptances": zero_copy_acceptances(
            [p for step in rank_plan_trees(w, 0)[1] for p in step]),
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
