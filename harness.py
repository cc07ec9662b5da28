"""Runs a synthetic workload through the CUDA library (no oracle here).

Shared by the GPU tests, __graft_entry__.smoke() and bench.py: it turns the
seeded inputs of ``synthetic`` into device tensors laid out as include/gdn_tree.h
describes and drives verify -> commit steps through the C ABI.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

import synthetic as S
from gated_deltanet_tree_gb300 import _native as N
from gated_deltanet_tree_gb300.runtime import DeviceSchedule, TreeVerifier, make_dims, paths_tensor


def dims_for(w: S.Workload) -> N.gdn_dims:
    return make_dims(w.Hk, w.Hv, w.dk, w.dv, w.K, w.conv_mode, w.act,
                     N.GDN_DTYPE_BF16 if w.in_dtype == S.DTYPE_BF16 else N.GDN_DTYPE_F32, w.q_scale, w.l2_eps)


def host_to_device(a: np.ndarray, device, bf16: bool) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if bf16 else torch.from_numpy(a)
    return t.to(device)


class WorkloadPlan:
    """Trees and accepted paths of every step (host), generated up front."""

    def __init__(self, w: S.Workload, trees: Optional[List[List[np.ndarray]]] = None,
                 paths: Optional[List[List[np.ndarray]]] = None, per_node: bool = False,
                 chain_walk: bool = False, ut_simt: bool = False, tc_per_head: bool = False):
        self.w = w
        self.per_node = per_node   # per-node-state schedules instead of heavy-light ones
        self.chain_walk = chain_walk or per_node   # walk the schedule's chains (else the tree-masked UT form)
        self.ut_simt = ut_simt     # the UT form on the CUDA cores even where the tensor-core kernel applies
        self.tc_per_head = tc_per_head   # the tensor-core UT form with a CTA per v-head instead of the persistent one
        self.chains = False        # every tree is a chain: long chains solved in segments on the tensor cores
        self.depth_hint = True   # pass the trees' depth, which sends trees deeper than GDN_UT_MAX_DEPTH to the walk
        self.trees = trees if trees is not None else [S.step_trees(w, s) for s in range(w.steps)]
        self.paths = paths if paths is not None else [S.step_paths(w, self.trees[s], s) for s in range(w.steps)]
        self.nb_cap = 0
        for s in range(w.steps):
            P = np.full((w.B, w.n_max), -1, dtype=np.int32)
            n = np.zeros(w.B, dtype=np.int32)
            for b, p in enumerate(self.trees[s]):
                P[b, :len(p)] = p
                n[b] = len(p)
            _, nb = (N.gdn_pack_schedules_per_node if per_node else N.gdn_pack_schedules)(P, n)
            self.nb_cap = max(self.nb_cap, nb)


class GpuSession:
    """Device state of a workload: recurrent state, conv window, per-step inputs, outputs."""

    def __init__(self, w: S.Workload, plan: Optional[WorkloadPlan] = None, device="cuda",
                 preload_steps: Sequence[int] = (), layer_ids: Optional[Sequence[int]] = None):
        self.w = w
        self.plan = plan or WorkloadPlan(w)
        self.device = torch.device(device)
        self.dims = dims_for(w)
        self.bf16 = w.in_dtype == S.DTYPE_BF16
        # the call covers these layers of the workload (all by default; a subset for layer-chunked calls)
        self.layer_ids = list(range(w.layers)) if layer_ids is None else list(layer_ids)
        B, L, n = w.B, len(self.layer_ids), w.n_max
        self.ver = TreeVerifier(self.dims, B, L, n, device)
        f32 = dict(dtype=torch.float32, device=self.device)
        self.state = torch.empty(B, L, w.Hv, w.dk, w.dv, **f32)
        self.conv_state = torch.empty(B, L, max(w.K - 1, 0), w.C, **f32)
        for b in range(B):
            T, W = S.batch_state(w, requests=[b], layers=self.layer_ids)
            self.state[b].copy_(torch.from_numpy(T[0]))
            self.conv_state[b].copy_(torch.from_numpy(W[0]))
        self.conv_w = torch.from_numpy(S.batch_conv_weight(w, layers=self.layer_ids)).to(self.device)
        self.out_o = torch.zeros(B, L, n, w.Hv, w.dv, **f32)
        self.nb_cap = max(self.plan.nb_cap, 1)
        self.boundary = torch.zeros(B, L, self.nb_cap, w.Hv, w.dk, w.dv, **f32)
        self.inputs: Dict[int, tuple] = {}
        for s in preload_steps:
            self.inputs[s] = self._upload_step(s)
        self.scheds: Dict[int, DeviceSchedule] = {}
        self.path_t: Dict[int, tuple] = {}

    def _upload_step(self, step: int):
        w = self.w
        in_dt = torch.bfloat16 if self.bf16 else torch.float32
        L = len(self.layer_ids)
        X = torch.empty(w.B, L, w.n_max, w.C, dtype=in_dt, device=self.device)
        BE = torch.empty(w.B, L, w.n_max, w.Hv, dtype=in_dt, device=self.device)
        AG = torch.empty(w.B, L, w.n_max, w.Hv, dtype=in_dt, device=self.device)
        for b in range(w.B):
            x, be, ag = S.batch_node_inputs(w, step, requests=[b], layers=self.layer_ids)
            X[b].copy_(host_to_device(x[0], "cpu", self.bf16))
            BE[b].copy_(host_to_device(be[0], "cpu", self.bf16))
            AG[b].copy_(host_to_device(ag[0], "cpu", self.bf16))
        return X, BE, AG

    def step_inputs(self, step: int):
        if step not in self.inputs:
            self.inputs[step] = self._upload_step(step)
        return self.inputs[step]

    def schedule(self, step: int) -> DeviceSchedule:
        if step not in self.scheds:
            self.scheds[step] = self.ver.schedule(self.plan.trees[step], nb_cap=self.nb_cap,
                                                  per_node=self.plan.per_node)
            if not self.plan.depth_hint:
                self.scheds[step].struct.depth_max = 0
        return self.scheds[step]

    def paths(self, step: int):
        if step not in self.path_t:
            self.path_t[step] = paths_tensor(self.plan.paths[step], self.w.n_max, self.device)
        return self.path_t[step]

    def verify(self, step: int, stream=None, boundary_scratch: bool = False):
        X, BE, AG = self.step_inputs(step)
        self.ver.verify(self.schedule(step), X, self.conv_w, BE, AG, self.state, self.conv_state, self.out_o,
                        self.boundary, stream, boundary_scratch, self.plan.chain_walk, self.plan.ut_simt,
                        self.plan.tc_per_head, self.plan.chains)

    def local_layer(self, l: int) -> int:
        return self.layer_ids.index(l)

    def commit(self, step: int, compact: bool = False, stream=None):
        P, L = self.paths(step)
        self.ver.commit(self.schedule(step), P, L, compact, stream)

    def finish(self, stream=None):
        self.ver.finish(self.state, self.conv_state, stream)

    def drop_step(self, step: int):
        self.inputs.pop(step, None)
