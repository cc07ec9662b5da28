"""Buffer ownership around the C ABI: factor banks, workspace, schedules.

PyTorch provides device memory and streams; every computation is a call into
libgdn_tree.so through the ctypes binding.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import _native as N


def make_dims(Hk: int, Hv: int, dk: int, dv: int, K: int, conv_mode: int = 1, act: int = 1,
              in_dtype: int = N.GDN_DTYPE_BF16, q_scale: float = 1.0, l2_eps: float = 1e-6) -> N.gdn_dims:
    return N.gdn_dims(Hk=Hk, Hv=Hv, dk=dk, dv=dv, K=K, conv_mode=conv_mode, act=act, in_dtype=in_dtype,
                      q_scale=q_scale, l2_eps=l2_eps)


def channels(d: N.gdn_dims) -> int:
    return 2 * d.Hk * d.dk + d.Hv * d.dv


class DeviceSchedule:
    """A packed batch schedule resident on the device."""

    def __init__(self, parents: Sequence[np.ndarray], n_max: int, device, nb_cap: Optional[int] = None,
                 words_out: Optional[torch.Tensor] = None, stream=None, per_node: bool = False):
        B = len(parents)
        P = np.full((B, n_max), -1, dtype=np.int32)
        n = np.zeros(B, dtype=np.int32)
        for b, p in enumerate(parents):
            P[b, :len(p)] = p
            n[b] = len(p)
        pack = N.gdn_pack_schedules_per_node if per_node else N.gdn_pack_schedules
        words, nb, depth = pack(P, n, with_depth=True)
        self.parents, self.n, self.nb_max = P, n, nb if nb_cap is None else max(nb, nb_cap)
        self.depth_max = depth
        if words_out is None:
            self.words = torch.from_numpy(words).to(device)
        else:
            words_out.copy_(torch.from_numpy(words), non_blocking=False)
            self.words = words_out
        self.host_words = words
        self.struct = N.gdn_batch_schedule(B=B, n_max=n_max, nb_max=self.nb_max, depth_max=depth,
                                           words=self.words.data_ptr())


class TreeVerifier:
    """Factor banks, pending-path record, error words and workspace for one batch shape."""

    def __init__(self, dims: N.gdn_dims, B: int, layers: int, n_max: int, device="cuda"):
        self.dims, self.B, self.layers, self.n_max = dims, B, layers, n_max
        self.device = torch.device(device)
        f32 = dict(dtype=torch.float32, device=self.device)
        C = channels(dims)
        rows = B * layers * n_max
        self.bank_k = [torch.zeros(rows * dims.Hk * dims.dk, **f32) for _ in range(2)]
        self.bank_u = [torch.zeros(rows * dims.Hv * dims.dv, **f32) for _ in range(2)]
        self.bank_a = [torch.zeros(rows * dims.Hv, **f32) for _ in range(2)]
        self.bank_x = [torch.zeros(rows * C, **f32) if dims.conv_mode == 1 else None for _ in range(2)]
        i32 = dict(dtype=torch.int32, device=self.device)
        self.pend_path = torch.zeros(B * n_max, **i32)
        self.pend_len = torch.zeros(B, **i32)
        self.err = torch.zeros(4, **i32)
        self.ws_bytes = N.gdn_workspace_bytes(dims, B, layers, n_max)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.banks = N.gdn_banks()
        for i in range(2):
            self.banks.k[i] = self.bank_k[i].data_ptr()
            self.banks.u[i] = self.bank_u[i].data_ptr()
            self.banks.a[i] = self.bank_a[i].data_ptr()
            self.banks.x[i] = self.bank_x[i].data_ptr() if self.bank_x[i] is not None else None
        self.banks.pend_path = self.pend_path.data_ptr()
        self.banks.pend_len = self.pend_len.data_ptr()
        self.banks.err = self.err.data_ptr()
        N.gdn_banks_init(self.banks, B, layers, n_max)

    # bank views ---------------------------------------------------------------
    def bank_view(self, field: str, i: int) -> torch.Tensor:
        d, sh = self.dims, (self.B, self.layers, self.n_max)
        if field == "k":
            return self.bank_k[i].view(*sh, d.Hk, d.dk)
        if field == "u":
            return self.bank_u[i].view(*sh, d.Hv, d.dv)
        if field == "a":
            return self.bank_a[i].view(*sh, d.Hv)
        if field == "x":
            return self.bank_x[i].view(*sh, channels(d))
        raise KeyError(field)

    # calls ---------------------------------------------------------------------
    def schedule(self, parents: Sequence[np.ndarray], nb_cap: Optional[int] = None,
                 per_node: bool = False) -> DeviceSchedule:
        return DeviceSchedule(parents, self.n_max, self.device, nb_cap, per_node=per_node)

    def verify(self, sched: DeviceSchedule, x_raw, conv_w, beta, log_g, state, conv_state, out_o, boundary,
               stream=None, boundary_scratch: bool = False, chain_walk: bool = False, ut_simt: bool = False,
               tc_per_head: bool = False, chains: bool = False):
        flags = (N.GDN_VERIFY_BOUNDARY_SCRATCH if boundary_scratch else 0) | \
                (N.GDN_VERIFY_CHAIN_WALK if chain_walk else 0) | \
                (N.GDN_VERIFY_UT_SIMT if ut_simt else 0) | \
                (N.GDN_VERIFY_TC_PER_HEAD if tc_per_head else 0) | \
                (N.GDN_VERIFY_CHAINS if chains else 0)
        N.gdn_tree_verify(self.dims, self.layers, sched.struct, x_raw, conv_w, beta, log_g, state, conv_state,
                          out_o, boundary, self.banks, self.workspace, self.ws_bytes, flags, stream)

    def commit(self, sched: DeviceSchedule, path: torch.Tensor, length: torch.Tensor, compact: bool = False,
               stream=None):
        N.gdn_commit_fold(self.dims, self.layers, sched.struct, path, length,
                          N.GDN_COMMIT_COMPACT if compact else 0, self.banks, stream)

    def finish(self, state, conv_state, stream=None):
        N.gdn_finish(self.dims, self.B, self.layers, state, conv_state, self.banks, stream)

    def check_error(self, stream=None):
        N.gdn_check_error(self.banks, stream)


def paths_tensor(paths: Sequence[Sequence[int]], n_max: int, device) -> tuple:
    """Host paths -> (path [B, n_max] int32, len [B] int32) device tensors."""
    B = len(paths)
    P = np.zeros((B, n_max), dtype=np.int32)
    L = np.zeros(B, dtype=np.int32)
    for b, p in enumerate(paths):
        P[b, :len(p)] = p
        L[b] = len(p)
    return torch.from_numpy(P).to(device), torch.from_numpy(L).to(device)
