"""ctypes binding of libgdn_tree.so -- argument marshalling only.

The functions carry the names of the C entry points declared in
include/gdn_tree.h.  Every step of the computation runs in the CUDA library;
this module only turns tensors into pointers and statuses into exceptions.  If
the library has not been built, loading it raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from .build import LIB_PATH

c_i32 = ctypes.c_int32
c_p = ctypes.c_void_p

GDN_OK = 0
GDN_ERR_INVALID_ARG = -1
GDN_ERR_INVALID_TREE = -2
GDN_ERR_INVALID_PATH = -3
GDN_ERR_UNSUPPORTED = -4
GDN_ERR_CUDA = -5
GDN_ERR_TIMEOUT = -6
GDN_ERR_CAPACITY = -7
GDN_ERR_STATE = -8
GDN_ERR_SCHEDULE = -9
GDN_DTYPE_F32 = 0
GDN_DTYPE_BF16 = 1
GDN_COMMIT_COMPACT = 1
GDN_VERIFY_BOUNDARY_SCRATCH = 1
GDN_VERIFY_CHAIN_WALK = 2
GDN_VERIFY_UT_SIMT = 4
GDN_VERIFY_TC_PER_HEAD = 8
GDN_VERIFY_CHAINS = 16
GDN_MAX_NODES = 64


class GdnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"gdn status {status}: {msg}")
        self.status = status


class gdn_dims(ctypes.Structure):
    _fields_ = [("Hk", c_i32), ("Hv", c_i32), ("dk", c_i32), ("dv", c_i32), ("K", c_i32),
                ("conv_mode", c_i32), ("act", c_i32), ("in_dtype", c_i32),
                ("q_scale", ctypes.c_float), ("l2_eps", ctypes.c_float)]


_SCHED_ARRAYS = ["subtree", "heavy", "chain_of", "pos_in_chain", "chain_head", "chain_len", "chain_off",
                 "chain_nodes", "chain_wave", "chain_src_slot", "wave_off", "boundary_slot", "boundary_node"]


class gdn_schedule(ctypes.Structure):
    _fields_ = [("n", c_i32), ("n_chains", c_i32), ("n_waves", c_i32), ("n_boundary", c_i32)] + \
               [(name, ctypes.POINTER(c_i32)) for name in _SCHED_ARRAYS]


class gdn_batch_schedule(ctypes.Structure):
    _fields_ = [("B", c_i32), ("n_max", c_i32), ("nb_max", c_i32), ("depth_max", c_i32), ("words", c_p)]


class gdn_banks(ctypes.Structure):
    _fields_ = [("k", c_p * 2), ("u", c_p * 2), ("a", c_p * 2), ("x", c_p * 2),
                ("pend_path", c_p), ("pend_len", c_p), ("err", c_p),
                ("B", c_i32), ("layers", c_i32), ("n_max", c_i32),
                ("write_bank", c_i32), ("pend_bank", c_i32), ("verified_bank", c_i32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} is not built; run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.gdn_abi_version.restype = c_i32
        L.gdn_last_error.restype = ctypes.c_char_p
        L.gdn_hld_schedule.argtypes = [P(c_i32), c_i32, P(gdn_schedule)]
        L.gdn_schedule_words.argtypes = [c_i32]
        L.gdn_schedule_words.restype = c_i32
        L.gdn_pack_schedules.argtypes = [P(c_i32), P(c_i32), c_i32, c_i32, P(c_i32), P(c_i32), P(c_i32)]
        L.gdn_pack_schedules_per_node.argtypes = [P(c_i32), P(c_i32), c_i32, c_i32, P(c_i32), P(c_i32), P(c_i32)]
        L.gdn_ddtree_build.argtypes = [P(ctypes.c_float), c_i32, c_i32, c_i32, ctypes.c_double, c_i32, P(c_i32),
                                       P(c_i32), P(c_i32), P(ctypes.c_double), P(c_i32)]
        L.gdn_ddtree_build_batch.argtypes = [P(ctypes.c_float), c_i32, c_i32, c_i32, c_i32, ctypes.c_double, c_i32,
                                             c_i32, P(c_i32), P(c_i32)]
        L.gdn_banks_init.argtypes = [P(gdn_banks), c_i32, c_i32, c_i32]
        L.gdn_workspace_bytes.argtypes = [P(gdn_dims), c_i32, c_i32, c_i32]
        L.gdn_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_tree_verify.argtypes = [P(gdn_dims), c_i32, P(gdn_batch_schedule), c_p, c_p, c_p, c_p, c_p, c_p, c_p,
                                      c_p, P(gdn_banks), c_p, ctypes.c_size_t, c_i32, c_p]
        L.gdn_tree_verify_noalloc.argtypes = [P(gdn_dims), c_i32, P(gdn_batch_schedule), c_p, c_p, c_p, c_p, c_p,
                                              c_p, c_p, c_p, P(gdn_banks), c_i32, c_p]
        L.gdn_commit_fold.argtypes = [P(gdn_dims), c_i32, P(gdn_batch_schedule), c_p, c_p, c_i32, P(gdn_banks), c_p]
        L.gdn_finish.argtypes = [P(gdn_dims), c_i32, c_i32, c_p, c_p, P(gdn_banks), c_p]
        L.gdn_check_error.argtypes = [P(gdn_banks), c_p]
        L.gdn_selftest_wait_timeout.argtypes = [P(gdn_banks), c_p]
        for name in ("gdn_hld_schedule", "gdn_pack_schedules", "gdn_pack_schedules_per_node", "gdn_ddtree_build",
                     "gdn_ddtree_build_batch", "gdn_banks_init", "gdn_tree_verify",
                     "gdn_tree_verify_noalloc", "gdn_commit_fold", "gdn_finish", "gdn_check_error",
                     "gdn_selftest_wait_timeout"):
            getattr(L, name).restype = c_i32
        _lib = L
    return _lib


def _check(status: int):
    if status != GDN_OK:
        raise GdnError(status, lib().gdn_last_error().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gdn_abi_version() -> int:
    return lib().gdn_abi_version()


def gdn_last_error() -> str:
    return lib().gdn_last_error().decode()


def gdn_hld_schedule(parent) -> dict:
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    n = int(parent.shape[0])
    size = max(n, 1) + 1
    arrays = {name: np.full(size, -7, dtype=np.int32) for name in _SCHED_ARRAYS}
    s = gdn_schedule()
    for name in _SCHED_ARRAYS:
        setattr(s, name, arrays[name].ctypes.data_as(ctypes.POINTER(c_i32)))
    _check(lib().gdn_hld_schedule(parent.ctypes.data_as(ctypes.POINTER(c_i32)), n, ctypes.byref(s)))
    lengths = dict(subtree=n, heavy=n, chain_of=n, pos_in_chain=n, chain_head=s.n_chains, chain_len=s.n_chains,
                   chain_off=s.n_chains + 1, chain_nodes=n, chain_wave=s.n_chains, chain_src_slot=s.n_chains,
                   wave_off=s.n_waves + 1, boundary_slot=n, boundary_node=s.n_boundary)
    out = dict(n=s.n, n_chains=s.n_chains, n_waves=s.n_waves, n_boundary=s.n_boundary)
    for name in _SCHED_ARRAYS:
        out[name] = arrays[name][:lengths[name]].tolist()
    return out


def gdn_schedule_words(n_max: int) -> int:
    return lib().gdn_schedule_words(n_max)


def _pack(fn, parents: np.ndarray, n: np.ndarray, with_depth: bool):
    parents = np.ascontiguousarray(parents, dtype=np.int32)
    n = np.ascontiguousarray(n, dtype=np.int32)
    B, n_max = parents.shape
    words = np.empty((B, gdn_schedule_words(n_max)), dtype=np.int32)
    nb, depth = c_i32(0), c_i32(0)
    P = ctypes.POINTER(c_i32)
    _check(fn(parents.ctypes.data_as(P), n.ctypes.data_as(P), B, n_max, words.ctypes.data_as(P), ctypes.byref(nb),
              ctypes.byref(depth)))
    return (words, int(nb.value), int(depth.value)) if with_depth else (words, int(nb.value))


def gdn_pack_schedules(parents: np.ndarray, n: np.ndarray, with_depth: bool = False):
    """parents [B, n_max] int32 (rows padded with anything past n[b]), n [B] -> (words [B, W] int32, nb_max),
    and the deepest node's depth as a third value with with_depth."""
    return _pack(lib().gdn_pack_schedules, parents, n, with_depth)


def gdn_pack_schedules_per_node(parents: np.ndarray, n: np.ndarray, with_depth: bool = False):
    """Per-node-state schedule in the packed layout -> (words, nb_max[, depth_max])."""
    return _pack(lib().gdn_pack_schedules_per_node, parents, n, with_depth)


GDN_DDTREE_CHAIN_SEED = 1


def gdn_ddtree_build(logp: np.ndarray, budget: int, tau: Optional[float] = None, chain_seed: bool = True):
    """DDTree of one draft table logp [depth_max][top_k] -> dict(parent, depth, rank, score) in DFS preorder.
    tau None disables pruning."""
    logp = np.ascontiguousarray(logp, dtype=np.float32)
    depth_max, top_k = logp.shape
    P = ctypes.POINTER(c_i32)
    parent = np.empty(budget, dtype=np.int32)
    depth = np.empty(budget, dtype=np.int32)
    rank = np.empty(budget, dtype=np.int32)
    score = np.empty(budget, dtype=np.float64)
    n = c_i32(0)
    _check(lib().gdn_ddtree_build(logp.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), depth_max, top_k, budget,
                                  -1.0 if tau is None else float(tau), GDN_DDTREE_CHAIN_SEED if chain_seed else 0,
                                  parent.ctypes.data_as(P), depth.ctypes.data_as(P), rank.ctypes.data_as(P),
                                  score.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), ctypes.byref(n)))
    k = int(n.value)
    return {"parent": parent[:k].copy(), "depth": depth[:k].copy(), "rank": rank[:k].copy(), "score": score[:k].copy()}


def gdn_ddtree_build_batch(logp: np.ndarray, budget: int, n_max: int, tau: Optional[float] = None,
                           chain_seed: bool = True):
    """B DDTrees from logp [B][depth_max][top_k] -> (parents [B][n_max] padded with -1, n [B])."""
    logp = np.ascontiguousarray(logp, dtype=np.float32)
    B, depth_max, top_k = logp.shape
    P = ctypes.POINTER(c_i32)
    parents = np.empty((B, n_max), dtype=np.int32)
    n = np.empty(B, dtype=np.int32)
    _check(lib().gdn_ddtree_build_batch(logp.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), B, depth_max, top_k,
                                        budget, -1.0 if tau is None else float(tau),
                                        GDN_DDTREE_CHAIN_SEED if chain_seed else 0, n_max,
                                        parents.ctypes.data_as(P), n.ctypes.data_as(P)))
    return parents, n


def gdn_banks_init(banks: gdn_banks, B: int, layers: int, n_max: int):
    _check(lib().gdn_banks_init(ctypes.byref(banks), B, layers, n_max))


def gdn_workspace_bytes(dims: gdn_dims, B: int, layers: int, n_max: int) -> int:
    return int(lib().gdn_workspace_bytes(ctypes.byref(dims), B, layers, n_max))


def gdn_tree_verify(dims: gdn_dims, layers: int, sched: gdn_batch_schedule, x_raw, conv_w, beta, log_g, state,
                    conv_state, out_o, boundary_states, banks: gdn_banks, workspace, workspace_bytes: int,
                    flags: int = 0, stream=None):
    _check(lib().gdn_tree_verify(ctypes.byref(dims), layers, ctypes.byref(sched), _ptr(x_raw), _ptr(conv_w),
                                 _ptr(beta), _ptr(log_g), _ptr(state), _ptr(conv_state), _ptr(out_o),
                                 _ptr(boundary_states), ctypes.byref(banks), _ptr(workspace), workspace_bytes,
                                 flags, _stream(stream)))


def gdn_tree_verify_noalloc(dims: gdn_dims, layers: int, sched: gdn_batch_schedule, x_raw, conv_w, beta, log_g,
                            state, conv_state, out_o, boundary_states, banks: gdn_banks, flags: int = 0,
                            stream=None):
    """gdn_tree_verify without a workspace: the library's fixed device scratch is used instead."""
    _check(lib().gdn_tree_verify_noalloc(ctypes.byref(dims), layers, ctypes.byref(sched), _ptr(x_raw), _ptr(conv_w),
                                         _ptr(beta), _ptr(log_g), _ptr(state), _ptr(conv_state), _ptr(out_o),
                                         _ptr(boundary_states), ctypes.byref(banks), flags, _stream(stream)))


def gdn_commit_fold(dims: gdn_dims, layers: int, sched: gdn_batch_schedule, path, length, flags: int,
                    banks: gdn_banks, stream=None):
    _check(lib().gdn_commit_fold(ctypes.byref(dims), layers, ctypes.byref(sched), _ptr(path), _ptr(length), flags,
                                 ctypes.byref(banks), _stream(stream)))


def gdn_finish(dims: gdn_dims, B: int, layers: int, state, conv_state, banks: gdn_banks, stream=None):
    _check(lib().gdn_finish(ctypes.byref(dims), B, layers, _ptr(state), _ptr(conv_state), ctypes.byref(banks),
                            _stream(stream)))


def gdn_check_error(banks: gdn_banks, stream=None):
    _check(lib().gdn_check_error(ctypes.byref(banks), _stream(stream)))


def gdn_selftest_wait_timeout(banks: gdn_banks, stream=None):
    _check(lib().gdn_selftest_wait_timeout(ctypes.byref(banks), _stream(stream)))
