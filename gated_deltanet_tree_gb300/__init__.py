"""State-resident verification of speculative draft trees through Gated DeltaNet layers on GB300.

The computation lives in libgdn_tree.so (hand-written CUDA for sm_103a behind a
C ABI, include/gdn_tree.h).  This package is its ctypes binding plus buffer
ownership; it has no CPU fallback.
"""
from . import _native
from ._native import (GdnError, gdn_abi_version, gdn_banks, gdn_banks_init, gdn_batch_schedule, gdn_check_error,
                      gdn_commit_fold, gdn_dims, gdn_finish, gdn_hld_schedule, gdn_last_error, gdn_pack_schedules,
                      gdn_schedule_words, gdn_tree_verify, gdn_workspace_bytes)
from .build import LIB_PATH

__all__ = ["GdnError", "gdn_abi_version", "gdn_banks", "gdn_banks_init", "gdn_batch_schedule", "gdn_check_error",
           "gdn_commit_fold", "gdn_dims", "gdn_finish", "gdn_hld_schedule", "gdn_last_error", "gdn_pack_schedules",
           "gdn_schedule_words", "gdn_tree_verify", "gdn_workspace_bytes", "LIB_PATH"]
