"""Host-side checks of the C ABI library (no GPU needed).

The library must load, export every function include/gdn_tree.h declares, give
the oracle's heavy-light schedule bit for bit, pack it in the documented
layout, and reject bad arguments before launching anything.  Calls here never
reach a kernel launch: every argument set fails a host check first.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import gdn_oracle as O
import synthetic as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def N():
    from gated_deltanet_tree_gb300.build import build
    build()
    from gated_deltanet_tree_gb300 import _native
    _native.lib()
    return _native


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn_tree.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:gdn_status|size_t|int32_t|const char\s*\*)\s*(gdn_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_function(N):
    names = declared_functions()
    assert len(names) >= 11, names
    lib = ctypes.CDLL(N.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in gdn_tree.h but not exported"
    version = re.search(r"#define GDN_ABI_VERSION (\d+)", open(os.path.join(ROOT, "include", "gdn_tree.h")).read())
    assert N.gdn_abi_version() == int(version.group(1))


def _compare(N, parent):
    got = N.gdn_hld_schedule(parent)
    ref = O.hld_schedule(list(parent))
    for key, val in ref.items():
        assert got[key] == val, (key, list(parent))


def test_hld_matches_oracle_on_every_small_tree(N):
    for n in range(1, 9):
        for parent in S.all_trees(n):
            _compare(N, parent)


def test_hld_matches_oracle_on_random_and_ddtrees(N):
    rng = np.random.default_rng(2024)
    for _ in range(10000):
        _compare(N, S.random_tree(int(rng.integers(1, 65)), rng))
    for seed in range(50):
        _compare(N, S.ddtree(22, 4, 10, np.random.default_rng(seed)))
        _compare(N, S.ddtree(64, 8, 16, np.random.default_rng(seed)))
    _compare(N, S.chain_tree(64))


def test_invalid_trees_rejected(N):
    for bad in ([0], [-1, 1], [-1, 0, 3, 1], [-1, -1], [-1, 0, 0, 5], [-1, 0, -2]):
        with pytest.raises(N.GdnError) as e:
            N.gdn_hld_schedule(np.array(bad, dtype=np.int32))
        assert e.value.status == N.GDN_ERR_INVALID_TREE
    with pytest.raises(N.GdnError):
        N.gdn_hld_schedule(np.zeros(0, dtype=np.int32))


RELOAD, RELOAD_GLOBAL, PUSH, PUSH_GLOBAL, LEAF = 1 << 8, 1 << 9, 1 << 12, 1 << 13, 1 << 16


def walk_order(parent, heavy_last):
    """Depth-first preorder; children by index, or light ones by index and the heavy child last."""
    m = len(parent)
    kids = [[] for _ in range(m)]
    for v in range(1, m):
        kids[parent[v]].append(v)
    if heavy_last:
        heavy = O.hld_schedule(list(parent))["heavy"]
        kids = [[c for c in k if c != heavy[v]] + ([heavy[v]] if heavy[v] >= 0 else []) for v, k in enumerate(kids)]
    order, stack = [], [0]
    while stack:
        v = stack.pop()
        order.append(v)
        stack.extend(reversed(kids[v]))
    return order, kids


def simulate_walk(parent, w, n_max):
    """Run the verify's walk over the ops with abstract registers and stashes; every node must start
    from its parent's state.  Returns (ops, levels, nodes pushed to HBM, nodes reloaded)."""
    m = len(parent)
    bslot = list(w[5 + n_max:5 + n_max + m])
    nflags = list(w[5 + 2 * n_max:5 + 2 * n_max + m])
    ops = [int(x) for x in w[5 + 3 * n_max:5 + 3 * n_max + m]]
    levels = int(w[4])
    assert 0 <= levels <= 2
    kids = np.bincount(np.asarray(parent[1:], dtype=np.int64), minlength=m) if m > 1 else np.zeros(1, int)
    reg, tmem, glob = None, {}, {}
    pushed_global, reloaded, used = [], [], -1
    for i, op in enumerate(ops):
        v = op & 0xFF
        if op & RELOAD:
            assert v != 0
            if op & RELOAD_GLOBAL:
                src = glob.get(bslot[parent[v]])
            else:
                lvl = (op >> 10) & 3
                assert lvl < levels
                src = tmem.get(lvl)
            assert src == parent[v], (i, v)
            reloaded.append(v)
        else:
            assert (i == 0 and v == 0) or reg == parent[v], (i, v)
        leaf = bool(op & LEAF)
        assert leaf == (kids[v] == 0)
        reg = None if leaf else v
        assert bool(op & PUSH) == bool(nflags[v] & 1)
        if op & PUSH:
            assert not leaf
            if op & PUSH_GLOBAL:
                assert bslot[v] >= 0
                glob[bslot[v]] = v
                pushed_global.append(v)
            else:
                lvl = (op >> 14) & 3
                assert lvl < levels
                tmem[lvl] = v
                used = max(used, lvl)
    assert levels == used + 1
    return ops, pushed_global, reloaded


def test_packed_layout(N):
    rng = np.random.default_rng(3)
    n_max = 24
    trees = [S.random_tree(int(rng.integers(1, n_max + 1)), rng) for _ in range(40)] + \
            [S.ddtree(22, 4, 10, rng) for _ in range(10)] + [S.chain_tree(n_max)]
    P = np.full((len(trees), n_max), -1, dtype=np.int32)
    n = np.array([len(t) for t in trees], dtype=np.int32)
    for b, t in enumerate(trees):
        P[b, :len(t)] = t
    words, nb_max = N.gdn_pack_schedules(P, n)
    assert words.shape == (len(trees), 5 + 4 * n_max)
    assert nb_max == max(O.hld_schedule(list(t))["n_boundary"] for t in trees)
    for b, t in enumerate(trees):
        s = O.hld_schedule(list(t))
        w = words[b]
        m = len(t)
        assert list(w[:4]) == [m, s["n_chains"], s["n_boundary"], s["n_waves"]]
        assert list(w[5:5 + m]) == list(t)
        assert list(w[5 + n_max:5 + n_max + m]) == s["boundary_slot"]
        ops, pushed_global, reloaded = simulate_walk(list(t), w, n_max)
        order, kids = walk_order(list(t), heavy_last=True)
        assert [op & 0xFF for op in ops] == order
        # chains stay in registers: only the later children of a branching node reload
        assert sorted(reloaded) == sorted(c for v in range(m) if len(kids[v]) >= 2 for c in kids[v][1:])
        # stashed = the boundary nodes; those at a stash depth of two or more spill to HBM
        assert sorted(v for v in range(m) if w[5 + 2 * n_max + v] & 1) == s["boundary_node"]
        light_depth = [0] * m
        for v in range(1, m):
            light_depth[v] = light_depth[t[v]] + (1 if s["heavy"][t[v]] != v else 0)
        assert sorted(pushed_global) == [v for v in s["boundary_node"] if light_depth[v] >= 2]
    with pytest.raises(N.GdnError) as e:
        N.gdn_pack_schedules(np.full((1, 65), -1, dtype=np.int32), np.array([3], dtype=np.int32))
    assert e.value.status == N.GDN_ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# argument checks of the device calls, all failing before any launch
# ---------------------------------------------------------------------------

FAKE = 1 << 20          # aligned, never dereferenced: every call below fails a host check first


def _setup(N, **dims_kw):
    kw = dict(Hk=2, Hv=4, dk=32, dv=32, K=4, conv_mode=1, act=1, in_dtype=0, q_scale=1.0, l2_eps=1e-6)
    kw.update(dims_kw)
    d = N.gdn_dims(**kw)
    banks = N.gdn_banks()
    for i in range(2):
        banks.k[i] = banks.u[i] = banks.a[i] = banks.x[i] = FAKE
    banks.pend_path = banks.pend_len = banks.err = FAKE
    N.gdn_banks_init(banks, 1, 1, 8)
    sched = N.gdn_batch_schedule(B=1, n_max=8, nb_max=2, words=FAKE)
    return d, banks, sched


def _verify(N, d, banks, sched, ws_bytes=None, **ptrs):
    p = dict(x_raw=FAKE, conv_w=FAKE, beta=FAKE, log_g=FAKE, state=FAKE, conv_state=FAKE, out_o=FAKE,
             boundary_states=FAKE, workspace=FAKE)
    p.update(ptrs)
    if ws_bytes is None:
        ws_bytes = N.gdn_workspace_bytes(d, 1, 1, 8) - 1      # always one byte short unless a test says otherwise
    return N.gdn_tree_verify(d, 1, sched, p["x_raw"], p["conv_w"], p["beta"], p["log_g"], p["state"],
                             p["conv_state"], p["out_o"], p["boundary_states"], banks, p["workspace"], ws_bytes,
                             stream=0)


def _status(fn):
    from gated_deltanet_tree_gb300._native import GdnError
    try:
        fn()
    except GdnError as e:
        return e.status
    return 0


def test_verify_rejects_bad_arguments(N):
    d, banks, sched = _setup(N)
    # the complete, well-formed argument set still stops at the 1-byte-short workspace
    assert _status(lambda: _verify(N, d, banks, sched)) == N.GDN_ERR_CAPACITY
    assert "workspace" in N.gdn_last_error()
    assert _status(lambda: _verify(N, d, banks, sched, x_raw=None)) == N.GDN_ERR_INVALID_ARG
    assert _status(lambda: _verify(N, d, banks, sched, state=FAKE + 4)) == N.GDN_ERR_INVALID_ARG
    assert "aligned" in N.gdn_last_error()
    assert _status(lambda: _verify(N, d, banks, sched, boundary_states=None)) == N.GDN_ERR_INVALID_ARG
    for bad in (dict(dk=48), dict(dv=256), dict(K=9)):
        d2, b2, s2 = _setup(N, **bad)
        assert _status(lambda: _verify(N, d2, b2, s2)) == N.GDN_ERR_UNSUPPORTED, bad
    for bad in (dict(Hv=5), dict(conv_mode=2), dict(act=3), dict(in_dtype=7), dict(l2_eps=-1.0)):
        d2, b2, s2 = _setup(N, **bad)
        assert _status(lambda: _verify(N, d2, b2, s2)) == N.GDN_ERR_INVALID_ARG, bad
    # banks sized for another batch
    d2, b2, s2 = _setup(N)
    N.gdn_banks_init(b2, 2, 1, 8)
    assert _status(lambda: _verify(N, d2, b2, s2)) == N.GDN_ERR_CAPACITY
    # schedule with too many nodes
    s3 = N.gdn_batch_schedule(B=1, n_max=65, nb_max=0, words=FAKE)
    assert _status(lambda: _verify(N, d, banks, s3)) == N.GDN_ERR_UNSUPPORTED
    # bypass mode does not need conv pointers, but still checks the rest
    d4, b4, s4 = _setup(N, conv_mode=0, act=0)
    assert _status(lambda: _verify(N, d4, b4, s4, conv_w=None, conv_state=None)) == N.GDN_ERR_CAPACITY


def test_commit_and_finish_lifecycle_checks(N):
    d, banks, sched = _setup(N)
    st = _status(lambda: N.gdn_commit_fold(d, 1, sched, FAKE, FAKE, 0, banks, stream=0))
    assert st == N.GDN_ERR_STATE                         # no verify since the last commit
    st = _status(lambda: N.gdn_commit_fold(d, 1, sched, FAKE, FAKE, 4, banks, stream=0))
    assert st == N.GDN_ERR_INVALID_ARG                   # unknown flag
    st = _status(lambda: N.gdn_commit_fold(d, 1, sched, None, FAKE, 0, banks, stream=0))
    assert st == N.GDN_ERR_INVALID_ARG
    # finish with nothing pending is a no-op that touches nothing
    assert _status(lambda: N.gdn_finish(d, 1, 1, FAKE, FAKE, banks, stream=0)) == 0
    banks.pend_bank = 0                                  # inconsistent with write_bank = 0
    assert _status(lambda: N.gdn_finish(d, 1, 1, FAKE, FAKE, banks, stream=0)) == N.GDN_ERR_STATE
    with pytest.raises(N.GdnError):
        N.gdn_banks_init(banks, 0, 1, 8)


def test_workspace_bytes(N):
    d = N.gdn_dims(Hk=16, Hv=48, dk=128, dv=128, K=4, conv_mode=1, act=1, in_dtype=1, q_scale=1.0, l2_eps=1e-6)
    got = N.gdn_workspace_bytes(d, 32, 48, 22)
    rows = 32 * 48 * 22
    assert got >= rows * (16 * 128 + 48 * 128) * 4 and got % 256 == 0


def test_per_node_schedule_layout(N):
    rng = np.random.default_rng(9)
    n_max = 20
    trees = [S.random_tree(int(rng.integers(1, n_max + 1)), rng) for _ in range(30)] + [S.chain_tree(n_max)]
    P = np.full((len(trees), n_max), -1, dtype=np.int32)
    n = np.array([len(t) for t in trees], dtype=np.int32)
    for b, t in enumerate(trees):
        P[b, :len(t)] = t
    words, nb_max = N.gdn_pack_schedules_per_node(P, n)
    for b, t in enumerate(trees):
        m, w = len(t), words[b]
        kids = np.bincount(t[1:], minlength=m) if m > 1 else np.zeros(1, dtype=int)
        internal = [v for v in range(m) if kids[v] > 0]
        assert list(w[:3]) == [m, m, len(internal)] and w[4] == 0
        bslot = list(w[5 + n_max:5 + n_max + m])
        assert [v for v in range(m) if bslot[v] >= 0] == internal
        ops, pushed_global, reloaded = simulate_walk(list(t), w, n_max)
        assert [op & 0xFF for op in ops] == walk_order(list(t), heavy_last=False)[0]
        assert sorted(pushed_global) == internal          # every state with children goes to HBM ...
        assert sorted(reloaded) == list(range(1, m))      # ... and every child reloads it
    assert nb_max == max(int((np.bincount(t[1:], minlength=len(t)) > 0).sum()) if len(t) > 1 else 0 for t in trees)
