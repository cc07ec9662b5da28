"""Pins of the oracle's heavy-light schedule.

Hand-derived schedules (tests/golden/hld_hand.txt) plus the structural facts
the SpecLA article fixes for the decomposition (section "链分解与依赖波 HLD 调度"):
chains partition the nodes, a heavy child has the largest subtree, light edges
start chains (so #chains = #leaves and boundary nodes = branching nodes), a
chain's source state is materialised by a chain of the previous wave, and the
number of waves is at most floor(log2 n) + 1.
"""
import math
import os

import numpy as np
import pytest

from oracle import gdn_oracle as O
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_records(name):
    recs, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].rstrip()
            if not line.strip():
                if cur:
                    recs.append(cur)
                    cur = {}
                continue
            key, val = line.split(":", 1)
            cur[key.strip()] = [int(t) for t in val.split()]
    if cur:
        recs.append(cur)
    return recs


HAND = read_records("hld_hand.txt")


@pytest.mark.parametrize("rec", HAND, ids=[" ".join(map(str, r["parent"])) for r in HAND])
def test_hand_schedules(rec):
    s = O.hld_schedule(rec["parent"])
    for key, val in rec.items():
        if key == "parent":
            continue
        got = s[key]
        got = [got] if isinstance(got, int) else list(got)
        assert got == val, key


def brute_subtree(parent):
    n = len(parent)
    return [sum(1 for m in range(n) if v in O.root_path(parent, m)) for v in range(n)]


def check_invariants(parent):
    n = len(parent)
    s = O.hld_schedule(parent)
    sub = brute_subtree(parent)
    assert s["subtree"] == sub
    children = [[c for c in range(n) if parent[c] == v] for v in range(n)]
    for v in range(n):
        if children[v]:
            best = max(sub[c] for c in children[v])
            assert s["heavy"][v] == min(c for c in children[v] if sub[c] == best)
        else:
            assert s["heavy"][v] == -1
    # chains partition the nodes, each chain follows heavy edges head -> leaf
    nodes = s["chain_nodes"]
    assert sorted(nodes) == list(range(n))
    leaves = [v for v in range(n) if not children[v]]
    assert s["n_chains"] == len(leaves)
    for c in range(s["n_chains"]):
        ch = nodes[s["chain_off"][c]:s["chain_off"][c + 1]]
        assert ch[0] == s["chain_head"][c] and len(ch) == s["chain_len"][c]
        for a, b in zip(ch, ch[1:]):
            assert s["heavy"][a] == b
        assert s["heavy"][ch[-1]] == -1
        for i, v in enumerate(ch):
            assert s["chain_of"][v] == c and s["pos_in_chain"][v] == i
        h = ch[0]
        if h == 0:
            assert s["chain_wave"][c] == 0 and s["chain_src_slot"][c] == -1
        else:
            src = parent[h]
            assert s["heavy"][src] != h
            assert s["boundary_node"][s["chain_src_slot"][c]] == src
            assert s["chain_wave"][s["chain_of"][src]] == s["chain_wave"][c] - 1
    # boundary nodes are exactly the branching nodes
    assert s["boundary_node"] == [v for v in range(n) if len(children[v]) >= 2]
    for v in range(n):
        assert (s["boundary_slot"][v] >= 0) == (v in s["boundary_node"])
    # waves: sorted, contiguous, log-bounded
    assert s["chain_wave"] == sorted(s["chain_wave"])
    assert s["n_waves"] <= math.floor(math.log2(n)) + 1
    for w in range(s["n_waves"]):
        seg = s["chain_wave"][s["wave_off"][w]:s["wave_off"][w + 1]]
        assert seg and all(x == w for x in seg)
        heads = s["chain_head"][s["wave_off"][w]:s["wave_off"][w + 1]]
        assert heads == sorted(heads)
    return s


@pytest.mark.parametrize("n", range(1, 8))
def test_invariants_all_small_trees(n):
    for parent in S.all_trees(n):
        check_invariants(list(parent))


def test_invariants_random_and_ddtrees():
    rng = np.random.default_rng(123)
    for _ in range(300):
        n = int(rng.integers(1, 65))
        check_invariants(list(S.random_tree(n, rng)))
    for seed in range(40):
        check_invariants(list(S.ddtree(22, 4, 10, np.random.default_rng(seed))))
        check_invariants(list(S.ddtree(64, 8, 16, np.random.default_rng(seed))))
    check_invariants(list(S.chain_tree(64)))


def test_deterministic():
    rng = np.random.default_rng(7)
    for _ in range(20):
        p = list(S.random_tree(30, rng))
        assert O.hld_schedule(p) == O.hld_schedule(list(p))
