"""Pins of the DDTree oracle (oracle/ddtree.py) to things other than itself.

Hand-derived trees (tests/golden/ddtree_hand.txt), closed forms (a top-1 draft
gives a chain; an unlimited budget gives the full K-ary tree), and the
properties the pages name for the builder's CPU tests (SpecLA article, section
"正确性如何保证": cumulative-score pruning, ancestor closure, budget cap) plus
best-first optimality, checked on random draft tables.
"""
import math
import os

import numpy as np
import pytest

from oracle import ddtree as D

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ddtree_hand.txt")


def load_cases():
    cases, cur = [], {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line:
            if cur:
                cases.append(cur)
                cur = {}
            continue
        if line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        cur[key.strip()] = val.strip()
    if cur:
        cases.append(cur)
    out = []
    for c in cases:
        rows = [[float(x) for x in part.split()] for part in c["logp"].split("|")]
        out.append(dict(
            logp=np.array(rows, dtype=np.float32),
            budget=int(c["budget"]),
            tau=None if c["tau"] == "off" else float(c["tau"]),
            chain=c["chain"] == "1",
            parent=[int(x) for x in c["parent"].split()],
            depth=[int(x) for x in c["depth"].split()],
            rank=[int(x) for x in c["rank"].split()],
            score=[float(x) for x in c["score"].split()],
        ))
    return out


CASES = load_cases()


def test_golden_file_has_cases():
    assert len(CASES) >= 10


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_hand_derived_trees(case):
    t = D.ddtree(case["logp"], case["budget"], case["tau"], case["chain"])
    assert t["parent"].tolist() == case["parent"]
    assert t["depth"].tolist() == case["depth"]
    assert t["rank"].tolist() == case["rank"]
    assert t["score"].tolist() == case["score"]


def random_logp(rng, depth, k, quantised=False):
    z = rng.normal(0.0, 2.0, size=(depth, k))
    if quantised:                      # coarse values make exact score ties common
        z = np.round(z * 2) / 2
    z = np.sort(z, axis=1)[:, ::-1]
    lp = z - (z.max(axis=1, keepdims=True) + np.log(np.exp(z - z.max(axis=1, keepdims=True)).sum(axis=1, keepdims=True)))
    if quantised:
        lp = np.minimum(np.round(lp * 4) / 4, 0.0)
    return lp.astype(np.float32)


def test_top1_draft_gives_a_chain():
    lp = np.array([[-0.5], [-0.25], [-1.0], [-0.125]], dtype=np.float32)
    for budget in range(1, 8):
        t = D.ddtree(lp, budget, None, True)
        n = min(budget, 5)
        assert t["parent"].tolist() == [-1] + list(range(n - 1))
        assert t["depth"].tolist() == list(range(n))
        assert t["score"].tolist() == [0.0, -0.5, -0.75, -1.75, -1.875][:n]


@pytest.mark.parametrize("depth,k", [(1, 3), (2, 3), (3, 2), (3, 3)])
def test_unlimited_budget_gives_the_full_tree(depth, k):
    rng = np.random.default_rng(7)
    lp = random_logp(rng, depth, k)
    total = sum(k ** d for d in range(depth + 1))
    for chain in (True, False):
        t = D.ddtree(lp, total + 5, None, chain)
        assert len(t["parent"]) == total
        kids = np.bincount(t["parent"][1:], minlength=total)
        for i in range(total):
            assert kids[i] == (k if t["depth"][i] < depth else 0)
            # children visited by rank in DFS preorder: ranks of i's children are 0..k-1 in order
            ch = np.nonzero(t["parent"] == i)[0]
            assert t["rank"][ch].tolist() == list(range(len(ch)))


def order_key(score, seq):
    return (-score, len(seq), seq)


def check_properties(lp, budget, tau, chain, t):
    lp64 = lp.astype(np.float64)
    n = len(t["parent"])
    seqs = D.sequences(t)
    # a valid tree in DFS preorder: parent before child, root first, the budget cap
    assert 1 <= n <= budget
    assert t["parent"][0] == -1 and all(0 <= t["parent"][i] < i for i in range(1, n))
    assert seqs == sorted(seqs)
    # cumulative scores, summed from the root down
    for i in range(n):
        s = 0.0
        for d, r in enumerate(seqs[i]):
            s = s + float(lp64[d, r])
        assert t["score"][i] == s
    q_star = float(lp64[0].max()) if lp.shape[0] > 0 else 0.0
    thr = -math.inf if tau is None else q_star - tau
    assert all(t["score"][i] >= thr for i in range(1, n))          # pruning
    kept = set(seqs)
    assert all(s[:-1] in kept for s in seqs if s)                    # ancestor closure
    # the greedy chain, as far as it is kept, is a prefix chain of best ranks
    greedy = D.greedy_chain(lp64)
    chain_kept = [g for g in greedy if g in kept]
    if chain:
        for a, g in enumerate(greedy):
            if g not in kept:
                assert all(h not in kept for h in greedy[a:])
                break
    # best-first optimality: every eligible frontier candidate left out is worse than every kept
    # non-chain node, and it is left out only because the budget is full
    K = lp.shape[1]
    frontier = []
    for s in seqs:
        if len(s) < lp.shape[0]:
            for r in range(K):
                c = s + (r,)
                if c not in kept:
                    sc = t["score"][seqs.index(s)] + float(lp64[len(s), r])
                    if sc >= thr:
                        frontier.append((sc, c))
    if frontier:
        assert n == budget
        others = [(t["score"][i], seqs[i]) for i in range(1, n) if not (chain and seqs[i] in chain_kept)]
        if others:
            worst = max(order_key(sc, s) for sc, s in others)
            best_out = min(order_key(sc, s) for sc, s in frontier)
            assert worst < best_out


@pytest.mark.parametrize("quantised", [False, True])
def test_properties_on_random_drafts(quantised):
    rng = np.random.default_rng(11 if quantised else 5)
    for trial in range(60):
        depth = int(rng.integers(1, 6))
        k = int(rng.integers(1, 4))
        lp = random_logp(rng, depth, k, quantised)
        budget = int(rng.integers(1, 30))
        tau = [None, 0.0, 1.0, 3.0, 6.0][trial % 5]
        chain = bool(trial % 2)
        check_properties(lp, budget, tau, chain, D.ddtree(lp, budget, tau, chain))


def test_budget_nesting_and_large_tau():
    rng = np.random.default_rng(3)
    for _ in range(20):
        lp = random_logp(rng, 4, 3)
        for chain in (True, False):
            prev = None
            for budget in range(1, 40):
                cur = set(D.sequences(D.ddtree(lp, budget, None, chain)))
                if prev is not None:
                    assert prev <= cur and len(cur) - len(prev) <= 1
                prev = cur
            # a margin wider than every score gap prunes nothing
            big = float(-lp.astype(np.float64).sum(axis=0).min()) * 4 + 10.0
            a = D.ddtree(lp, 30, None, chain)
            b = D.ddtree(lp, 30, big, chain)
            assert a["parent"].tolist() == b["parent"].tolist()


def test_tau_grows_the_unbudgeted_tree():
    rng = np.random.default_rng(4)
    for _ in range(20):
        lp = random_logp(rng, 4, 3)
        prev = None
        for tau in (0.0, 0.5, 1.0, 2.0, 4.0, 8.0):
            cur = set(D.sequences(D.ddtree(lp, 10 ** 6, tau, True)))
            if prev is not None:
                assert prev <= cur
            prev = cur


def test_invalid_drafts_are_rejected():
    with pytest.raises(D.InvalidDraft):
        D.ddtree(np.array([[0.5, -1.0]], dtype=np.float32), 4)
    with pytest.raises(D.InvalidDraft):
        D.ddtree(np.array([[np.nan, -1.0]], dtype=np.float32), 4)
    with pytest.raises(D.InvalidDraft):
        D.ddtree(np.array([[-1.0]], dtype=np.float32), 0)
