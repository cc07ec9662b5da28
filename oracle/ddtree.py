"""Plain CPU oracle for DDTree construction with confidence pruning.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this file; only the tests use it.

What it states (sources: the Luce DFlash README, sections "How it works" and
the server flag table -- "--ddtree-budget" is the candidate budget, 22 by
default, and "--ddtree-tau" is a confidence margin that SpecLA sets to 6; and
the SpecLA article, section "一键开启", where nodes whose score falls below
q* - tau are pruned, and section "正确性如何保证", whose CPU tests cover
cumulative-score pruning, ancestor closure and the budget cap):

* the draft gives, for each depth d = 1..D, log-probabilities logp[d-1][r] of
  its top-K tokens r = 0..K-1;
* a candidate is a sequence of ranks (r_1, ..., r_d); its score is the
  cumulative log-probability sum_i logp[i-1][r_i], added from the root down in
  double precision; the root (the empty sequence) scores 0;
* the tree is a best-first tree of at most ``budget`` nodes, root included
  (README: "a best-first tree of up to 22 nodes spans the top-K branches at
  each position").

Readings where the pages are silent (each also listed in the design notes):
* q* is the best score of any candidate.  Log-probabilities are <= 0, so a
  score never rises along a path and q* = max_r logp[0][r];
* a candidate is eligible when score >= q* - tau; tau = None disables pruning;
* with ``chain_seed`` the greedy chain (the best rank at every depth, ties to
  the lower rank) is inserted first, as far as it stays eligible and the
  budget allows;
* the other nodes are the best eligible candidates in the total order
  (higher score, then lower depth, then lexicographically smaller rank
  sequence), as many as the budget leaves.  Because scores never rise along a
  path and ties go to the lower depth, every ancestor of a chosen candidate
  precedes it in this order, so the chosen set is closed under ancestors;
* the nodes are numbered in DFS preorder with children visited by rank, so
  parent[i] < i and node 0 is the root.

This is the definition written out over an exhaustive enumeration of every
candidate, so it is meant for small K^D only.
"""
from __future__ import annotations

import itertools
from typing import Dict, List, Optional, Tuple

import numpy as np


class InvalidDraft(ValueError):
    pass


def check_logp(logp: np.ndarray) -> np.ndarray:
    """The draft's table as float64; entries must be log-probabilities (<= 0, not NaN)."""
    lp = np.asarray(logp, dtype=np.float64)
    if lp.ndim != 2:
        raise InvalidDraft("logp must be [depth][top_k]")
    if np.isnan(lp).any() or (lp > 0).any():
        raise InvalidDraft("logp entries must be log-probabilities (<= 0)")
    return lp


def score_of(lp: np.ndarray, seq: Tuple[int, ...]) -> float:
    """Cumulative log-probability, summed from the root down."""
    s = 0.0
    for i, r in enumerate(seq):
        s = s + float(lp[i, r])
    return s


def all_candidates(lp: np.ndarray) -> List[Tuple[int, ...]]:
    D, K = lp.shape
    out: List[Tuple[int, ...]] = []
    for d in range(1, D + 1):
        out.extend(itertools.product(range(K), repeat=d))
    return out


def greedy_chain(lp: np.ndarray) -> List[Tuple[int, ...]]:
    """Prefixes of the best-rank-per-depth sequence (argmax, ties to the lower rank)."""
    seq: Tuple[int, ...] = ()
    out = []
    for d in range(lp.shape[0]):
        seq = seq + (int(np.argmax(lp[d])),)
        out.append(seq)
    return out


def ddtree(logp: np.ndarray, budget: int, tau: Optional[float] = None, chain_seed: bool = True) -> Dict[str, np.ndarray]:
    """The DDTree of the definition above.

    Returns parent, depth, rank (root: -1) and score arrays in DFS preorder."""
    lp = check_logp(logp)
    if budget < 1:
        raise InvalidDraft("budget must be >= 1")
    D = lp.shape[0]
    K = lp.shape[1] if D > 0 else 0
    cands = all_candidates(lp) if K > 0 else []
    score = {c: score_of(lp, c) for c in cands}
    score[()] = 0.0
    if tau is None or not cands:
        eligible = set(cands)
    else:
        q_star = max(score[c] for c in cands)
        thr = q_star - float(tau)
        eligible = {c for c in cands if score[c] >= thr}

    chosen: List[Tuple[int, ...]] = [()]
    if chain_seed and K > 0:
        for c in greedy_chain(lp):
            if len(chosen) >= budget or c not in eligible:
                break
            chosen.append(c)
    in_set = set(chosen)
    rest = sorted((c for c in eligible if c not in in_set), key=lambda c: (-score[c], len(c), c))
    chosen.extend(rest[:max(0, budget - len(chosen))])
    in_set = set(chosen)
    for c in chosen:   # closure holds by construction; state it
        assert c == () or c[:-1] in in_set

    # DFS preorder, children by rank: that is the lexicographic order of the rank sequences
    order = sorted(chosen)
    index = {c: i for i, c in enumerate(order)}
    n = len(order)
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int32)
    rank = np.full(n, -1, dtype=np.int32)
    sc = np.zeros(n, dtype=np.float64)
    for c, i in index.items():
        depth[i] = len(c)
        sc[i] = score[c]
        if c:
            parent[i] = index[c[:-1]]
            rank[i] = c[-1]
    return {"parent": parent, "depth": depth, "rank": rank, "score": sc}


def sequences(tree: Dict[str, np.ndarray]) -> List[Tuple[int, ...]]:
    """The rank sequence of every node of a returned tree."""
    parent, rank = tree["parent"], tree["rank"]
    seqs: List[Tuple[int, ...]] = []
    for i in range(len(parent)):
        seqs.append(() if parent[i] < 0 else seqs[parent[i]] + (int(rank[i]),))
    return seqs
