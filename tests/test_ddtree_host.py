"""The library's DDTree builder (gdn_ddtree_build) against the oracle (host, no GPU).

Bit-exact on every small draft table the oracle can enumerate (parent, depth,
rank and the double score), the hand-derived trees, and on full-size drafts
(top-8, depth 16, budget 64) the properties the oracle is pinned by: budget
cap, pruning threshold, ancestor closure, best-first optimality.
"""
import numpy as np
import pytest

from oracle import ddtree as D
from test_ddtree_oracle import CASES, check_properties, random_logp


@pytest.fixture(scope="module")
def N():
    from gated_deltanet_tree_gb300.build import build
    build()
    from gated_deltanet_tree_gb300 import _native
    _native.lib()
    return _native


def same(a, b):
    for key in ("parent", "depth", "rank", "score"):
        assert a[key].tolist() == b[key].tolist(), key


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_hand_derived_trees(N, case):
    t = N.gdn_ddtree_build(case["logp"], case["budget"], case["tau"], case["chain"])
    assert t["parent"].tolist() == case["parent"]
    assert t["score"].tolist() == case["score"]


@pytest.mark.parametrize("quantised", [False, True])
def test_matches_oracle_on_small_drafts(N, quantised):
    rng = np.random.default_rng(21 if quantised else 20)
    for trial in range(300):
        depth = int(rng.integers(0, 6))
        k = int(rng.integers(1, 5))
        if k ** depth > 1500:
            depth = 3
        lp = random_logp(rng, depth, k, quantised) if depth > 0 else np.zeros((0, k), np.float32)
        budget = int(rng.integers(1, 65))
        tau = [None, 0.0, 0.5, 2.0, 6.0][trial % 5]
        chain = bool(trial % 3)
        same(N.gdn_ddtree_build(lp, budget, tau, chain), D.ddtree(lp, budget, tau, chain))


@pytest.mark.parametrize("tau", [None, 6.0, 2.0])
def test_full_size_drafts_keep_the_properties(N, tau):
    rng = np.random.default_rng(30)
    for trial in range(40):
        lp = random_logp(rng, 16, 8, quantised=bool(trial % 4 == 0))
        for budget in (16, 22, 64):
            for chain in (True, False):
                t = N.gdn_ddtree_build(lp, budget, tau, chain)
                check_properties(lp, budget, tau, chain, t)


def test_batch_matches_single_and_feeds_the_schedule(N):
    rng = np.random.default_rng(40)
    B, n_max = 12, 24
    lp = np.stack([random_logp(rng, 10, 4) for _ in range(B)])
    parents, n = N.gdn_ddtree_build_batch(lp, 22, n_max, tau=6.0)
    for b in range(B):
        one = N.gdn_ddtree_build(lp[b], 22, 6.0, True)
        assert n[b] == len(one["parent"])
        assert parents[b, :n[b]].tolist() == one["parent"].tolist()
        assert (parents[b, n[b]:] == -1).all()
    words, nb = N.gdn_pack_schedules(parents, n)
    assert words.shape == (B, N.gdn_schedule_words(n_max)) and nb >= 0


def test_rejects_bad_arguments(N):
    ok = np.array([[-0.5, -1.0]], dtype=np.float32)
    for bad, status in ((np.array([[0.5, -1.0]], np.float32), N.GDN_ERR_INVALID_ARG),
                        (np.array([[np.nan, -1.0]], np.float32), N.GDN_ERR_INVALID_ARG)):
        with pytest.raises(N.GdnError) as e:
            N.gdn_ddtree_build(bad, 4)
        assert e.value.status == status
    for budget in (0, N.GDN_MAX_NODES + 1):
        with pytest.raises(N.GdnError) as e:
            N.gdn_ddtree_build(ok, budget)
        assert e.value.status == N.GDN_ERR_UNSUPPORTED
    with pytest.raises(N.GdnError) as e:
        N.gdn_ddtree_build(ok, 4, tau=float("nan"))
    assert e.value.status == N.GDN_ERR_INVALID_ARG
    with pytest.raises(N.GdnError) as e:
        N.gdn_ddtree_build_batch(ok[None], 8, 4)
    assert e.value.status == N.GDN_ERR_INVALID_ARG


def test_rebuilds_the_workload_trees_from_their_draft_tables(N):
    # the batched workload's trees come from a separate Python generator; built from the same draws by the
    # library they come out identical (DFS numbering included)
    import synthetic as S
    for cfg in (4, 5):
        w = S.workload(cfg)
        for step in range(2):
            lp = np.stack([S.draft_logp(w, b, step) for b in range(8)])
            parents, n = N.gdn_ddtree_build_batch(lp, w.budget, w.n_max)
            for b in range(8):
                assert parents[b, :n[b]].tolist() == S.tree_for(w, b, step).tolist()
