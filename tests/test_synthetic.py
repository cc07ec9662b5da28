"""Checks of the seeded input generators (shapes, value recipes, determinism)."""
import numpy as np
import torch

import synthetic as S


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 100000), rng.normal(0, 1e3, 1000), [0.0, -0.0, 1.0, -2.5]]).astype(np.float32)
    ours = S.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = S.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_ddtree_shape():
    for seed in range(20):
        p = S.ddtree(22, 4, 10, np.random.default_rng(seed))
        assert len(p) == 22 and p[0] == -1 and all(0 <= p[i] < i for i in range(1, 22))
        depth = [0] * 22
        for i in range(1, 22):
            depth[i] = depth[p[i]] + 1
        assert max(depth) == 10                           # greedy chain pre-seed to depth 10
        kids = np.bincount(p[1:], minlength=22)
        assert kids.max() <= 4                            # top-4 branching
        # DFS preorder: every subtree is a contiguous index range
        for v in range(22):
            sub = [m for m in range(22) if v in _anc(p, m)]
            assert sub == list(range(v, v + len(sub)))
    p = S.ddtree(64, 8, 16, np.random.default_rng(1))
    assert len(p) == 64 and np.bincount(p[1:]).max() <= 8


def _anc(p, m):
    out = [m]
    while p[out[-1]] >= 0:
        out.append(p[out[-1]])
    return out


def test_tiny_tree_recipe():
    p = S.tiny_tree(8, 0)
    rng = np.random.default_rng(0)
    assert p[0] == -1 and all(p[i] == rng.integers(0, i) for i in range(1, 8))


def test_blocks_are_independent_of_batch():
    w = S.workload(2).replace(B=3, layers=2, n_max=5, Hk=2, Hv=4, dk=8, dv=8)
    X, BE, AG = S.batch_node_inputs(w, step=1)
    x1, b1, a1 = S.node_inputs(w, 2, 1, 1)
    np.testing.assert_array_equal(X[2, 1], x1)
    np.testing.assert_array_equal(AG[2, 1], a1)
    bf = S.bf16_bits_to_f32(BE)
    assert np.all((bf > 0) & (bf < 1))
    assert np.all(S.bf16_bits_to_f32(AG) < 0)


def test_paths_are_root_paths():
    w = S.workload(4)
    for step in range(3):
        trees = S.step_trees(w.replace(B=8), step)
        for b, p in enumerate(trees):
            path = S.path_for(w, p, b, step)
            assert path[0] == 0 and 1 <= len(path) <= 10
            for i in range(1, len(path)):
                assert p[path[i]] == path[i - 1]
