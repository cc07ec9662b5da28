"""Seeded synthetic inputs for Gated DeltaNet tree verification.

This module is shared by the oracle side (tests, CPU baseline) and the CUDA side
(tests, bench).  It holds input generation only -- tree shapes, accepted paths
and tensor values -- and none of the arithmetic of the method itself (no conv,
no normalisation, no delta rule, no tree decomposition).

Workload shapes follow the SpecLA article ("Lucebox SpecLA 与 Gated DeltaNet
状态驻留验证原理指南", sections "实测收益" and "一键开启": 22-node DDTree, top-4,
tau 6) and the Luce DFlash README ("How it works", DDTree tree verify: best-first
tree with chain pre-seed; "Architecture note": 3 of every 4 layers are GDN).

Every array is a pure function of (config id, stream, request, layer, step): a
``numpy.random.Generator(PCG64(SeedSequence([...])))`` is built per block, so
any (request, layer) block can be regenerated on its own without generating the
rest of the batch.
"""
from __future__ import annotations

import dataclasses
import heapq
from typing import List, Optional, Sequence

import numpy as np

# stream ids of the seed sequence
S_TREE, S_PATH, S_X, S_BETA, S_GATE, S_STATE, S_CONVSTATE, S_CONVW = range(8)

DTYPE_F32 = 0
DTYPE_BF16 = 1


def rng_for(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


# ----------------------------------------------------------------------------
# bf16 helpers (bit patterns held in uint16; no torch needed)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  Inputs are finite here.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# tree shapes
# ----------------------------------------------------------------------------

def tiny_tree(n: int = 8, seed: int = 0) -> np.ndarray:
    """parent[0] = -1; parent[i] drawn uniformly from 0..i-1, for i = 1..n-1 in order."""
    rng = np.random.default_rng(seed)
    parent = np.empty(n, dtype=np.int32)
    parent[0] = -1
    for i in range(1, n):
        parent[i] = rng.integers(0, i)
    return parent


def random_tree(n: int, rng: np.random.Generator) -> np.ndarray:
    parent = np.empty(n, dtype=np.int32)
    parent[0] = -1
    for i in range(1, n):
        parent[i] = rng.integers(0, i)
    return parent


def chain_tree(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def all_trees(n: int):
    """Every parent array of n nodes in topological order (parent[i] < i): (n-1)! trees."""
    if n == 1:
        yield np.array([-1], dtype=np.int32)
        return
    ranges = [range(i) for i in range(1, n)]
    import itertools
    for combo in itertools.product(*ranges):
        yield np.array((-1,) + combo, dtype=np.int32)


def ddtree(budget: int, top_k: int, depth_max: int, rng: np.random.Generator,
           sigma: float = 2.0, chain_seed: bool = True) -> np.ndarray:
    """Synthetic DDTree-shaped candidate tree.

    Stand-in for the draft model: per depth d = 1..depth_max, top_k logits
    z ~ N(0, sigma^2), sorted descending, turned into log-probabilities
    (log-softmax over the top_k).  A node is a sequence of ranks; its score is
    the sum of the log-probabilities along it.  With ``chain_seed`` the greedy
    (rank-0) chain to depth_max is inserted first, then nodes are added
    best-first by score until ``budget`` nodes (root included).  Ties: lower
    depth, then lower parent id, then lower rank.  Nodes are finally renumbered
    in DFS preorder with children visited by rank, so parent[i] < i.
    """
    z = np.sort(rng.normal(0.0, sigma, size=(depth_max + 1, top_k)), axis=1)[:, ::-1]
    m = z.max(axis=1, keepdims=True)
    logp = z - (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))

    # nodes: (depth, rank, parent_build_id, score)
    depth = [0]
    rank = [0]
    par = [-1]
    score = [0.0]
    children = {0: {}}

    def add(p, r):
        d = depth[p] + 1
        nid = len(depth)
        depth.append(d)
        rank.append(r)
        par.append(p)
        score.append(score[p] + float(logp[d, r]))
        children[p][r] = nid
        children[nid] = {}
        return nid

    if chain_seed:
        cur = 0
        while len(depth) < budget and depth[cur] < depth_max:
            cur = add(cur, 0)
    heap = []

    def push_children(p):
        if depth[p] >= depth_max:
            return
        for r in range(top_k):
            if r in children[p]:
                continue
            d = depth[p] + 1
            heapq.heappush(heap, (-(score[p] + float(logp[d, r])), d, p, r))

    for nid in range(len(depth)):
        push_children(nid)
    while len(depth) < budget and heap:
        _, d, p, r = heapq.heappop(heap)
        if r in children[p]:
            continue
        nid = add(p, r)
        push_children(nid)

    # DFS preorder renumbering, children by rank
    order = []
    stack = [0]
    while stack:
        v = stack.pop()
        order.append(v)
        for r in sorted(children[v].keys(), reverse=True):
            stack.append(children[v][r])
    new_id = {old: i for i, old in enumerate(order)}
    parent = np.empty(len(order), dtype=np.int32)
    for old in order:
        parent[new_id[old]] = -1 if par[old] < 0 else new_id[par[old]]
    return parent


# ----------------------------------------------------------------------------
# accepted paths
# ----------------------------------------------------------------------------

def _children_lists(parent: np.ndarray) -> List[List[int]]:
    ch = [[] for _ in range(len(parent))]
    for i in range(1, len(parent)):
        ch[int(parent[i])].append(i)
    return ch


def random_walk_path(parent: np.ndarray, rng: np.random.Generator, max_len: Optional[int] = None,
                     uniform_len_on_walk: bool = False) -> np.ndarray:
    """A root path: from node 0 follow a uniformly chosen child.

    ``max_len`` given: the length is drawn uniformly from 1..max_len and
    clipped where the walk reaches a leaf.  ``uniform_len_on_walk``: walk to a
    leaf first and draw the length uniformly from 1..(walk length).
    """
    ch = _children_lists(parent)
    if uniform_len_on_walk:
        walk = [0]
        while ch[walk[-1]]:
            c = ch[walk[-1]]
            walk.append(c[int(rng.integers(0, len(c)))])
        L = int(rng.integers(1, len(walk) + 1))
        return np.asarray(walk[:L], dtype=np.int32)
    L = int(rng.integers(1, (max_len or len(parent)) + 1))
    walk = [0]
    while len(walk) < L and ch[walk[-1]]:
        c = ch[walk[-1]]
        walk.append(c[int(rng.integers(0, len(c)))])
    return np.asarray(walk, dtype=np.int32)


# ----------------------------------------------------------------------------
# workload configurations
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    cfg: int
    name: str
    B: int
    layers: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    K: int
    conv_mode: int          # 0 bypass, 1 causal depthwise conv
    act: int                # 0 none, 1 SiLU
    in_dtype: int           # DTYPE_F32 or DTYPE_BF16 for x, beta, log-gate
    n_max: int              # node stride
    steps: int
    tree: str               # 'tiny' | 'random' | 'ddtree' | 'chain'
    budget: int = 8
    top_k: int = 4
    depth_max: int = 10
    path: str = 'maxlen'    # 'maxlen' (L ~ U{1..path_max}, clipped) | 'walk'
    path_max: int = 10
    q_scale: float = 1.0
    l2_eps: float = 1e-6
    values: str = 'qwen'    # 'tiny' (U/N recipe) | 'qwen' (sigmoid/softplus recipe)
    edge: str = ''          # '' or a '+'-joined set of EDGE_RECIPES overwriting some of the drawn values

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def workload(cfg: int, **overrides) -> Workload:
    if cfg == 1:
        w = Workload(cfg=1, name="tiny: 1 layer, 4 heads, d=32, K=4, 8-node random tree", B=1, layers=1,
                     Hk=4, Hv=4, dk=32, dv=32, K=4, conv_mode=1, act=1, in_dtype=DTYPE_F32, n_max=8, steps=2,
                     tree='tiny', budget=8, path_max=8, values='tiny')
    elif cfg == 2:
        w = Workload(cfg=2, name="qwen-like GDN layer: Hk=16, Hv=48, d=128, K=4, 22-node top-4 DDTree, B=1",
                     B=1, layers=1, Hk=16, Hv=48, dk=128, dv=128, K=4, conv_mode=1, act=1, in_dtype=DTYPE_BF16,
                     n_max=22, steps=1, tree='ddtree', budget=22, top_k=4, depth_max=10)
    elif cfg == 3:
        w = Workload(cfg=3, name="48 qwen-like GDN layers, 22-node top-4 DDTree, B=1, commit folded before verify",
                     B=1, layers=48, Hk=16, Hv=48, dk=128, dv=128, K=4, conv_mode=1, act=1, in_dtype=DTYPE_BF16,
                     n_max=22, steps=2, tree='ddtree', budget=22, top_k=4, depth_max=10)
    elif cfg == 4:
        w = Workload(cfg=4, name="batched serving: 32 requests x 48 GDN layers, 22-node top-4 DDTree, 8 steps",
                     B=32, layers=48, Hk=16, Hv=48, dk=128, dv=128, K=4, conv_mode=1, act=1, in_dtype=DTYPE_BF16,
                     n_max=22, steps=8, tree='ddtree', budget=22, top_k=4, depth_max=10)
    elif cfg == 5:
        w = Workload(cfg=5, name="stress: 128 requests x 48 GDN layers, 64-node top-8 DDTree (depth<=16), 8 steps",
                     B=128, layers=48, Hk=16, Hv=48, dk=128, dv=128, K=4, conv_mode=1, act=1, in_dtype=DTYPE_BF16,
                     n_max=64, steps=8, tree='ddtree', budget=64, top_k=8, depth_max=16, path='walk')
    elif cfg == 6:
        w = Workload(cfg=6, name="stress: 128 requests x 48 GDN layers, 64-node pure chain, 8 steps",
                     B=128, layers=48, Hk=16, Hv=48, dk=128, dv=128, K=4, conv_mode=1, act=1, in_dtype=DTYPE_BF16,
                     n_max=64, steps=8, tree='chain', budget=64, path='walk')
    else:
        raise ValueError(f"unknown workload {cfg}")
    return w.replace(**overrides) if overrides else w


def tree_for(w: Workload, b: int, step: int) -> np.ndarray:
    if w.tree == 'tiny':
        return tiny_tree(w.budget, seed=0) if step == 0 else random_tree(w.budget, rng_for(w.cfg, S_TREE, b, step))
    if w.tree == 'random':
        return random_tree(w.budget, rng_for(w.cfg, S_TREE, b, step))
    if w.tree == 'chain':
        return chain_tree(w.budget)
    if w.tree == 'ddtree':
        return ddtree(w.budget, w.top_k, w.depth_max, rng_for(w.cfg, S_TREE, b, step))
    raise ValueError(w.tree)


def draft_logp(w: Workload, b: int, step: int) -> np.ndarray:
    """The synthetic draft's per-depth top-K log-probabilities behind tree_for's DDTree, [depth_max][top_k]
    fp32 (row d-1 = depth d), drawn from the same stream as the tree."""
    rng = rng_for(w.cfg, S_TREE, b, step)
    z = np.sort(rng.normal(0.0, 2.0, size=(w.depth_max + 1, w.top_k)), axis=1)[:, ::-1]
    m = z.max(axis=1, keepdims=True)
    logp = z - (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))
    return np.ascontiguousarray(logp[1:], dtype=np.float32)


def path_for(w: Workload, parent: np.ndarray, b: int, step: int) -> np.ndarray:
    rng = rng_for(w.cfg, S_PATH, b, step)
    if w.path == 'walk':
        return random_walk_path(parent, rng, uniform_len_on_walk=True)
    return random_walk_path(parent, rng, max_len=min(w.path_max, len(parent)))


def _to_in_dtype(w: Workload, x32: np.ndarray) -> np.ndarray:
    return f32_to_bf16_bits(x32) if w.in_dtype == DTYPE_BF16 else x32.astype(np.float32)


def node_inputs(w: Workload, b: int, l: int, step: int):
    """Per-node inputs of one (request, layer) block at one step.

    Returns (x [n_max, C], beta [n_max, Hv], log_g [n_max, Hv]) in the input
    dtype (uint16 bf16 bits or float32).  Rows past the tree's node count are
    generated too (they are never read by a correct implementation).
    """
    n, C, Hv = w.n_max, w.C, w.Hv
    rx = rng_for(w.cfg, S_X, b, l, step)
    rb = rng_for(w.cfg, S_BETA, b, l, step)
    rg = rng_for(w.cfg, S_GATE, b, l, step)
    if w.values == 'tiny':
        x = rx.standard_normal((n, C), dtype=np.float32)
        beta = rb.random((n, Hv), dtype=np.float32)
        log_g = -rg.random((n, Hv), dtype=np.float32)
    else:
        x = rx.standard_normal((n, C), dtype=np.float32)
        zb = rb.standard_normal((n, Hv), dtype=np.float32)
        beta = (1.0 / (1.0 + np.exp(-zb.astype(np.float64)))).astype(np.float32)
        zg = rg.standard_normal((n, Hv), dtype=np.float32).astype(np.float64)
        log_g = (-np.logaddexp(0.0, zg)).astype(np.float32)
    if w.edge:
        x, beta, log_g = apply_edges(w, x, beta, log_g)
    return _to_in_dtype(w, x), _to_in_dtype(w, beta), _to_in_dtype(w, log_g)


# Edge-case recipes: deterministic overwrites of the drawn values that drive the method into its degenerate
# cases.  Node and head selections depend only on indices, so every (request, layer, step) block gets them.
EDGE_RECIPES = {
    "gate_zero": "log-gate -inf (g = 0, full forget) on every third node (1, 4, 7, ...) of the even v-heads",
    "gate_floor": "log-gate -14 (g = 8.3e-7) on every node of v-heads h % 3 == 1, so gate products fall below "
                  "1e-12 after two nodes",
    "beta01": "beta = 0 on odd nodes, beta = 1 on even nodes",
    "zero_rows": "raw input row all zeros on nodes 2, 5, 8, ... (with the conv: also k-head 0's conv taps zero)",
}


def apply_edges(w: Workload, x: np.ndarray, beta: np.ndarray, log_g: np.ndarray):
    """x [n, C], beta/log_g [n, Hv] float32 -> copies with the workload's edge recipes applied."""
    x, beta, log_g = x.copy(), beta.copy(), log_g.copy()
    n = x.shape[0]
    nodes = np.arange(n)
    heads = np.arange(w.Hv)
    for e in w.edge.split("+"):
        if e == "gate_zero":
            log_g[np.ix_(nodes % 3 == 1, heads % 2 == 0)] = -np.inf
        elif e == "gate_floor":
            log_g[:, heads % 3 == 1] = -14.0
        elif e == "beta01":
            beta[nodes % 2 == 1] = 0.0
            beta[nodes % 2 == 0] = 1.0
        elif e == "zero_rows":
            x[nodes % 3 == 2] = 0.0
        else:
            raise ValueError(f"unknown edge recipe {e!r}")
    return x, beta, log_g


def init_state(w: Workload, b: int, l: int) -> np.ndarray:
    """Initial recurrent state of one (request, layer) block: [Hv, dk, dv] fp32, N(0, 0.1^2)."""
    r = rng_for(w.cfg, S_STATE, b, l)
    return (r.standard_normal((w.Hv, w.dk, w.dv), dtype=np.float32) * np.float32(0.1)).astype(np.float32)


def init_conv_state(w: Workload, b: int, l: int) -> np.ndarray:
    """Initial committed conv window of one (request, layer) block: [K-1, C] fp32, N(0, 1)."""
    r = rng_for(w.cfg, S_CONVSTATE, b, l)
    return r.standard_normal((max(w.K - 1, 0), w.C), dtype=np.float32)


def conv_weight(w: Workload, l: int) -> np.ndarray:
    """Depthwise conv weights of one layer: [C, K] fp32, N(0, 1/K)."""
    r = rng_for(w.cfg, S_CONVW, l)
    cw = (r.standard_normal((w.C, w.K), dtype=np.float32) * np.float32(1.0 / np.sqrt(w.K))).astype(np.float32)
    if "zero_rows" in w.edge.split("+"):   # k-head 0 convolves to zero: only eps keeps its k_hat finite
        cw[w.Hk * w.dk:w.Hk * w.dk + w.dk] = 0.0
    return cw


def step_trees(w: Workload, step: int) -> List[np.ndarray]:
    return [tree_for(w, b, step) for b in range(w.B)]


def step_paths(w: Workload, trees: Sequence[np.ndarray], step: int) -> List[np.ndarray]:
    return [path_for(w, trees[b], b, step) for b in range(w.B)]


def batch_node_inputs(w: Workload, step: int, requests: Optional[Sequence[int]] = None,
                      layers: Optional[Sequence[int]] = None):
    """Stacked node inputs [B', L', n_max, ...] for the chosen requests and layers."""
    requests = list(range(w.B)) if requests is None else list(requests)
    layers = list(range(w.layers)) if layers is None else list(layers)
    dt = np.uint16 if w.in_dtype == DTYPE_BF16 else np.float32
    X = np.empty((len(requests), len(layers), w.n_max, w.C), dtype=dt)
    BE = np.empty((len(requests), len(layers), w.n_max, w.Hv), dtype=dt)
    AG = np.empty((len(requests), len(layers), w.n_max, w.Hv), dtype=dt)
    for i, b in enumerate(requests):
        for j, l in enumerate(layers):
            X[i, j], BE[i, j], AG[i, j] = node_inputs(w, b, l, step)
    return X, BE, AG


def batch_state(w: Workload, requests=None, layers=None):
    requests = list(range(w.B)) if requests is None else list(requests)
    layers = list(range(w.layers)) if layers is None else list(layers)
    T = np.empty((len(requests), len(layers), w.Hv, w.dk, w.dv), dtype=np.float32)
    W = np.empty((len(requests), len(layers), max(w.K - 1, 0), w.C), dtype=np.float32)
    for i, b in enumerate(requests):
        for j, l in enumerate(layers):
            T[i, j] = init_state(w, b, l)
            W[i, j] = init_conv_state(w, b, l)
    return T, W


def batch_conv_weight(w: Workload, layers=None):
    layers = list(range(w.layers)) if layers is None else list(layers)
    return np.stack([conv_weight(w, l) for l in layers])
