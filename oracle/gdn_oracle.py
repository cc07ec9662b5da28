"""Plain, slow, fp64 CPU oracle for Gated DeltaNet tree verification.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the CUDA library and
its Python binding) imports, calls or links this file; it is used by the tests,
by ``__graft_entry__.smoke()`` and by the CPU-baseline legs of ``bench.py``.

What it states (sources: the SpecLA article "Lucebox SpecLA 与 Gated DeltaNet
状态驻留验证原理指南" and the Luce DFlash README):

* the gated delta rule, per head, S' = g S (I - beta k k^T) + beta v k^T and
  o = S' q, with L2-normalised q and k -- written here in the transposed form
  T = S^T stored [d_k][d_v]:  T' = g T + k u^T,  u = beta (v - (g T)^T k),
  o = T'^T q  (article section "为什么线性注意力模型的投机解码更难": the state
  rolls every token and the update is sequential);
* the causal depthwise conv window along the root-to-node path, so siblings
  never see each other's inputs (README "How it works", ggml_ssm_conv_tree;
  article section "状态驻留验证", ggml_ssm_conv_specla);
* tree verification as ONE FULL REPLAY PER NODE from the committed state along
  that node's root path -- no memoisation, no chains, no factor banks;
* commit = append the accepted path's raw rows to the committed history; the
  committed state is the replay of that history (article section "延迟融合提交":
  the deferred fold is exact, so the state after commit-then-verify must be
  the state of the concatenated sequence);
* the heavy-light decomposition the article specifies in words (section
  "链分解与依赖波 HLD 调度": heavy child = largest subtree, heavy edges continue
  a chain, light edges start one, only boundary states are materialised, chains
  grouped into dependency waves), with the tie-breaks read as below;
* the DFS-to-path compaction of a factor bank (section "接受因子缓存").

Readings where the pages are silent (each also listed in the design notes):
state orientation T = S^T; conv tap j of K multiplies the j-th oldest row of
the K-row window (the last tap multiplies the current token); no conv bias;
optional SiLU after the conv; q, k normalised as y / sqrt(sum y^2 + eps) after
the activation, then q scaled by q_scale; v-head h reads k-head floor(h / R);
channel order [q | k | v], head-major; HLD ties go to the smaller node index;
chains are ordered by (wave, head index); boundary slots by node index.

Every function here is pinned by tests/test_oracle_pins.py and
tests/test_hld_oracle.py against closed forms, library routines, invariants,
brute force and hand-derived fixtures -- none is "parity unpinned".
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

DTYPE_F32 = 0
DTYPE_BF16 = 1


class InvalidTree(ValueError):
    pass


class InvalidPath(ValueError):
    pass


@dataclasses.dataclass(frozen=True)
class Dims:
    Hk: int
    Hv: int
    dk: int
    dv: int
    K: int
    conv_mode: int = 1     # 0: bypass (y = x); 1: causal depthwise conv over the K-row window
    act: int = 1           # 0: none; 1: SiLU
    q_scale: float = 1.0
    l2_eps: float = 1e-6

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    @property
    def R(self) -> int:
        return self.Hv // self.Hk


def dims_of(w) -> Dims:
    """Dims of a synthetic.Workload (duck-typed to keep the oracle independent)."""
    return Dims(Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv, K=w.K, conv_mode=w.conv_mode, act=w.act,
                q_scale=w.q_scale, l2_eps=w.l2_eps)


def as_f64(a, in_dtype: int) -> np.ndarray:
    """Exact upcast of the stored input values (bf16 bit patterns or fp32) to float64."""
    a = np.asarray(a)
    if in_dtype == DTYPE_BF16:
        return (a.astype(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# one token step  sigma(T, W; x, beta, a)
# ----------------------------------------------------------------------------

def conv_window(W: np.ndarray, x: np.ndarray, conv_w: np.ndarray) -> np.ndarray:
    """Depthwise causal conv of one token: y[c] = sum_j conv_w[c, j] * X[j, c], X = [W; x] (K rows, oldest first)."""
    X = np.vstack([W, x[None, :]])
    K = X.shape[0]
    y = np.zeros(X.shape[1])
    for j in range(K):
        y += conv_w[:, j] * X[j]
    return y


def silu(y: np.ndarray) -> np.ndarray:
    return y / (1.0 + np.exp(-y))


def l2_normalise(v: np.ndarray, eps: float) -> np.ndarray:
    """Rows of v divided by sqrt(sum of squares + eps)."""
    return v / np.sqrt((v * v).sum(axis=-1, keepdims=True) + eps)


def project(W: np.ndarray, x: np.ndarray, conv_w: Optional[np.ndarray], d: Dims):
    """conv (or bypass), activation, split into q/k/v heads, L2-normalise q and k."""
    y = conv_window(W, x, conv_w) if d.conv_mode == 1 else x.copy()
    if d.act == 1:
        y = silu(y)
    nq = d.Hk * d.dk
    q = y[:nq].reshape(d.Hk, d.dk)
    k = y[nq:2 * nq].reshape(d.Hk, d.dk)
    v = y[2 * nq:].reshape(d.Hv, d.dv)
    q_hat = l2_normalise(q, d.l2_eps) * d.q_scale
    k_hat = l2_normalise(k, d.l2_eps)
    return q_hat, k_hat, v


def delta_rule(T: np.ndarray, q_hat: np.ndarray, k_hat: np.ndarray, v: np.ndarray,
               beta: np.ndarray, log_g: np.ndarray, d: Dims):
    """Gated delta rule for all v-heads.  T [Hv, dk, dv] (T = S^T).

    Per v-head h with k-head kh = h // R:  g = exp(a_h);  T <- g T;
    p = T^T k;  u = beta_h (v_h - p);  T <- T + k u^T;  o = T^T q.
    Returns (T', o [Hv, dv], u [Hv, dv]).
    """
    kh_of = np.arange(d.Hv) // d.R
    kk = k_hat[kh_of]                                  # [Hv, dk]
    qq = q_hat[kh_of]
    g = np.exp(log_g)
    T = g[:, None, None] * T
    p = np.einsum('hij,hi->hj', T, kk)
    u = beta[:, None] * (v - p)
    T = T + kk[:, :, None] * u[:, None, :]
    o = np.einsum('hij,hi->hj', T, qq)
    return T, o, u


def token_step(T: np.ndarray, W: np.ndarray, x: np.ndarray, beta: np.ndarray, log_g: np.ndarray,
               conv_w: Optional[np.ndarray], d: Dims):
    """sigma: one token through one GDN layer.  All arguments fp64.

    Returns (T', W', o, k_hat, u).  W is the committed raw-input window
    [K-1, C]; in bypass mode it is carried unchanged.
    """
    q_hat, k_hat, v = project(W, x, conv_w, d)
    T2, o, u = delta_rule(T, q_hat, k_hat, v, beta, log_g, d)
    if d.conv_mode == 1:
        W2 = np.vstack([W, x[None, :]])[1:]
    else:
        W2 = W
    return T2, W2, o, k_hat, u


def replay(T: np.ndarray, W: np.ndarray, rows, conv_w, d: Dims):
    """Apply sigma to a sequence of (x, beta, log_g) rows in order."""
    for x, beta, log_g in rows:
        T, W, _, _, _ = token_step(T, W, x, beta, log_g, conv_w, d)
    return T, W


# ----------------------------------------------------------------------------
# trees
# ----------------------------------------------------------------------------

def check_tree(parent: Sequence[int]) -> List[int]:
    p = [int(v) for v in parent]
    n = len(p)
    if n < 1 or p[0] != -1:
        raise InvalidTree("node 0 must be the root (parent -1)")
    for i in range(1, n):
        if not (0 <= p[i] < i):
            raise InvalidTree(f"parent[{i}] = {p[i]} is not an earlier node")
    return p


def root_path(parent: Sequence[int], node: int) -> List[int]:
    path = [node]
    while parent[path[-1]] != -1:
        path.append(int(parent[path[-1]]))
    return path[::-1]


def hld_schedule(parent: Sequence[int]) -> Dict[str, object]:
    """Heavy-light decomposition of a draft tree into chains and dependency waves.

    Rules (article section "链分解与依赖波 HLD 调度", with the tie-breaks read
    here): subtree sizes; heavy child = the child with the largest subtree,
    ties to the smallest index; chain heads = the root and every child that is
    not its parent's heavy child; a chain runs head -> heavy -> heavy ... to a
    leaf; wave of the root chain = 0, of any other chain = wave of the chain
    holding its head's parent + 1; chains ordered by (wave, head); boundary
    nodes = parents of non-root heads, slots in ascending node index; a chain's
    source slot is its head's parent's slot (-1 for the root chain).
    """
    p = check_tree(parent)
    n = len(p)
    children = [[] for _ in range(n)]
    for i in range(1, n):
        children[p[i]].append(i)
    subtree = [1] * n
    for i in range(n - 1, 0, -1):
        subtree[p[i]] += subtree[i]
    heavy = [-1] * n
    for v in range(n):
        for c in children[v]:
            if heavy[v] == -1 or subtree[c] > subtree[heavy[v]]:
                heavy[v] = c
    heads = [0] + [c for c in range(1, n) if heavy[p[c]] != c]
    members = {}
    head_of = [-1] * n
    pos = [-1] * n
    for h in heads:
        nodes = [h]
        while heavy[nodes[-1]] != -1:
            nodes.append(heavy[nodes[-1]])
        members[h] = nodes
        for i, v in enumerate(nodes):
            head_of[v] = h
            pos[v] = i
    wave_of_head = {}
    for h in sorted(heads):
        wave_of_head[h] = 0 if h == 0 else wave_of_head[head_of[p[h]]] + 1
    order = sorted(heads, key=lambda h: (wave_of_head[h], h))
    bnodes = sorted({p[h] for h in heads if h != 0})
    slot_of = {b: s for s, b in enumerate(bnodes)}
    n_waves = max(wave_of_head.values()) + 1
    chain_id = {h: i for i, h in enumerate(order)}
    chain_off = [0]
    chain_nodes: List[int] = []
    for h in order:
        chain_nodes += members[h]
        chain_off.append(len(chain_nodes))
    wave_off = [0] * (n_waves + 1)
    for h in order:
        wave_off[wave_of_head[h] + 1] += 1
    for w in range(n_waves):
        wave_off[w + 1] += wave_off[w]
    return dict(
        n=n, n_chains=len(order), n_waves=n_waves, n_boundary=len(bnodes),
        heavy=heavy, subtree=subtree,
        chain_of=[chain_id[head_of[v]] for v in range(n)], pos_in_chain=pos,
        chain_head=list(order), chain_len=[len(members[h]) for h in order],
        chain_off=chain_off, chain_nodes=chain_nodes,
        chain_wave=[wave_of_head[h] for h in order],
        chain_src_slot=[-1 if h == 0 else slot_of[p[h]] for h in order],
        wave_off=wave_off,
        boundary_slot=[slot_of.get(v, -1) for v in range(n)],
        boundary_node=bnodes,
    )


def check_path(parent: Sequence[int], path: Sequence[int]) -> List[int]:
    """A committed path is a root path: path[0] = 0, parent[path[i]] = path[i-1], 0 <= L <= n."""
    path = [int(v) for v in path]
    n = len(parent)
    if len(path) > n:
        raise InvalidPath("longer than the tree")
    if not path:
        return path
    if path[0] != 0:
        raise InvalidPath("does not start at the root")
    for i in range(1, len(path)):
        if not (0 <= path[i] < n) or int(parent[path[i]]) != path[i - 1]:
            raise InvalidPath(f"step {i} is not a child of step {i - 1}")
    return path


def is_zero_copy(path: Sequence[int]) -> bool:
    """Chain acceptance: the accepted nodes already sit at slots 0..L-1."""
    return all(int(v) == i for i, v in enumerate(path))


def compact(bank: np.ndarray, path: Sequence[int]) -> np.ndarray:
    """DFS-to-path compaction of one bank field [n_slots, ...]: slot i <- slot path[i] for i < L."""
    out = bank.copy()
    for i, src in enumerate(path):
        out[i] = bank[int(src)]
    return out


# ----------------------------------------------------------------------------
# verification of one tree for one (request, layer)
# ----------------------------------------------------------------------------

def verify_tree(T: np.ndarray, W: np.ndarray, parent: Sequence[int], X: np.ndarray, BETA: np.ndarray,
                LOGG: np.ndarray, conv_w: Optional[np.ndarray], d: Dims,
                boundary_nodes: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Verify every node of one tree by replaying its root path from (T, W).

    T [Hv, dk, dv], W [K-1, C], X [n, C], BETA/LOGG [n, Hv] all fp64.
    Returns o [n, Hv, dv]; the factors of each node k [n, Hk, dk], u [n, Hv, dv],
    a [n, Hv], x [n, C]; and the state after each boundary node
    boundary [len(boundary_nodes), Hv, dk, dv].
    """
    p = check_tree(parent)
    n = len(p)
    if boundary_nodes is None:
        boundary_nodes = hld_schedule(p)["boundary_node"]
    slot = {int(b): s for s, b in enumerate(boundary_nodes)}
    o = np.zeros((n, d.Hv, d.dv))
    kf = np.zeros((n, d.Hk, d.dk))
    uf = np.zeros((n, d.Hv, d.dv))
    bst = np.zeros((len(boundary_nodes), d.Hv, d.dk, d.dv))
    for node in range(n):
        Tn, Wn = T.copy(), W.copy()
        for m in root_path(p, node):
            Tn, Wn, on, kn, un = token_step(Tn, Wn, X[m], BETA[m], LOGG[m], conv_w, d)
        o[node], kf[node], uf[node] = on, kn, un
        if node in slot:
            bst[slot[node]] = Tn
    return dict(o=o, k=kf, u=uf, a=LOGG[:n].copy(), x=X[:n].copy(), boundary=bst)


class Session:
    """Committed history of one (request, layer) across verify -> commit steps.

    The committed state is the replay of every committed row from the initial
    (T, W); a verify replays each node's root path from that state; commit
    appends the accepted path's raw rows; finish returns the committed state.
    """

    def __init__(self, T0: np.ndarray, W0: np.ndarray, conv_w: Optional[np.ndarray], d: Dims):
        self.d = d
        self.conv_w = None if conv_w is None else np.asarray(conv_w, np.float64)
        self.T = np.asarray(T0, np.float64).copy()
        self.W = np.asarray(W0, np.float64).copy()
        self.history_len = 0

    def verify(self, parent, X, BETA, LOGG, boundary_nodes=None):
        return verify_tree(self.T, self.W, parent, X, BETA, LOGG, self.conv_w, self.d, boundary_nodes)

    def commit(self, parent, path, X, BETA, LOGG):
        path = check_path(parent, path)
        rows = [(X[m], BETA[m], LOGG[m]) for m in path]
        self.T, self.W = replay(self.T, self.W, rows, self.conv_w, self.d)
        self.history_len += len(rows)
        return path

    def committed(self):
        return self.T.copy(), self.W.copy()
