"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a closed form of the gated delta rule, the
rule as printed (S' = g S (I - beta k k^T) + beta v k^T, o = S' q), a library
routine (numpy convolve / norm, scipy expit / linear solve), a structural
invariant the pages state (chain == sequential, sibling isolation, exact
deferred commit), or a hand-derived fixture under tests/golden/.  A plausible
slip in the oracle -- a dropped gate, a wrong sign, a transposed state, a wrong
tap order, a wrong GQA map, a sibling leaking into the window -- fails one of
them.
"""
import dataclasses
import itertools
import os

import numpy as np
import pytest
import scipy.special

from oracle import gdn_oracle as O
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(*k):
    return np.random.default_rng(list(k))


def _rand_inputs(d, n, rng, scale_state=0.3):
    T = rng.normal(0, scale_state, (d.Hv, d.dk, d.dv))
    W = rng.normal(0, 1, (d.K - 1, d.C))
    X = rng.normal(0, 1, (n, d.C))
    BETA = rng.uniform(0, 1, (n, d.Hv))
    LOGG = rng.uniform(-1, 0, (n, d.Hv))
    cw = rng.normal(0, 0.5, (d.C, d.K))
    return T, W, X, BETA, LOGG, cw


# ---------------------------------------------------------------------------
# delta rule: closed forms
# ---------------------------------------------------------------------------

D_SMALL = O.Dims(Hk=2, Hv=4, dk=5, dv=7, K=4, conv_mode=0, act=0)


def _qkv(d, rng):
    q = O.l2_normalise(rng.normal(size=(d.Hk, d.dk)), 0.0)
    k = O.l2_normalise(rng.normal(size=(d.Hk, d.dk)), 0.0)
    v = rng.normal(size=(d.Hv, d.dv))
    return q, k, v


def test_beta_zero_is_pure_decay():
    d, rng = D_SMALL, _rng(1)
    T = rng.normal(size=(d.Hv, d.dk, d.dv))
    q, k, v = _qkv(d, rng)
    a = rng.uniform(-2, 0, d.Hv)
    T2, o, u = O.delta_rule(T, q, k, v, np.zeros(d.Hv), a, d)
    g = np.exp(a)
    np.testing.assert_allclose(T2, g[:, None, None] * T, rtol=0, atol=1e-14)
    np.testing.assert_allclose(u, 0.0, atol=0)
    for h in range(d.Hv):
        np.testing.assert_allclose(o[h], g[h] * T[h].T @ q[h // d.R], atol=1e-13)


def test_identity_when_no_decay_and_no_write():
    d, rng = D_SMALL, _rng(2)
    T = rng.normal(size=(d.Hv, d.dk, d.dv))
    q, k, v = _qkv(d, rng)
    T2, o, u = O.delta_rule(T, q, k, v, np.zeros(d.Hv), np.zeros(d.Hv), d)
    np.testing.assert_array_equal(T2, T)


def test_full_forget_writes_only_the_new_pair():
    # g = 0 (a -> -inf): S' = beta v k^T, i.e. T' = beta k v^T
    d, rng = D_SMALL, _rng(3)
    T = rng.normal(size=(d.Hv, d.dk, d.dv))
    q, k, v = _qkv(d, rng)
    beta = rng.uniform(0, 1, d.Hv)
    T2, o, u = O.delta_rule(T, q, k, v, beta, np.full(d.Hv, -np.inf), d)
    for h in range(d.Hv):
        np.testing.assert_allclose(T2[h], beta[h] * np.outer(k[h // d.R], v[h]), atol=1e-14)


def test_delta_write_property():
    # beta = 1, |k| = 1: the new state maps k exactly to v, whatever g and S
    d, rng = D_SMALL, _rng(4)
    T = rng.normal(size=(d.Hv, d.dk, d.dv))
    q, k, v = _qkv(d, rng)
    a = rng.uniform(-3, 0, d.Hv)
    T2, _, _ = O.delta_rule(T, q, k, v, np.ones(d.Hv), a, d)
    for h in range(d.Hv):
        np.testing.assert_allclose(T2[h].T @ k[h // d.R], v[h], atol=1e-12)


def test_orthonormal_keys_store_every_pair():
    # beta = 1, g = 1, orthonormal keys: S k_i = v_i for every pair written
    d = O.Dims(Hk=1, Hv=1, dk=6, dv=3, K=1, conv_mode=0, act=0)
    rng = _rng(5)
    Q, _ = np.linalg.qr(rng.normal(size=(6, 6)))
    T = rng.normal(size=(1, 6, 3))
    vs = rng.normal(size=(6, 3))
    for i in range(6):
        T, _, _ = O.delta_rule(T, Q[:, i][None], Q[:, i][None], vs[i][None], np.ones(1), np.zeros(1), d)
    for i in range(6):
        np.testing.assert_allclose(T[0].T @ Q[:, i], vs[i], atol=1e-12)


def test_matches_printed_rule_in_S_form():
    """S' = g S (I - beta k k^T) + beta v k^T, o = S' q, with S = T^T (d_v x d_k), GQA h -> h // R."""
    d, rng = D_SMALL, _rng(6)
    T = rng.normal(size=(d.Hv, d.dk, d.dv))
    q, k, v = _qkv(d, rng)
    beta = rng.uniform(0, 1, d.Hv)
    a = rng.uniform(-1, 0, d.Hv)
    T2, o, _ = O.delta_rule(T, q, k, v, beta, a, d)
    for h in range(d.Hv):
        S = T[h].T
        kk, qq = k[h // d.R], q[h // d.R]
        S2 = np.exp(a[h]) * S @ (np.eye(d.dk) - beta[h] * np.outer(kk, kk)) + beta[h] * np.outer(v[h], kk)
        np.testing.assert_allclose(T2[h], S2.T, atol=1e-13)
        np.testing.assert_allclose(o[h], S2 @ qq, atol=1e-13)


def test_hand_fixture_delta_rule():
    """Values worked out by hand on a 2x2 head (tests/golden/delta_rule_2x2.txt)."""
    fx = _read_fixture("delta_rule_2x2.txt")
    d = O.Dims(Hk=1, Hv=1, dk=2, dv=2, K=1, conv_mode=0, act=0, l2_eps=0.0)
    x = np.array(fx["q"] + fx["k"] + fx["v"], dtype=float)
    T0 = np.array(fx["T0"], dtype=float).reshape(1, 2, 2)
    T1, _, o, kh, u = O.token_step(T0, np.zeros((0, d.C)), x, np.array(fx["beta"]), np.array(fx["a"]), None, d)
    np.testing.assert_allclose(u[0], fx["u"], atol=1e-15)
    np.testing.assert_allclose(T1[0].ravel(), fx["T1"], atol=1e-15)
    np.testing.assert_allclose(o[0], fx["o"], atol=1e-15)


# ---------------------------------------------------------------------------
# projections: conv, activation, normalisation, head split
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", [1, 2, 3, 4, 8])
def test_conv_window_is_causal_convolution(K):
    # along a sequence, y_t = sum_j w[j] X[t-K+1+j]  ==  np.convolve(seq, w[::-1]) at position t
    rng = _rng(7)
    C, L = 5, 9
    w = rng.normal(size=(C, K))
    seq = rng.normal(size=(K - 1 + L, C))
    for t in range(L):
        y = O.conv_window(seq[t:t + K - 1], seq[t + K - 1], w)
        for c in range(C):
            ref = np.convolve(seq[:, c], w[c, ::-1], mode="valid")[t]
            assert abs(y[c] - ref) < 1e-12


def test_silu_and_l2_against_library():
    rng = _rng(8)
    y = rng.normal(0, 3, 1000)
    np.testing.assert_allclose(O.silu(y), y * scipy.special.expit(y), rtol=1e-14, atol=1e-300)
    v = rng.normal(size=(7, 13))
    np.testing.assert_allclose(O.l2_normalise(v, 0.0), v / np.linalg.norm(v, axis=1, keepdims=True), rtol=1e-14)
    e = 1e-6
    np.testing.assert_allclose(O.l2_normalise(v, e), v / np.sqrt(np.linalg.norm(v, axis=1, keepdims=True) ** 2 + e),
                               rtol=1e-14)


def test_head_split_and_gqa_map():
    # a one-hot input channel must land in the q / k / v head it belongs to
    d = O.Dims(Hk=2, Hv=6, dk=3, dv=4, K=1, conv_mode=0, act=0, l2_eps=1e-6)
    nq = d.Hk * d.dk
    x = np.zeros(d.C)
    x[1 * d.dk + 2] = 1.0                 # q head 1, element 2
    x[nq + 0 * d.dk + 1] = 1.0            # k head 0, element 1
    x[2 * nq + 4 * d.dv + 3] = 5.0        # v head 4, element 3
    q, k, v = O.project(np.zeros((0, d.C)), x, None, d)
    assert q[1, 2] > 0.999 and np.count_nonzero(q) == 1
    assert k[0, 1] > 0.999 and np.count_nonzero(k) == 1
    assert v[4, 3] == 5.0 and np.count_nonzero(v) == 1
    # v-heads 0..2 read k-head 0 and 3..5 read k-head 1: with beta=1, g=1, T=0 only heads 0..2 get written
    T, o, u = O.delta_rule(np.zeros((d.Hv, d.dk, d.dv)), q, k, v + 1.0, np.ones(d.Hv), np.zeros(d.Hv), d)
    assert np.all(T[:3, 1, :] != 0) and np.all(T[:3, [0, 2], :] == 0)
    assert np.all(T[3:] == 0)


def test_bf16_decode_against_torch_and_by_hand():
    """as_f64 on bf16 bit patterns equals torch's bfloat16 -> float64 conversion on random patterns and on
    the special values (+-0, subnormals, the extreme normals, +-inf); a few patterns are decoded by hand from
    the format (1 sign, 8 exponent bits with bias 127, 7 fraction bits)."""
    import torch
    rng = _rng(30)
    bits = rng.integers(0, 1 << 16, 20000, dtype=np.uint32).astype(np.uint16)
    special = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80,
                        0x3F80, 0xC000, 0x3E80, 0x4049], dtype=np.uint16)
    allbits = np.concatenate([bits, special])
    finite = (allbits & 0x7F80) != 0x7F80
    finite |= (allbits & 0x7F) == 0            # keep +-inf, drop NaN patterns (NaN != NaN)
    allbits = allbits[finite]
    ref = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.as_f64(allbits, O.DTYPE_BF16)
    np.testing.assert_array_equal(got, ref)
    assert np.signbit(O.as_f64(np.array([0x8000], np.uint16), O.DTYPE_BF16)[0])
    hand = {0x3F80: 1.0, 0xC000: -2.0, 0x3E80: 0.25, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
            0x0080: 2.0 ** -126, 0x7F7F: (2.0 - 2.0 ** -7) * 2.0 ** 127, 0xFF80: -np.inf}
    for b, v in hand.items():
        assert O.as_f64(np.array([b], np.uint16), O.DTYPE_BF16)[0] == v, hex(b)
    # fp32 inputs are upcast unchanged
    x = rng.normal(size=100).astype(np.float32)
    np.testing.assert_array_equal(O.as_f64(x, O.DTYPE_F32), x.astype(np.float64))


@pytest.mark.parametrize("conv_mode", [0, 1])
def test_q_scale_multiplies_the_output_only(conv_mode):
    """The printed rule gives o = S' q_hat; a query scale s multiplies the normalised q, so o(s) = s o(1)
    while u, k_hat and every state are unchanged.  A scale applied before the L2 normalisation would cancel
    (o(s) = o(1)) and fails this."""
    import dataclasses
    d1 = O.Dims(Hk=2, Hv=4, dk=4, dv=6, K=4, conv_mode=conv_mode, act=1)
    rng = _rng(31)
    parent = np.array([-1, 0, 1, 1, 0, 4], dtype=np.int32)
    T, W, X, BETA, LOGG, cw = _rand_inputs(d1, len(parent), rng)
    base = O.verify_tree(T, W, parent, X, BETA, LOGG, cw, d1)
    for s in (0.5, 1.0 / np.sqrt(d1.dk), 3.0):
        ds = dataclasses.replace(d1, q_scale=s)
        r = O.verify_tree(T, W, parent, X, BETA, LOGG, cw, ds)
        np.testing.assert_allclose(r["o"], s * base["o"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["u"], base["u"], rtol=0, atol=0)
        np.testing.assert_allclose(r["k"], base["k"], rtol=0, atol=0)
        np.testing.assert_allclose(r["boundary"], base["boundary"], rtol=0, atol=0)
        assert not np.allclose(r["o"], base["o"])
    # one token by hand: with T = 0, beta = 1, g = 1: T' = k v^T, so o = s (k_hat . q_hat) v
    d = O.Dims(Hk=1, Hv=1, dk=2, dv=2, K=1, conv_mode=0, act=0, l2_eps=0.0, q_scale=0.25)
    x = np.array([3.0, 4.0, 1.0, 0.0, 2.0, -1.0])          # q = (3, 4), k = (1, 0), v = (2, -1)
    _, _, o, _, _ = O.token_step(np.zeros((1, 2, 2)), np.zeros((0, 6)), x, np.ones(1), np.zeros(1), None, d)
    np.testing.assert_allclose(o[0], 0.25 * (3.0 / 5.0) * np.array([2.0, -1.0]), atol=1e-15)


def test_edge_recipes_reach_the_degenerate_cases():
    """The seeded edge-case inputs the GPU parity tests use do what they are named for, and the oracle's
    results on them keep the closed forms: g = 0 forgets the state, beta = 0 writes nothing, an all-zero
    row (bypass mode) has q_hat = k_hat = 0 so its o is 0 and its u is beta v."""
    w = S.workload(1).replace(Hk=2, Hv=6, conv_mode=0, act=0, edge="gate_zero+beta01+zero_rows", budget=8)
    x, be, ag = (O.as_f64(a, w.in_dtype) for a in S.node_inputs(w, 0, 0, 0))
    assert np.isneginf(ag[1, 0]) and np.isfinite(ag[1, 1]) and np.isneginf(ag[4, 2])
    assert np.all(be[1::2] == 0) and np.all(be[0::2] == 1) and np.all(x[2::3] == 0)
    d = O.dims_of(w)
    parent = np.arange(-1, 7, dtype=np.int32)              # a chain
    T0 = S.init_state(w, 0, 0).astype(np.float64)
    r = O.verify_tree(T0, np.zeros((w.K - 1, w.C)), parent, x, be, ag, None, d)
    assert np.all(np.isfinite(r["o"])) and np.all(np.isfinite(r["u"]))
    np.testing.assert_array_equal(r["o"][2], 0.0)          # zero row: q_hat = 0
    np.testing.assert_allclose(r["u"][2], be[2][:, None] * x[2, 2 * w.Hk * w.dk:].reshape(w.Hv, w.dv), atol=0)
    np.testing.assert_array_equal(r["u"][1], 0.0)          # beta = 0 on node 1
    # node 1 forgets the even heads' state: the state after node 1 is beta k v^T = 0 there (beta = 0)
    Tn, Wn = T0.copy(), np.zeros((w.K - 1, w.C))
    for m in (0, 1):
        Tn, Wn, _, _, _ = O.token_step(Tn, Wn, x[m], be[m], ag[m], None, d)
    np.testing.assert_array_equal(Tn[0::2], 0.0)
    wf = S.workload(1).replace(edge="gate_floor", Hk=2, Hv=6)
    _, _, agf = S.node_inputs(wf, 0, 0, 0)
    assert np.all(agf[:, 1::3] == -14.0) and np.exp(-28.0) < 1e-12
    wz = S.workload(1).replace(edge="zero_rows", Hk=2, Hv=6)
    cwz = S.conv_weight(wz, 0)
    assert np.all(cwz[wz.Hk * wz.dk:wz.Hk * wz.dk + wz.dk] == 0) and np.any(cwz[wz.Hk * wz.dk + wz.dk:] != 0)


# ---------------------------------------------------------------------------
# tree semantics
# ---------------------------------------------------------------------------

D_CONV = O.Dims(Hk=2, Hv=4, dk=4, dv=6, K=4, conv_mode=1, act=1)


def _sequential_gdn(T, W, X, BETA, LOGG, cw, d):
    """Plain sequential GDN over a token sequence written from the printed rule (S form) and np.convolve."""
    L = X.shape[0]
    seq = np.vstack([W, X])
    nq = d.Hk * d.dk
    S_ = [T[h].T.copy() for h in range(d.Hv)]
    outs = []
    for t in range(L):
        y = np.array([np.convolve(seq[:, c], cw[c, ::-1], mode="valid")[t] for c in range(d.C)])
        y = y * scipy.special.expit(y)
        q = y[:nq].reshape(d.Hk, d.dk)
        k = y[nq:2 * nq].reshape(d.Hk, d.dk)
        v = y[2 * nq:].reshape(d.Hv, d.dv)
        o_t = np.zeros((d.Hv, d.dv))
        for h in range(d.Hv):
            qq = q[h // d.R] / np.sqrt(q[h // d.R] @ q[h // d.R] + d.l2_eps)
            kk = k[h // d.R] / np.sqrt(k[h // d.R] @ k[h // d.R] + d.l2_eps)
            b, g = BETA[t, h], np.exp(LOGG[t, h])
            S_[h] = g * S_[h] @ (np.eye(d.dk) - b * np.outer(kk, kk)) + b * np.outer(v[h], kk)
            o_t[h] = S_[h] @ qq
        outs.append(o_t)
    return np.array(outs), np.array([s.T for s in S_])


@pytest.mark.parametrize("K", [1, 2, 4, 8])
def test_chain_tree_equals_sequential_gdn(K):
    d, rng = dataclasses.replace(D_CONV, K=K), _rng(9)
    n = 7
    T, W, X, BETA, LOGG, cw = _rand_inputs(d, n, rng)
    res = O.verify_tree(T, W, S.chain_tree(n), X, BETA, LOGG, cw, d)
    o_seq, T_seq = _sequential_gdn(T, W, X, BETA, LOGG, cw, d)
    np.testing.assert_allclose(res["o"], o_seq, atol=1e-11)
    # chain acceptance of the whole chain gives the sequential final state
    sess = O.Session(T, W, cw, d)
    sess.commit(S.chain_tree(n), list(range(n)), X, BETA, LOGG)
    Tc, Wc = sess.committed()
    np.testing.assert_allclose(Tc, T_seq, atol=1e-11)
    seq = np.vstack([W, X])
    np.testing.assert_array_equal(Wc, seq[len(seq) - (d.K - 1):])   # the last K-1 raw rows (none for K = 1)


def test_siblings_never_see_each_other():
    d, rng = D_CONV, _rng(10)
    parent = np.array([-1, 0, 0, 1, 2, 2, 3, 1], dtype=np.int32)
    n = len(parent)
    T, W, X, BETA, LOGG, cw = _rand_inputs(d, n, rng)
    base = O.verify_tree(T, W, parent, X, BETA, LOGG, cw, d)
    for m in range(n):
        X2, B2, G2 = X.copy(), BETA.copy(), LOGG.copy()
        X2[m] += rng.normal(size=d.C)
        B2[m] = rng.uniform(0, 1, d.Hv)
        G2[m] = rng.uniform(-1, 0, d.Hv)
        pert = O.verify_tree(T, W, parent, X2, B2, G2, cw, d)
        for node in range(n):
            anc = set(O.root_path(parent, node))
            if m in anc:
                assert np.abs(pert["o"][node] - base["o"][node]).max() > 1e-9
            else:
                np.testing.assert_array_equal(pert["o"][node], base["o"][node])


def test_commit_then_verify_equals_concatenated_path():
    d, rng = D_CONV, _rng(11)
    p1 = np.array([-1, 0, 1, 1, 2, 0, 5], dtype=np.int32)
    path = [0, 1, 2, 4]
    p2 = np.array([-1, 0, 0, 1, 2, 2], dtype=np.int32)
    T, W, X1, B1, G1, cw = _rand_inputs(d, len(p1), rng)
    _, _, X2, B2, G2, _ = _rand_inputs(d, len(p2), rng)
    sess = O.Session(T, W, cw, d)
    sess.verify(p1, X1, B1, G1)
    sess.commit(p1, path, X1, B1, G1)
    r2 = sess.verify(p2, X2, B2, G2)
    # one tree: the accepted path as a chain with tree 2 hung under its last node
    L = len(path)
    parent = [-1] + [i - 1 for i in range(1, L)] + [(L + int(p)) if p >= 0 else L - 1 for p in p2]
    Xc = np.vstack([X1[path], X2])
    Bc = np.vstack([B1[path], B2])
    Gc = np.vstack([G1[path], G2])
    rc = O.verify_tree(T, W, parent, Xc, Bc, Gc, cw, d)
    np.testing.assert_allclose(r2["o"], rc["o"][L:], atol=1e-11)
    # and the committed state is the state the first verify reached at the path's last node
    Tn = T.copy(); Wn = W.copy()
    for m in path:
        Tn, Wn, *_ = O.token_step(Tn, Wn, X1[m], B1[m], G1[m], cw, d)
    Tc, Wc = sess.committed()
    np.testing.assert_array_equal(Tc, Tn)
    np.testing.assert_array_equal(Wc, Wn)


def _ut_form(T0, parent, q, k, v, beta, g):
    """Tree-masked UT form of one head (independent of the per-node replay).

    Gam[n] = product of g over n's root path.  With A[a, c] = beta_a Gam_a / Gam_c (k_a . k_c)
    for c a strict ancestor of a, the residuals solve (I + A) U = beta (V - Gam K T0); then
    o_n = Gam_n T0^T q_n + sum_{a <= n} Gam_n / Gam_a (k_a . q_n) u_a and
    T_n = Gam_n T0 + sum_{a <= n} Gam_n / Gam_a k_a u_a^T.
    """
    n = len(parent)
    anc = [set(O.root_path(parent, i)) for i in range(n)]
    Gam = np.array([np.prod([g[m] for m in O.root_path(parent, i)]) for i in range(n)])
    A = np.zeros((n, n))
    for a in range(n):
        for c in anc[a] - {a}:
            A[a, c] = beta[a] * Gam[a] / Gam[c] * (k[a] @ k[c])
    rhs = beta[:, None] * (v - Gam[:, None] * (k @ T0))
    U = np.linalg.solve(np.eye(n) + A, rhs)
    o = np.zeros((n, T0.shape[1]))
    Ts = np.zeros((n,) + T0.shape)
    for i in range(n):
        o[i] = Gam[i] * (T0.T @ q[i])
        Ts[i] = Gam[i] * T0
        for a in anc[i]:
            o[i] += Gam[i] / Gam[a] * (k[a] @ q[i]) * U[a]
            Ts[i] += Gam[i] / Gam[a] * np.outer(k[a], U[a])
    return o, Ts, U


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7])
def test_every_tree_matches_ut_form(n):
    d = O.Dims(Hk=1, Hv=2, dk=4, dv=5, K=1, conv_mode=0, act=0)
    rng = _rng(12, n)
    T0 = rng.normal(0, 0.5, (d.Hv, d.dk, d.dv))
    X = rng.normal(size=(n, d.C))
    BETA = rng.uniform(0, 1, (n, d.Hv))
    LOGG = rng.uniform(-1, 0, (n, d.Hv))
    q, k, v = [], [], []
    for i in range(n):
        qi, ki, vi = O.project(np.zeros((0, d.C)), X[i], None, d)
        q.append(qi); k.append(ki); v.append(vi)
    q, k, v = np.array(q), np.array(k), np.array(v)
    for parent in S.all_trees(n):
        sched = O.hld_schedule(parent)
        res = O.verify_tree(T0, np.zeros((0, d.C)), parent, X, BETA, LOGG, None, d, sched["boundary_node"])
        for h in range(d.Hv):
            o, Ts, U = _ut_form(T0[h], parent, q[:, 0], k[:, 0], v[:, h], BETA[:, h], np.exp(LOGG[:, h]))
            np.testing.assert_allclose(res["o"][:, h], o, atol=1e-12)
            np.testing.assert_allclose(res["u"][:, h], U, atol=1e-12)
            for s, b in enumerate(sched["boundary_node"]):
                np.testing.assert_allclose(res["boundary"][s, h], Ts[b], atol=1e-12)


def _chunked_chain_form(T0, q, k, v, beta, g, C):
    """Chunked UT/WY form of one head on a chain (independent of the per-node replay): the chain is cut
    into chunks of C nodes; inside a chunk with start state Tj and gates accumulated from the chunk's
    start (Gam), the residuals solve (I + A) U = beta (V - Gam K Tj) with A[t, s] = beta_t Gam_t / Gam_s
    (k_t . k_s) for s < t in the chunk; o_t = Gam_t Tj^T q_t + sum_{s <= t} Gam_t / Gam_s (k_s . q_t) u_s;
    the next chunk starts from Gam_end Tj + sum_s Gam_end / Gam_s k_s u_s^T (a rank-C update)."""
    n = len(q)
    T = T0.copy()
    o = np.zeros((n, T0.shape[1]))
    U = np.zeros((n, T0.shape[1]))
    for c0 in range(0, n, C):
        idx = np.arange(c0, min(n, c0 + C))
        m = len(idx)
        Gam = np.cumprod(g[idx])
        A = np.zeros((m, m))
        for t in range(m):
            for s_ in range(t):
                A[t, s_] = beta[idx[t]] * Gam[t] / Gam[s_] * (k[idx[t]] @ k[idx[s_]])
        rhs = beta[idx, None] * (v[idx] - Gam[:, None] * (k[idx] @ T))
        Uc = np.linalg.solve(np.eye(m) + A, rhs)
        for t in range(m):
            o[idx[t]] = Gam[t] * (T.T @ q[idx[t]])
            for s_ in range(t + 1):
                o[idx[t]] += Gam[t] / Gam[s_] * (k[idx[s_]] @ q[idx[t]]) * Uc[s_]
        U[idx] = Uc
        T = Gam[-1] * T + sum(Gam[-1] / Gam[s_] * np.outer(k[idx[s_]], Uc[s_]) for s_ in range(m))
    return o, U, T


@pytest.mark.parametrize("C", [1, 5, 16, 64])
def test_chain_matches_chunked_ut_form(C):
    # the long-chain stress shape: a 64-node chain, its outputs, residuals and end state against the
    # chunked UT/WY form for chunk sizes that divide it and that leave a ragged last chunk
    n = 64
    d = O.Dims(Hk=1, Hv=2, dk=4, dv=5, K=1, conv_mode=0, act=0)
    rng = _rng(16, C)
    T0 = rng.normal(0, 0.5, (d.Hv, d.dk, d.dv))
    X = rng.normal(size=(n, d.C))
    BETA = rng.uniform(0, 1, (n, d.Hv))
    LOGG = rng.uniform(-1, 0, (n, d.Hv))
    parent = S.chain_tree(n)
    q, k, v = [], [], []
    for i in range(n):
        qi, ki, vi = O.project(np.zeros((0, d.C)), X[i], None, d)
        q.append(qi); k.append(ki); v.append(vi)
    q, k, v = np.array(q), np.array(k), np.array(v)
    res = O.verify_tree(T0, np.zeros((0, d.C)), parent, X, BETA, LOGG, None, d, [n - 1])
    for h in range(d.Hv):
        o, U, T_end = _chunked_chain_form(T0[h], q[:, 0], k[:, 0], v[:, h], BETA[:, h], np.exp(LOGG[:, h]), C)
        np.testing.assert_allclose(res["o"][:, h], o, atol=1e-12)
        np.testing.assert_allclose(res["u"][:, h], U, atol=1e-12)
        np.testing.assert_allclose(res["boundary"][0, h], T_end, atol=1e-12)


def test_factors_replay_the_accepted_path():
    # the factor bank (k, u, a) alone reproduces the committed state: T <- exp(a) T + k u^T
    d, rng = D_CONV, _rng(13)
    parent = np.array([-1, 0, 1, 1, 3, 0, 5, 3], dtype=np.int32)
    T, W, X, BETA, LOGG, cw = _rand_inputs(d, len(parent), rng)
    r = O.verify_tree(T, W, parent, X, BETA, LOGG, cw, d)
    path = [0, 1, 3, 7]
    Tf = T.copy()
    for m in path:
        for h in range(d.Hv):
            Tf[h] = np.exp(r["a"][m, h]) * Tf[h] + np.outer(r["k"][m, h // d.R], r["u"][m, h])
    sess = O.Session(T, W, cw, d)
    sess.commit(parent, path, X, BETA, LOGG)
    np.testing.assert_allclose(Tf, sess.committed()[0], atol=1e-12)
    # the raw rows of the path's last K-1 nodes are the committed conv window
    np.testing.assert_array_equal(sess.committed()[1], X[path[-(d.K - 1):]])


def test_compaction_and_paths():
    parent = np.array([-1, 0, 1, 0, 3, 4, 3], dtype=np.int32)
    bank = np.arange(7 * 3).reshape(7, 3)
    path = O.check_path(parent, [0, 3, 4, 5])
    out = O.compact(bank, path)
    np.testing.assert_array_equal(out[:4], bank[[0, 3, 4, 5]])
    np.testing.assert_array_equal(out[4:], bank[4:])
    assert O.is_zero_copy([0, 1, 2]) and not O.is_zero_copy([0, 3])
    assert O.check_path(parent, []) == []
    for bad in ([1], [0, 4], [0, 3, 6, 5], [0, 1, 2, 3, 4, 5, 6, 0]):
        with pytest.raises(O.InvalidPath):
            O.check_path(parent, bad)


def test_invalid_trees_rejected():
    for bad in ([], [0], [-1, 1], [-1, 0, 3, 1], [-1, -1], [-1, 0, 0, 5]):
        with pytest.raises(O.InvalidTree):
            O.check_tree(bad)


# ---------------------------------------------------------------------------
# golden fixtures
# ---------------------------------------------------------------------------

def _read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = [float(t) for t in val.split()]
    return out
