"""Oracle side of the GPU parity tests: expected values per (request, layer) unit and the tolerances.

Tolerances (fixed by the method's accuracy statement for this build): outputs
max |o_gpu - o_ref| <= 1e-3 * max |o_ref|; states (committed, boundary, after
finish) relative Frobenius error <= 1e-5 per head; the factor bank's log-gate
and raw input are exact copies (bitwise); its keys and update vectors are fp32
results held to max error <= 1e-5 (unit-norm keys) and 1e-4 * max |u_ref|.
"""
from __future__ import annotations

import numpy as np

import synthetic as S
from oracle import gdn_oracle as O

O_TOL = 1e-3
STATE_TOL = 1e-5
K_TOL = 1e-5
U_TOL = 1e-4


def unit_inputs(w, b, l, step, n):
    x, be, ag = S.node_inputs(w, b, l, step)
    return (O.as_f64(x[:n], w.in_dtype), O.as_f64(be[:n], w.in_dtype), O.as_f64(ag[:n], w.in_dtype))


class OracleUnit:
    """Oracle replay of one (request, layer) across the steps of a plan."""

    def __init__(self, w, plan, b, l):
        self.w, self.plan, self.b, self.l = w, plan, b, l
        self.d = O.dims_of(w)
        cw = S.conv_weight(w, l).astype(np.float64) if w.conv_mode == 1 else None
        self.sess = O.Session(S.init_state(w, b, l).astype(np.float64),
                              S.init_conv_state(w, b, l).astype(np.float64), cw, self.d)

    def verify(self, step):
        parent = self.plan.trees[step][self.b]
        n = len(parent)
        X, BE, AG = unit_inputs(self.w, self.b, self.l, step, n)
        sched = O.hld_schedule(parent)
        if getattr(self.plan, "per_node", False):
            # per-node-state schedule: every node with children is materialised, slots in node order
            internal = sorted({int(v) for v in parent[1:]})
            sched = dict(sched, boundary_node=internal, n_boundary=len(internal))
        exp = self.sess.verify(parent, X, BE, AG, sched["boundary_node"])
        exp["T"], exp["W"] = self.sess.committed()
        exp["n"], exp["sched"] = n, sched
        self._rows = (parent, X, BE, AG)
        return exp

    def commit(self, step, path=None):
        parent, X, BE, AG = self._rows
        path = self.plan.paths[step][self.b] if path is None else path
        self.sess.commit(parent, path, X, BE, AG)

    def committed(self):
        return self.sess.committed()


def rel_frob(got, ref, axes):
    num = np.sqrt(((got - ref) ** 2).sum(axis=axes))
    den = np.sqrt((ref ** 2).sum(axis=axes))
    return num / np.maximum(den, 1e-300)


def check_o(got, ref, what="o"):
    err = np.abs(got - ref).max() if ref.size else 0.0
    scale = np.abs(ref).max() if ref.size else 1.0
    assert err <= O_TOL * scale, f"{what}: max err {err:.3e} > {O_TOL} * {scale:.3e}"
    return err / max(scale, 1e-300)


def check_state(got, ref, what="state"):
    """got/ref [..., Hv, dk, dv]: relative Frobenius error per head."""
    if ref.size == 0:
        return 0.0
    e = rel_frob(got, ref, axes=(-2, -1))
    assert e.max() <= STATE_TOL, f"{what}: rel Frobenius {e.max():.3e} > {STATE_TOL}"
    return float(e.max())


def check_factors(gpu_k, gpu_u, gpu_a, gpu_x, exp, conv_mode):
    n = exp["n"]
    ek = np.abs(gpu_k[:n] - exp["k"]).max()
    assert ek <= K_TOL, f"bank k: max err {ek:.3e}"
    eu = np.abs(gpu_u[:n] - exp["u"]).max()
    su = np.abs(exp["u"]).max()
    assert eu <= U_TOL * su, f"bank u: max err {eu:.3e} > {U_TOL} * {su:.3e}"
    np.testing.assert_array_equal(gpu_a[:n].astype(np.float64), exp["a"], err_msg="bank a not bitwise")
    if conv_mode == 1:
        np.testing.assert_array_equal(gpu_x[:n].astype(np.float64), exp["x"], err_msg="bank x not bitwise")
