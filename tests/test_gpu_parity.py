"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every case compares element by element on seeded inputs -- outputs of every
node, boundary states, the factor bank written by the verify, the committed
state and conv window after each fold, and the state after finish -- with the
tolerances of tests/parity.py.  Full-size workloads are compared on sampled
(request, layer) units that the oracle replays across all steps.
"""
import numpy as np
import pytest
import torch

import synthetic as S
from parity import OracleUnit, check_factors, check_o, check_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gated_deltanet_tree_gb300.build import build
    build()
    import harness  # noqa: F401


def _np(t):
    return t.detach().cpu().numpy().astype(np.float64)


# verify kernels: "ut" the default dispatch (the tree-masked UT form, on the tensor cores in the persistent
# kernel where d_v = 128 and n_max <= 32), "tc1" the tensor-core UT form with a CTA per v-head, "simt" the UT
# form on the CUDA cores, "walk" the heavy-light chain walk
KERNELS = ["ut", "tc1", "simt", "walk"]


def set_kernel(plan, kernel):
    assert kernel in KERNELS, kernel
    plan.chain_walk = plan.chain_walk or kernel == "walk"
    plan.ut_simt = plan.ut_simt or kernel == "simt"
    plan.tc_per_head = plan.tc_per_head or kernel == "tc1"
    return plan


def run_parity(w, units=None, compact_steps=(), finish=True, plan=None, layer_ids=None, kernel="ut"):
    """Run every step of workload w on the GPU; compare the chosen units with the oracle.

    layer_ids: the layers one call covers (a layer chunk); units must lie in it.
    kernel: which verify kernel runs (KERNELS).
    """
    from harness import GpuSession, WorkloadPlan
    plan = set_kernel(plan or WorkloadPlan(w), kernel)
    gs = GpuSession(w, plan, layer_ids=layer_ids)
    if units is None:
        units = [(b, l) for b in range(w.B) for l in gs.layer_ids]
    oracles = {u: OracleUnit(w, plan, *u) for u in units}
    worst = dict(o=0.0, state=0.0, boundary=0.0)
    for s in range(w.steps):
        gs.verify(s)
        bank = gs.ver.banks.verified_bank
        torch.cuda.synchronize()
        for (b, lg), ou in oracles.items():
            l = gs.local_layer(lg)
            exp = ou.verify(s)
            n = exp["n"]
            worst["o"] = max(worst["o"], check_o(_np(gs.out_o[b, l, :n]), exp["o"], f"o step {s} unit {(b, l)}"))
            worst["state"] = max(worst["state"], check_state(_np(gs.state[b, l]), exp["T"],
                                                             f"committed state step {s} unit {(b, l)}"))
            if w.conv_mode == 1 and w.K > 1:
                np.testing.assert_allclose(_np(gs.conv_state[b, l]), exp["W"], rtol=0, atol=0,
                                           err_msg=f"conv window step {s} unit {(b, l)}")
            nb = exp["sched"]["n_boundary"]
            worst["boundary"] = max(worst["boundary"], check_state(_np(gs.boundary[b, l, :nb]), exp["boundary"],
                                                                   f"boundary step {s} unit {(b, l)}"))
            xb = _np(gs.ver.bank_view("x", bank)[b, l]) if w.conv_mode == 1 else None
            check_factors(_np(gs.ver.bank_view("k", bank)[b, l]), _np(gs.ver.bank_view("u", bank)[b, l]),
                          _np(gs.ver.bank_view("a", bank)[b, l]), xb, exp, w.conv_mode)
        compact = s in compact_steps
        if compact:
            pre = {f: gs.ver.bank_view(f, bank).clone() for f in (("k", "u", "a", "x") if w.conv_mode else ("k", "u", "a"))}
        gs.commit(s, compact=compact)
        if compact:
            torch.cuda.synchronize()
            for b in range(w.B):
                path = plan.paths[s][b]
                for f, t in pre.items():
                    post = gs.ver.bank_view(f, bank)[b]
                    assert torch.equal(post[:, :len(path)], t[b][:, torch.as_tensor(path, dtype=torch.long, device=t.device)]), f
                    assert torch.equal(post[:, len(path):], t[b][:, len(path):]), f
        for ou in oracles.values():
            ou.commit(s)
        gs.drop_step(s)
    if finish:
        gs.finish()
        torch.cuda.synchronize()
        for (b, lg), ou in oracles.items():
            l = gs.local_layer(lg)
            T, W = ou.committed()
            check_state(_np(gs.state[b, l]), T, f"state after finish unit {(b, l)}")
            if w.conv_mode == 1 and w.K > 1:
                np.testing.assert_array_equal(_np(gs.conv_state[b, l]), W)
    gs.ver.check_error()
    return gs, worst


# ---------------------------------------------------------------------------
# small cases, every element
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", ["ut", "walk"])
def test_tiny_conv_mode(kernel):
    w = S.workload(1).replace(steps=4)
    run_parity(w, kernel=kernel)


def test_tiny_bypass_mode():
    w = S.workload(1).replace(steps=4, conv_mode=0, act=0)
    run_parity(w)


@pytest.mark.parametrize("dk,dv", [(32, 64), (64, 32), (128, 32), (32, 128), (64, 128), (128, 128), (32, 32)])
@pytest.mark.parametrize("kernel", KERNELS)
def test_head_shapes_and_gqa(dk, dv, kernel):
    # d_k != d_v catches a transposed state; Hv = 3 Hk checks the v-head -> k-head map
    if kernel in ("simt", "tc1") and dv != 128:
        pytest.skip("the default UT dispatch already runs the CUDA-core kernel for this d_v")
    w = S.workload(1).replace(Hk=2, Hv=6, dk=dk, dv=dv, steps=3, tree="random", budget=12, n_max=12, path_max=12)
    run_parity(w, kernel=kernel)


@pytest.mark.parametrize("heads", ["tiny", "d128"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_ragged_batch_and_degenerate_trees(heads, kernel):
    # per-request tree sizes 1 .. n_max, a single-node tree, a full chain, L = 0 and L = n commits;
    # with 128-wide heads the UT form runs on the tensor cores, whose node padding these sizes cross
    n_max = 16 if heads == "tiny" else 32
    if heads == "tiny" and kernel in ("simt", "tc1"):
        pytest.skip("the default UT dispatch already runs the CUDA-core kernel for these heads")
    w = S.workload(1).replace(B=5, layers=2, n_max=n_max, steps=3, tree="random", budget=n_max, path_max=n_max)
    if heads == "d128":
        w = w.replace(Hk=2, Hv=6, dk=128, dv=128)
    rng = np.random.default_rng(5)
    trees, paths = [], []
    for s in range(w.steps):
        ts = [np.array([-1], dtype=np.int32), S.chain_tree(n_max), S.random_tree(7, rng), S.random_tree(n_max, rng),
              S.random_tree(3, rng)]
        ps = [np.array([0], dtype=np.int32), np.arange(n_max, dtype=np.int32), np.zeros(0, dtype=np.int32),
              S.random_walk_path(ts[3], rng, max_len=n_max), S.random_walk_path(ts[4], rng, max_len=3)]
        trees.append(ts)
        paths.append(ps)
    from harness import WorkloadPlan
    run_parity(w, plan=WorkloadPlan(w, trees, paths), kernel=kernel)


def test_compaction_is_exact_and_transparent():
    w = S.workload(1).replace(B=3, layers=2, steps=4, tree="random", budget=10, n_max=10, path_max=10)
    gs, _ = run_parity(w, compact_steps=(0, 1, 2, 3))


@pytest.mark.parametrize("cfg", [1, 2], ids=["tiny", "qwen"])
def test_per_node_state_schedule(cfg):
    # the per-node-state baseline (every node reloads its parent's stored state) gives the same results
    from harness import WorkloadPlan
    w = S.workload(cfg).replace(steps=3, B=2) if cfg == 1 else S.workload(cfg).replace(steps=3)
    plan = WorkloadPlan(w, per_node=True)
    run_parity(w, plan=plan)


def binary_tree(n):
    return np.array([-1] + [(i - 1) // 2 for i in range(1, n)], dtype=np.int32)


@pytest.mark.parametrize("cfg", [1, 2], ids=["tiny", "qwen"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_deep_light_depth_spills_stashes_to_hbm(cfg, kernel):
    # perfect binary trees (light depth 4 at 31 nodes) and random 32-node trees: stashes two or more
    # levels deep leave tensor memory for the boundary slots, and every node must still match
    from harness import WorkloadPlan
    n_max = 32
    w = S.workload(cfg).replace(B=3, layers=2 if cfg == 1 else 1, n_max=n_max, budget=n_max, path_max=n_max,
                                steps=3, tree="random")
    rng = np.random.default_rng(17)
    trees, paths = [], []
    for s in range(w.steps):
        ts = [binary_tree(31), binary_tree(n_max), S.random_tree(n_max, rng)]
        trees.append(ts)
        paths.append([S.random_walk_path(t, rng, max_len=n_max) for t in ts])
    if cfg == 1 and kernel in ("simt", "tc1"):
        pytest.skip("the default UT dispatch already runs the CUDA-core kernel for these heads")
    run_parity(w, plan=WorkloadPlan(w, trees, paths), kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_boundary_scratch_changes_no_result(kernel):
    # with boundary states as scratch the outputs, banks and committed states are bit-identical
    from harness import GpuSession, WorkloadPlan
    n_max = 32
    w = S.workload(2).replace(B=3, layers=2, n_max=n_max, budget=n_max, path_max=n_max, steps=3, tree="random")
    rng = np.random.default_rng(23)
    trees = [[binary_tree(31), S.ddtree(22, 4, 10, rng), S.random_tree(n_max, rng)] for _ in range(w.steps)]
    paths = [[S.random_walk_path(t, rng, max_len=n_max) for t in ts] for ts in trees]
    plan = set_kernel(WorkloadPlan(w, trees, paths), kernel)
    a, b = GpuSession(w, plan), GpuSession(w, plan)
    for s in range(w.steps):
        a.verify(s)
        b.verify(s, boundary_scratch=True)
        torch.cuda.synchronize()
        assert torch.equal(a.out_o, b.out_o), s
        assert torch.equal(a.state, b.state), s
        for f in ("k", "u", "a", "x"):
            assert torch.equal(a.ver.bank_view(f, a.ver.banks.verified_bank),
                               b.ver.bank_view(f, b.ver.banks.verified_bank)), (s, f)
        a.commit(s)
        b.commit(s)
    a.finish()
    b.finish()
    torch.cuda.synchronize()
    assert torch.equal(a.state, b.state)
    a.ver.check_error()
    b.ver.check_error()


@pytest.mark.parametrize("kernel", KERNELS)
def test_qwen_like_single_layer(kernel):
    w = S.workload(2).replace(steps=3)
    run_parity(w, kernel=kernel)


@pytest.mark.parametrize("kernel", ["chains_tc", "ut", "walk"])
def test_chain64_single_layer(kernel):
    # the pure-chain shape of the stress workload: 64-node chain, chain acceptance of the whole walk.
    # "chains_tc": the caller declares every tree a chain, and the tensor cores solve it in 16-node segments;
    # "ut": the UT form would hand a 63-deep chain to the walk; here it is made to solve it itself
    from harness import WorkloadPlan
    w = S.workload(6).replace(B=2, layers=1, steps=2)
    plan = WorkloadPlan(w)
    plan.depth_hint = kernel == "walk"
    plan.chains = kernel == "chains_tc"
    run_parity(w, plan=plan, kernel="ut" if kernel == "chains_tc" else kernel)


@pytest.mark.parametrize("n_chain", [1, 5, 16, 17, 31, 33, 48, 64])
def test_chain_segments_ragged(n_chain):
    # chains of every segment shape (one partial segment, exact multiples of 16, a last segment of 1 node),
    # several requests and layers, commits of the whole chain and of a prefix, 128-wide and 64-wide keys
    from harness import WorkloadPlan
    for dk in (128, 64):
        w = S.workload(6).replace(B=3, layers=2, steps=3, Hk=2, Hv=6, dk=dk, budget=n_chain, n_max=64)
        rng = np.random.default_rng(n_chain)
        trees = [[S.chain_tree(n_chain) for _ in range(w.B)] for _ in range(w.steps)]
        paths = [[np.arange(int(rng.integers(0, n_chain + 1)), dtype=np.int32) for _ in range(w.B)]
                 for _ in range(w.steps)]
        plan = WorkloadPlan(w, trees, paths)
        plan.chains = True
        run_parity(w, plan=plan)


def test_chains_flag_refuses_a_tree():
    # a tree that is not a chain under GDN_VERIFY_CHAINS is skipped with a schedule error, not solved wrongly
    from harness import GpuSession, WorkloadPlan
    import gated_deltanet_tree_gb300 as G
    w = S.workload(6).replace(B=2, layers=1, steps=1, Hk=2, Hv=6, budget=40, n_max=40)
    trees = [[S.chain_tree(40), np.array([-1] + [0] * 39, dtype=np.int32)]]
    plan = WorkloadPlan(w, trees, [[np.arange(3, dtype=np.int32), np.zeros(0, dtype=np.int32)]])
    plan.chains = True
    gs = GpuSession(w, plan)
    gs.verify(0)
    with pytest.raises(G.GdnError) as e:
        gs.ver.check_error()
    assert e.value.status == G._native.GDN_ERR_SCHEDULE


@pytest.mark.parametrize("kernel", ["ut", "simt", "walk"])
def test_ddtree64_top8_single_layer(kernel):
    # the default dispatch ("ut") solves these 64-node, depth <= 16 trees on the tensor cores in one segment
    w = S.workload(5).replace(B=2, layers=1, steps=2)
    run_parity(w, kernel=kernel)


def shallow_random_tree(n, rng, max_depth=16):
    while True:
        t = S.random_tree(n, rng)
        d = np.zeros(n, dtype=np.int64)
        for i in range(1, n):
            d[i] = d[t[i]] + 1
        if d.max() <= max_depth:
            return t


@pytest.mark.parametrize("dk", [128, 64])
def test_wide_trees_ragged(dk):
    # trees of 33 to 64 nodes (and smaller ones in the same batch) on the tensor cores: DDTrees, random trees,
    # a star, a node at depth 16, boundary states stored and replayed, commits of every length
    from harness import WorkloadPlan
    n_max = 64
    w = S.workload(5).replace(B=4, layers=2, steps=3, Hk=2, Hv=6, dk=dk, n_max=n_max, budget=n_max, path_max=n_max,
                              tree="random")
    rng = np.random.default_rng(41 + dk)
    deep = np.array([-1] + list(range(16)) + [0] * 20, dtype=np.int32)   # a 16-deep chain plus a star
    trees = [[S.ddtree(64, 8, 16, rng), shallow_random_tree(int(rng.integers(33, 65)), rng), deep,
              shallow_random_tree(int(rng.integers(1, 33)), rng)] for _ in range(w.steps)]
    paths = [[S.random_walk_path(t, rng, max_len=n_max) for t in ts] for ts in trees]
    run_parity(w, plan=WorkloadPlan(w, trees, paths))


# the method's degenerate cases, driven through every verify kernel: each variant below changes the Qwen-like
# layer (128-wide heads, 22-node DDTrees, fold of the previous step's path) in one way
EDGE_VARIANTS = {
    "gate_zero": dict(edge="gate_zero"),                        # log g = -inf: g = 0, the state is forgotten
    "gate_floor": dict(edge="gate_floor", path_max=22),         # gate products below 1e-12 (the lazy decay's floor)
    "beta01": dict(edge="beta01"),                              # beta = 0 writes nothing; beta = 1 with |k| = 1
    "zero_rows_bypass": dict(edge="zero_rows", conv_mode=0, act=0),   # q = k = 0: eps alone keeps q_hat, k_hat finite
    "zero_rows_conv": dict(edge="zero_rows"),                   # k-head 0 convolves to zero
    "q_scale": dict(q_scale=float(1.0 / np.sqrt(128.0))),       # the Qwen-style query scale
    "fp32_inputs": dict(in_dtype=S.DTYPE_F32),                  # fp32 x, beta, log g at 128-wide heads
}


@pytest.mark.parametrize("variant", sorted(EDGE_VARIANTS))
@pytest.mark.parametrize("kernel", KERNELS)
def test_edge_cases(variant, kernel):
    w = S.workload(2).replace(Hk=2, Hv=6, B=2, layers=2, steps=3, **EDGE_VARIANTS[variant])
    run_parity(w, kernel=kernel)


# ---------------------------------------------------------------------------
# full-size workloads, sampled units
# ---------------------------------------------------------------------------

def test_qwen_48_layers_commit_then_verify():
    w = S.workload(3)
    run_parity(w, units=[(0, 0), (0, 17), (0, 47)])


@pytest.mark.parametrize("kernel", KERNELS)
def test_batched_32x48_eight_steps(kernel):
    w = S.workload(4)
    run_parity(w, units=[(0, 0), (13, 29), (31, 47)], kernel=kernel)


@pytest.mark.parametrize("cfg", [5, 6], ids=["ddtree64_top8", "chain64"])
def test_stress_128_requests_layer_chunked(cfg):
    # 128 requests x 48 layers of 64-node trees, all 8 verify -> commit steps: the boundary states alone would
    # take ~360 GB, so a call covers 8 layers; the chunk holding the sampled units runs every step.  The
    # top-8 trees run on the tensor cores in one segment, the pure chains in 16-node segments.
    w = S.workload(cfg)
    assert w.steps == 8
    from harness import WorkloadPlan
    plan = WorkloadPlan(w)
    plan.chains = cfg == 6
    run_parity(w, units=[(0, 0), (127, 5)], plan=plan, layer_ids=range(0, 8))


def test_checkpoint_resume_is_bitwise():
    """finish -> save {state, conv window} -> fresh session -> continue equals the uninterrupted run."""
    import io
    from harness import GpuSession, WorkloadPlan
    w = S.workload(2).replace(B=2, layers=2, steps=4)
    plan = WorkloadPlan(w)
    ref = GpuSession(w, plan)
    outs = {}
    for s in range(w.steps):
        ref.verify(s)
        outs[s] = ref.out_o.clone()
        ref.commit(s)
    ref.finish()
    a = GpuSession(w, plan)
    for s in range(2):
        a.verify(s)
        a.commit(s)
    a.finish()
    buf = io.BytesIO()
    torch.save({"state": a.state.cpu(), "conv_state": a.conv_state.cpu()}, buf)
    buf.seek(0)
    ck = torch.load(buf)
    b = GpuSession(w, plan)
    b.state.copy_(ck["state"])
    b.conv_state.copy_(ck["conv_state"])
    for s in range(2, w.steps):
        b.verify(s)
        torch.cuda.synchronize()
        assert torch.equal(b.out_o, outs[s]), s
        b.commit(s)
    b.finish()
    torch.cuda.synchronize()
    assert torch.equal(b.state, ref.state)
    assert torch.equal(b.conv_state, ref.conv_state)


# ---------------------------------------------------------------------------
# lifecycle and device-side checks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", KERNELS)
def test_fold_reproduces_boundary_state_bitwise(kernel):
    """The committed state folded from the factor bank equals, bit for bit, the
    state the previous verify stored for the path's last node when that node was
    a boundary (same operation order in fold and verify)."""
    from harness import GpuSession, WorkloadPlan
    w = S.workload(2).replace(steps=2)
    plan = WorkloadPlan(w)
    p0 = plan.trees[0][0]
    kids = np.bincount(p0[1:], minlength=len(p0))
    target = max(i for i in range(len(p0)) if kids[i] >= 2)
    path = [target]
    while p0[path[-1]] >= 0:
        path.append(int(p0[path[-1]]))
    plan.paths[0][0] = np.array(path[::-1], dtype=np.int32)
    set_kernel(plan, kernel)
    gs = GpuSession(w, plan)
    gs.verify(0)
    slot = sorted(i for i in range(len(p0)) if kids[i] >= 2).index(target)
    saved = gs.boundary[0, 0, slot].clone()
    gs.commit(0)
    gs.verify(1)
    torch.cuda.synchronize()
    assert torch.equal(gs.state[0, 0], saved)


def test_invalid_path_sets_device_error_and_commits_nothing():
    from harness import GpuSession, WorkloadPlan
    import gated_deltanet_tree_gb300 as G
    w = S.workload(1).replace(B=2, steps=2, tree="random", budget=8, n_max=8)
    plan = WorkloadPlan(w)
    p = plan.trees[0][1]
    non_child = [i for i in range(1, len(p)) if p[i] != 0]
    # [0, v] with v not a child of the root, or (star tree) a path that does not start at the root
    plan.paths[0][1] = np.array([0, non_child[0]] if non_child else [1], dtype=np.int32)
    gs = GpuSession(w, plan)
    state0 = gs.state.clone()
    gs.verify(0)
    gs.commit(0)
    with pytest.raises(G.GdnError) as e:
        gs.ver.check_error()
    assert e.value.status == G._native.GDN_ERR_INVALID_PATH
    assert int(gs.ver.pend_len[1]) == 0
    gs.verify(1)
    torch.cuda.synchronize()
    assert torch.equal(gs.state[1], state0[1])       # nothing folded for the bad request
    assert not torch.equal(gs.state[0], state0[0])   # the good request folded its path
    gs.ver.check_error()


def test_bounded_wait_gives_up_and_reports_timeout():
    """A wait that nothing completes gives up after its bound, the host reads GDN_ERR_TIMEOUT, and the
    context still verifies correctly afterwards (the error word cleared by the read)."""
    from harness import GpuSession
    import gated_deltanet_tree_gb300 as G
    w = S.workload(2).replace(Hk=2, Hv=6, steps=2)
    gs = GpuSession(w)
    G._native.gdn_selftest_wait_timeout(gs.ver.banks)
    with pytest.raises(G.GdnError) as e:
        gs.ver.check_error()
    assert e.value.status == G._native.GDN_ERR_TIMEOUT
    run_parity(w)


def test_timeout_bit_is_sticky_until_checked():
    """While GDN_DEVERR_TIMEOUT is set, later verify and finish calls on the same banks do no work (outputs
    and state untouched) until gdn_check_error reads and clears it; afterwards the banks verify normally."""
    from harness import GpuSession
    import gated_deltanet_tree_gb300 as G
    w = S.workload(2).replace(Hk=2, Hv=6, steps=2)
    gs = GpuSession(w)
    gs.verify(0)
    gs.commit(0)
    torch.cuda.synchronize()
    gs.ver.check_error()
    G._native.gdn_selftest_wait_timeout(gs.ver.banks)
    state0, o0 = gs.state.clone(), gs.out_o.clone()
    gs.out_o.fill_(7.0)
    gs.verify(1)                        # no check in between: the pending fold and the verify must not run
    torch.cuda.synchronize()
    assert torch.equal(gs.state, state0)
    assert bool((gs.out_o == 7.0).all())
    with pytest.raises(G.GdnError) as e:
        gs.ver.check_error()
    assert e.value.status == G._native.GDN_ERR_TIMEOUT
    gs.ver.check_error()                # cleared by the read
    run_parity(w)                       # a fresh session on the same context is unaffected


def test_finish_without_pending_is_a_noop_and_commit_needs_verify():
    from harness import GpuSession
    import gated_deltanet_tree_gb300 as G
    w = S.workload(1)
    gs = GpuSession(w)
    s0 = gs.state.clone()
    gs.finish()
    torch.cuda.synchronize()
    assert torch.equal(gs.state, s0)
    with pytest.raises(G.GdnError) as e:
        gs.commit(0)
    assert e.value.status == G._native.GDN_ERR_STATE


def test_cuda_graph_replay_matches_eager():
    from harness import GpuSession, WorkloadPlan
    w = S.workload(2).replace(B=2, layers=3, steps=3)
    plan = WorkloadPlan(w)
    eager = GpuSession(w, plan)
    graphed = GpuSession(w, plan)
    for s in range(w.steps):
        graphed.step_inputs(s), graphed.schedule(s), graphed.paths(s)
    outs_e, outs_g = [], []
    for s in range(w.steps):
        eager.verify(s)
        outs_e.append(eager.out_o.clone())
        eager.commit(s)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    for s in range(w.steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            graphed.verify(s, stream=stream)
            graphed.commit(s, stream=stream)
        g.replay()
        torch.cuda.synchronize()
        outs_g.append(graphed.out_o.clone())
    for a, b in zip(outs_e, outs_g):
        assert torch.equal(a, b)
    assert torch.equal(eager.state, graphed.state)
