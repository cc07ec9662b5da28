"""gdn_tree_verify_noalloc: the verify call for callers that cannot allocate device memory.

Callers running inside a stream capture, engines whose device pool belongs to
their own allocator, and plugins handed only buffers and a stream cannot pass
the workspace gdn_tree_verify asks for.  The no-allocation entry point uses the
library's fixed device scratch instead.  These tests call it through the C ABI
and check that two calls in a row give, bit for bit, what the workspace entry
point gives on the same inputs, and that a batch too large for the fixed scratch is refused
before anything runs.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gated_deltanet_tree_gb300.build import build
    build()


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # both entry points launch the same kernels on the same inputs, so every result must be bit-identical
    # (which is within every tolerance the parity tests use); a difference would point at scratch addressing
    from gated_deltanet_tree_gb300 import _native as N
    from harness import GpuSession, WorkloadPlan
    w = S.workload(2).replace(steps=2)
    plan = WorkloadPlan(w)
    ref = GpuSession(w, plan)       # gdn_tree_verify with a caller workspace
    new = GpuSession(w, plan)       # gdn_tree_verify_noalloc
    for s in range(2):
        ref.verify(s)
        X, BE, AG = new.step_inputs(s)
        N.gdn_tree_verify_noalloc(new.dims, w.layers, new.schedule(s).struct, X, new.conv_w, BE, AG, new.state,
                                  new.conv_state, new.out_o, new.boundary, new.ver.banks)
        torch.cuda.synchronize()
        n = len(plan.trees[s][0])
        nb = new.schedule(s).nb_max
        assert torch.equal(new.out_o[:, :, :n], ref.out_o[:, :, :n])
        assert torch.equal(new.state, ref.state)
        assert torch.equal(new.conv_state, ref.conv_state)
        assert torch.equal(new.boundary[:, :, :nb], ref.boundary[:, :, :nb])
        bank = new.ver.banks.verified_bank
        assert bank == ref.ver.banks.verified_bank
        for f in ("k", "u", "a", "x"):
            assert torch.equal(new.ver.bank_view(f, bank)[:, :, :n], ref.ver.bank_view(f, bank)[:, :, :n]), f
        ref.commit(s)
        new.commit(s)
    new.ver.check_error()
    ref.ver.check_error()


def test_noalloc_refuses_batches_beyond_the_fixed_scratch():
    from gated_deltanet_tree_gb300 import _native as N
    from gated_deltanet_tree_gb300.runtime import TreeVerifier, make_dims
    d = make_dims(16, 48, 128, 128, 4)
    B, layers, n_max = 32, 48, 22
    need = N.gdn_workspace_bytes(d, B, layers, n_max)
    assert need > (64 << 20)
    words = torch.zeros(B, N.gdn_schedule_words(n_max), dtype=torch.int32, device="cuda")
    sched = N.gdn_batch_schedule(B=B, n_max=n_max, nb_max=1, words=words.data_ptr())
    ver = TreeVerifier(make_dims(16, 48, 128, 128, 4), 1, 1, n_max)   # real buffers; nothing is launched
    dummy = torch.zeros(256, device="cuda")
    with pytest.raises(N.GdnError) as e:
        N.gdn_tree_verify_noalloc(d, layers, sched, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                  ver.banks)
    assert e.value.status == N.GDN_ERR_CAPACITY
    assert "fixed scratch" in str(e.value)
