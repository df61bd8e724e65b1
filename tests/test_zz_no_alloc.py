"""muon_step_noalloc: the Muon step for callers that cannot allocate device memory.

Such callers (code inside an allocator or memory-pool callback, a runtime that
has given all device memory to its own pool, a plugin host that forbids device
allocations) cannot create the workspace muon_step needs; muon_step_noalloc runs
the same step in the library's static device scratch.  Its results must agree
with muon_step's, within the tolerances of the parity tests, on consecutive calls.
This file is collected last so a failure here stops a -x run after every other test.
"""
import numpy as np
import pytest

import synth
from gpu_util import TOL_BF16, Workload, nsm, rel_fro, to_numpy, ulp_distance

pytestmark = pytest.mark.gpu

SHAPES = [(256, 512), (384, 192, 2), (100, 300)]


def test_noalloc_matches_muon_step_on_two_calls():
    import torch
    m = nsm()
    ref = Workload(SHAPES, m_sigma=0.02, g_sigma=1e-3)
    got = Workload(SHAPES, m_sigma=0.02, g_sigma=1e-3)      # same seeded inputs
    plan_ref = m.muon_plan(ref.plan_shapes())
    m.allocate_workspace(plan_ref)
    plan = m.muon_plan(got.plan_shapes())                    # no workspace bound
    assert m.muon_plan_workspace_bytes(plan) <= m.muon_noalloc_scratch_bytes()
    for call in range(2):
        W0 = [to_numpy(t, synth.F32) for t in ref.dW]
        m.muon_step(plan_ref, ref.dW, ref.dG, ref.dM, 0.02, 0.95, True, 0.0, 5)
        m.muon_step_noalloc(plan, got.dW, got.dG, got.dM, 0.02, 0.95, True, 0.0, 5)
        st, nf = m.muon_sync(plan)
        assert st == m.MUON_OK and nf == 0
        torch.cuda.synchronize()
        for i in range(len(SHAPES)):
            w_ref, w_got = to_numpy(ref.dW[i], synth.F32), to_numpy(got.dW[i], synth.F32)
            m_ref, m_got = to_numpy(ref.dM[i], synth.F32), to_numpy(got.dM[i], synth.F32)
            assert int(ulp_distance(m_got, m_ref).max()) <= 1, f"call {call} tensor {i}: momentum"
            for j in range(w_ref.shape[0]):
                d_ref = w_ref[j].astype(np.float64) - W0[i][j]
                d_got = w_got[j].astype(np.float64) - W0[i][j]
                assert rel_fro(d_got, d_ref) <= TOL_BF16, f"call {call} tensor {i} matrix {j}"
        got.dW = [t.clone().copy_(r) for t, r in zip(got.dW, ref.dW)]  # same state for the next call
        got.dM = [t.clone().copy_(r) for t, r in zip(got.dM, ref.dM)]


def test_noalloc_rejects_a_plan_larger_than_the_scratch():
    m = nsm()
    plan = m.muon_plan([(4096, 4096, 2)])
    assert m.muon_plan_workspace_bytes(plan) > m.muon_noalloc_scratch_bytes()
    with pytest.raises(m.MuonError) as e:
        m.muon_step_noalloc(plan, [16], [32], [48], 0.02, 0.95, True, 0.0, 5)
    assert e.value.status == m.MUON_ERR_NO_WORKSPACE
