"""muon_step_noalloc: the Muon step for callers that cannot allocate device memory.

Such callers (code inside an allocator or memory-pool callback, a runtime that
has given all device memory to its own pool, a plugin host that forbids device
allocations) cannot create the workspace muon_step needs; muon_step_noalloc runs
the same step in the library's static device scratch.  Its results must agree
with muon_step's, within the tolerances of the parity tests, on consecutive calls;
calls of different plans enqueued back to back on one non-blocking stream must
each match the oracle; and the device status word must keep a non-finite count
across another plan's call until muon_sync reads it.
This file is collected last so a failure here stops a -x run after every other test.
"""
import numpy as np
import pytest

import synth
from gpu_util import TOL_BF16, Workload, check_step, nsm, rel_fro, to_numpy, ulp_distance

pytestmark = pytest.mark.gpu

SHAPES = [(256, 512), (384, 192, 2), (100, 300)]
# a second plan: a grouped-GEMM bucket and a small-matrix bucket (cap 900 000 bytes)
SHAPES_B = [(320, 640, 2), (128, 512, 3)]
CAP_B = 900_000


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


def test_noalloc_two_plans_alternating_on_one_nonblocking_stream():
    # six calls, plans A B A B A B, enqueued on one torch side stream (created
    # non-blocking) with no host synchronisation between them; each re-binds the
    # scratch to its plan.  The state before and after every call is copied on
    # the same stream and every call is checked against the oracle afterwards.
    import torch
    m = nsm()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        wls = [Workload(SHAPES, m_sigma=0.02, g_sigma=1e-3),
               Workload(SHAPES_B, m_sigma=0.02, g_sigma=1e-3, seed=synth.SEED + 1)]
    plans = [m.muon_plan(wls[0].plan_shapes()), m.muon_plan(wls[1].plan_shapes(), bucket_cap_bytes=CAP_B)]
    assert m.muon_get_plan_info(plans[1]).n_buckets == 2
    assert [m.muon_get_bucket_info(plans[1], b).ns_single_kernel for b in range(2)] == [0, 1]
    s.synchronize()
    records = []
    with torch.cuda.stream(s):
        for call in range(6):
            k = call % 2
            wl = wls[k]
            if call >= 2:
                wl.new_grads(call)                                  # uploaded on s
            before = [t.clone() for t in wl.dW + wl.dM]
            m.muon_step_noalloc(plans[k], wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5, stream=s)
            after = [t.clone() for t in wl.dW + wl.dM]
            records.append((k, list(wl.G), before, after))
    assert m.muon_sync(plans[0], stream=s) == (m.MUON_OK, 0)
    torch.cuda.synchronize()
    for call, (k, G, before, after) in enumerate(records):
        wl = wls[k]
        n = len(wl.shapes)
        wl.G = G
        host = [to_numpy(t, synth.F32) for t in before + after]
        _, rel = check_step(wl, host[:n], host[n:2 * n], host[2 * n:3 * n], host[3 * n:],
                            lr=0.02, mu=0.95, nesterov=True, wd=0.0, ns_steps=5)
        assert rel <= TOL_BF16, f"call {call} (plan {'AB'[k]})"


def test_noalloc_nonfinite_count_survives_another_plans_call():
    # a NaN gradient in plan A's call, then a call of plan B (which re-binds the
    # scratch) and one more of A: the shared status word still holds A's counts
    # when muon_sync reads it, and reading clears it.  The NaN stays in that
    # matrix's momentum, so both calls of A count it: 2.
    import torch
    m = nsm()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = Workload([(64, 128, 3)], m_sigma=0.02, g_sigma=1e-3)
        b = Workload(SHAPES_B, m_sigma=0.02, g_sigma=1e-3, seed=synth.SEED + 2)
        g_nan = a.dG[0].clone()
        g_nan[1, 5, 7] = float("nan")
        W0 = a.dW[0].clone()
    plan_a = m.muon_plan(a.plan_shapes())
    plan_b = m.muon_plan(b.plan_shapes(), bucket_cap_bytes=CAP_B)
    with torch.cuda.stream(s):
        m.muon_step_noalloc(plan_a, a.dW, [g_nan], a.dM, 0.02, 0.95, True, 0.0, 5, stream=s)
        W1 = a.dW[0].clone()
        m.muon_step_noalloc(plan_b, b.dW, b.dG, b.dM, 0.02, 0.95, True, 0.0, 5, stream=s)
        m.muon_step_noalloc(plan_a, a.dW, a.dG, a.dM, 0.02, 0.95, True, 0.0, 5, stream=s)
    st, nf = m.muon_sync(plan_b, stream=s)
    assert st == m.MUON_WARN_NONFINITE and nf == 2
    assert m.muon_sync(plan_a, stream=s) == (m.MUON_OK, 0)   # cleared by the read
    torch.cuda.synchronize()
    assert torch.equal(W1[1], W0[1])                          # the NaN matrix was skipped
    assert not torch.equal(W1[0], W0[0]) and not torch.equal(W1[2], W0[2])
    assert torch.isfinite(W1).all() and torch.isfinite(b.dW[0]).all()


def test_noalloc_rejects_a_plan_larger_than_the_scratch():
    m = nsm()
    plan = m.muon_plan([(4096, 4096, 2)])
    assert m.muon_plan_workspace_bytes(plan) > m.muon_noalloc_scratch_bytes()
    with pytest.raises(m.MuonError) as e:
        m.muon_step_noalloc(plan, [16], [32], [48], 0.02, 0.95, True, 0.0, 5)
    assert e.value.status == m.MUON_ERR_NO_WORKSPACE
