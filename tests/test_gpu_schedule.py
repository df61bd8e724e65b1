"""Per-iteration Newton-Schulz coefficients on the GPU, against the fp64 oracle.

The schedule is the oracle's minimax construction (an input to both sides, rounded
to the fp32 values the GPU uses), fitted on intervals widened by 5% at the top:
bf16 rounding pushes singular values a little past an interval's upper end, where
an unwidened fit is steep (a CPU simulation of the bf16 path gives 5.0e-2 against
the oracle for five unwidened steps, 1.0e-2 with the widening); the GPU runs it through the grouped GEMM
launches (CTA pairs and single CTAs, bf16 and 3xTF32) and through the
single-launch kernel for matrices of at most 128 rows.  A schedule shorter than
the iteration count repeats its last triple; an empty one restores the
configuration's coefficients.  The updates' singular values also land in the band
the schedule guarantees, which is how the pages' aim -- fewer iterations to the
same polar accuracy -- shows on the device.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_BF16, TOL_TF32X3, Workload, nsm, run_steps, to_numpy

pytestmark = pytest.mark.gpu

LOWER = 1e-3
SAFETY = 1.05


@pytest.fixture(scope="module")
def m():
    return nsm()


def _schedule(n):
    co, _ = oracle.polar_express_schedule(n, LOWER, SAFETY)
    return co


@pytest.mark.parametrize("shapes", [
    [(256, 512)],                      # one CTA-pair tile row
    [(700, 1000), (1000, 700)],        # ragged, wide and tall
    [(100, 700), (700, 1000)],         # single-CTA tiles (a group of <= 128 rows)
    [(128, 2560, 3), (96, 1000)],      # the single-launch small-matrix kernel
])
@pytest.mark.parametrize("ns_steps", [4, 5])
def test_minimax_schedule_matches_oracle(m, shapes, ns_steps):
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    ulp, rel = run_steps(m, wl, steps=2, ns_steps=ns_steps, schedule=_schedule(ns_steps))
    assert ulp <= 1 and rel <= TOL_BF16


def test_short_schedule_repeats_its_last_triple(m):
    # the sixth triple is fitted on an interval near 1, where it contracts toward
    # 1; repeating a triple fitted for a wide interval would not converge (the
    # singular values keep moving inside its band, and rounding grows)
    wl = Workload([(384, 640), (128, 512, 2)], m_sigma=0.02, g_sigma=1e-3)
    run_steps(m, wl, ns_steps=8, schedule=_schedule(6))


def test_sixteen_iterations(m):
    wl = Workload([(300, 500), (64, 700)], m_sigma=0.02, g_sigma=1e-3)
    run_steps(m, wl, ns_steps=16, schedule=_schedule(16))


def test_schedule_in_3xtf32(m):
    wl = Workload([(256, 384), (300, 200)], m_sigma=0.02, g_sigma=1e-3)
    cfg = m.muon_config_default(ns_precision=m.MUON_NS_TF32X3)
    ulp, rel = run_steps(m, wl, ns_steps=4, schedule=_schedule(4), cfg=cfg, tol=TOL_TF32X3)
    assert ulp <= 1 and rel <= TOL_TF32X3


def test_empty_schedule_restores_the_configuration(m):
    import torch
    outs = []
    for sched in (None, []):
        wl = Workload([(384, 640), (128, 512, 2)], m_sigma=0.02, g_sigma=1e-3)
        plan = m.muon_plan(wl.plan_shapes())
        m.allocate_workspace(plan)
        if sched is not None:
            m.muon_set_ns_schedule(plan, _schedule(5))
            m.muon_set_ns_schedule(plan, sched)
        m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5)
        torch.cuda.synchronize()
        outs.append([to_numpy(t, synth.F32) for t in wl.dW])
    for a, b in zip(*outs):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("kernel_shape", [(512, 1024), (128, 1024)])
def test_update_singular_values_lie_in_the_schedules_band(m, kernel_shape):
    # weights start at 0 and lr = 1, so W_new = -U: the update itself.  Four
    # minimax steps from [1e-3, 1] guarantee |1 - sigma| <= E_3 for every input
    # singular value at least 1e-3 of the norm; bf16 adds at most a few percent.
    import torch
    r, c = kernel_shape
    co, errs = oracle.polar_express_schedule(4, LOWER, SAFETY)
    wl = Workload([(r, c)], w_sigma=0.0, g_sigma=1.0, g_dtype=synth.F32)
    plan = m.muon_plan(wl.plan_shapes(), config=m.muon_config_default(grad_dtype=m.MUON_DTYPE_F32))
    m.allocate_workspace(plan)
    m.muon_set_ns_schedule(plan, co)
    m.muon_step(plan, wl.dW, wl.dG, wl.dM, 1.0, 0.0, False, 0.0, 4)
    torch.cuda.synchronize()
    U = -to_numpy(wl.dW[0], synth.F32)[0].astype(np.float64)
    G = synth.as_f64(wl.G[0][0], wl.g_dtype)
    s_in = np.linalg.svd(G, compute_uv=False)
    s_out = np.linalg.svd(U, compute_uv=False)
    assert s_in.min() / np.linalg.norm(G) >= LOWER  # a Gaussian matrix this wide: every value in range
    band = errs[3] + 0.03
    assert np.all(np.abs(1.0 - s_out) <= band), (s_out.min(), s_out.max(), errs[3])
