"""The debug build (libmuon_debug.so, compiled with -DMUON_DEBUG): device-side range
checks that record a status bit and skip the access instead of touching memory out
of range, read back by muon_sync as MUON_ERR_DEVICE.

On valid inputs its results match the oracle like the release build's.  The one
input a caller can corrupt on the device is the workspace, whose tile schedules the
grouped GEMM reads: with the workspace overwritten after binding, every GEMM launch
finds its schedule out of range, runs no tile, and muon_sync reports it; the weights
are untouched and a fresh plan steps on and matches the oracle.  (Only the debug
build is given the corrupted workspace: the release build has no such checks.)
"""
import gc

import pytest

import synth
from gpu_util import TOL_BF16, Workload, nsm, run_steps, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    mod = nsm()
    was_debug = mod.using_debug_library()
    gc.collect()                     # no plan of the other library is alive
    mod.use_debug_library(True)
    yield mod
    gc.collect()                     # the debug library's plans go before it does
    mod.use_debug_library(was_debug)


@pytest.mark.parametrize("shapes,kw", [
    ([(256, 512), (300, 200, 2), (777, 129)], {}),                      # grouped GEMM buckets
    ([(128, 2560, 3), (100, 704)], {}),                                 # small-matrix kernel, momentum inside
    ([(128, 640, 2), (64, 1024)], {"ns_method": 1}),                    # the gram method
    ([(256, 512), (512, 256)], {"ns_precision": 1}),                    # 3xTF32 GEMMs
])
def test_debug_build_matches_oracle(m, shapes, kw):
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    cfg = m.muon_config_default(**kw)
    tol = 1e-4 if kw.get("ns_precision") == 1 else TOL_BF16
    ulp, rel = run_steps(m, wl, steps=2, cfg=cfg, tol=tol, method="gram" if kw.get("ns_method") == 1 else "standard")
    assert ulp <= 1 and rel <= tol


def test_debug_build_catches_a_corrupted_schedule(m):
    import torch
    shapes = [(256, 512), (384, 192, 2)]
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    plan = m.muon_plan(wl.plan_shapes())
    ws = m.allocate_workspace(plan)
    ws[1024:].fill_(0x7F)            # everything after the status word, the tile schedules included
    W0 = [to_numpy(t, synth.F32) for t in wl.dW]
    m.muon_step(plan, wl.dW, wl.dG, wl.dM, 0.02, 0.95, True, 0.0, 5)
    with pytest.raises(m.MuonError) as e:
        m.muon_sync(plan)
    assert e.value.status == m.MUON_ERR_DEVICE and "range check" in str(e.value)
    torch.cuda.synchronize()
    for w0, w in zip(W0, wl.dW):     # no tile ran, so no weight update either
        assert (to_numpy(w, synth.F32) == w0).all()
    assert m.muon_sync(plan) == (m.MUON_OK, 0)   # the status word was cleared
    del plan, ws
    # the context is usable: a fresh plan and workspace step and match the oracle
    wl = Workload(shapes, m_sigma=0.02, g_sigma=1e-3)
    ulp, rel = run_steps(m, wl, steps=1)
    assert ulp <= 1 and rel <= TOL_BF16
