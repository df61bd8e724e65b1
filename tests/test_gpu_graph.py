"""muon_step captured in a CUDA graph and replayed.

muon_step only enqueues work on the caller's stream (kernel launches, no host
synchronisation), so a caller can capture one step with stream capture and replay
it every iteration: the launches' arguments (tensor maps, pointers, lr, mu) are
those of the captured call, and each replay reads the gradients then in the
captured tensors.  Checked here on a plan with a grouped-GEMM bucket (wide and tall
matrices) and a small-matrix bucket: every replayed step against the fp64 oracle
(teacher forced), and the replays bit for bit against eager steps on a copy of the
same state.
"""
import numpy as np
import pytest

import synth
from gpu_util import TOL_BF16, Workload, check_step, nsm, to_numpy

pytestmark = pytest.mark.gpu

LR, MU, WD, NS = 0.02, 0.95, 0.01, 5


@pytest.mark.parametrize("method, shapes, kinds", [
    # a grouped-GEMM bucket (wide and tall matrices) and a small-matrix bucket
    ("standard", [(256, 512, 1), (384, 192, 2), (128, 640, 5)], {0, 1}),
    # the gram method runs in the small-matrix kernel only (m <= 128; one tall matrix)
    ("gram", [(128, 640, 5), (300, 96, 2)], {1}),
])
def test_graph_replay_matches_the_oracle_and_the_eager_step(method, shapes, kinds):
    import torch
    m = nsm()
    wl = Workload(shapes, w_sigma=0.02, m_sigma=0.02, g_sigma=1e-3, g_dtype=synth.BF16)
    cfg = m.muon_config_default(grad_dtype=synth.BF16,
                                ns_method=m.MUON_NS_METHOD_GRAM if method == "gram" else m.MUON_NS_METHOD_STANDARD)
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=1 << 20, config=cfg)
    m.allocate_workspace(plan)
    info = m.muon_get_plan_info(plan)
    assert {m.muon_get_bucket_info(plan, b).ns_single_kernel for b in range(info.n_buckets)} == kinds

    # eager twin of the state, stepped alongside the replays
    eW = [t.clone() for t in wl.dW]
    eM = [t.clone() for t in wl.dM]
    eG = [t.clone() for t in wl.dG]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    W_start = [t.clone() for t in wl.dW]
    M_start = [t.clone() for t in wl.dM]
    captured_G = list(wl.dG)
    with torch.cuda.graph(graph, stream=side):
        m.muon_step(plan, wl.dW, captured_G, wl.dM, LR, MU, True, WD, NS, side)
    # capture enqueues nothing: the state is as before
    torch.cuda.synchronize()
    for a, b in zip(wl.dW, W_start):
        assert torch.equal(a, b)
    for a, b in zip(wl.dM, M_start):
        assert torch.equal(a, b)

    for step in range(3):
        if step > 0:
            wl.new_grads(step)          # fresh gradients, copied into the captured tensors
            for src, cap, eager in zip(wl.dG, captured_G, eG):
                cap.copy_(src)
                eager.copy_(src)
        W_prev = [to_numpy(t, wl.w_dtype) for t in eW]
        M_prev = [to_numpy(t, synth.F32) for t in eM]
        graph.replay()
        m.muon_step(plan, eW, eG, eM, LR, MU, True, WD, NS, torch.cuda.current_stream())
        torch.cuda.synchronize()
        st, nf = m.muon_sync(plan)
        assert st == m.MUON_OK and nf == 0
        for a, b in zip(wl.dW, eW):
            assert torch.equal(a, b)
        for a, b in zip(wl.dM, eM):
            assert torch.equal(a, b)
        W_new = [to_numpy(t, wl.w_dtype) for t in wl.dW]
        M_new = [to_numpy(t, synth.F32) for t in wl.dM]
        ulp, rel = check_step(wl, W_prev, M_prev, W_new, M_new, lr=LR, mu=MU, nesterov=True, wd=WD,
                              ns_steps=NS, method=method)
        assert ulp <= 1 and rel <= TOL_BF16
