"""Helpers of the GPU parity tests: seeded inputs on both sides, teacher-forced oracle
comparison per logical matrix, and the error measures the tolerances apply to."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# per-matrix tolerances (relative Frobenius error of the update)
TOL_BF16 = 3e-2
TOL_TF32X3 = 1e-4
# bf16 weights: the most the bf16-weight bound may allow, over ||dW||, in the tests
# built to discriminate (W0 = 0, or an lr at which the update dominates the bf16
# rounding of W): the 3e-2 tolerance plus at most 0.5e-2 of rounding allowance
TOL_BF16_W = 3.5e-2


def nsm():
    """The binding, built; with MUON_TEST_DEBUG_LIB=1 in the environment every test
    runs against the debug build (device range checks) instead."""
    import os
    import newton_schulz_muon_gb300.build as b
    b.build()
    import newton_schulz_muon_gb300 as m
    if os.environ.get("MUON_TEST_DEBUG_LIB") == "1" and m._LIB is None:
        m.use_debug_library(True)
    return m


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in fp32 units in the last place, via the ordered integer encoding."""
    ai = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ai = np.where(ai < 0, -(ai & 0x7FFFFFFF), ai)
    bi = np.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    return np.abs(ai - bi)


def rel_fro(x: np.ndarray, ref: np.ndarray) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x))


def f32(x):
    return float(np.float32(x))


def f32_coeffs(coeffs):
    """One (a, b, c) or a per-iteration list of them, as the fp32 values the GPU uses."""
    flat = list(coeffs)
    if flat and isinstance(flat[0], (tuple, list, np.ndarray)):
        return [tuple(f32(v) for v in t) for t in flat]
    return tuple(f32(v) for v in flat)


def oracle_constants(mu: float, form: str):
    """mu and (1 - mu) exactly as the kernels use them (fp32 values)."""
    mu32 = np.float32(mu)
    omu = 1.0 if form == "sgd" else float(np.float32(1.0) - mu32)
    return float(mu32), omu


def torch_from(arr: np.ndarray, dtype_code: int):
    """numpy fp32 array or bf16 bit array -> torch CUDA tensor."""
    import torch
    if dtype_code == synth.BF16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def to_numpy(t, dtype_code: int) -> np.ndarray:
    import torch
    if dtype_code == synth.BF16:
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().float().cpu().numpy()


def widen(arr: np.ndarray, dtype_code: int) -> np.ndarray:
    return synth.as_f64(arr, dtype_code)


class Workload:
    """Tensors (rows, cols, count) with seeded W, M, G on the host and the device."""

    def __init__(self, shapes, *, w_sigma=0.02, m_sigma=0.0, g_sigma=1.0, g_dtype=synth.BF16,
                 w_dtype=synth.F32, seed=synth.SEED, step=0):
        self.shapes = [tuple(s) + (1,) * (3 - len(s)) for s in shapes]
        self.g_dtype, self.w_dtype = g_dtype, w_dtype
        self.g_sigma = g_sigma
        self.seed = seed
        self.W, self.M, self.G = [], [], []
        for i, (r, c, k) in enumerate(self.shapes):
            n = (k, r, c)
            if w_sigma > 0:
                self.W.append(synth.tensor(seed, synth.stream_id(i, synth.ROLE_W), 0, n, w_sigma, w_dtype))
            else:
                self.W.append(np.zeros(n, np.uint16 if w_dtype == synth.BF16 else np.float32))
            if m_sigma > 0:
                self.M.append(synth.tensor(seed, synth.stream_id(i, synth.ROLE_M), 0, n, m_sigma, synth.F32))
            else:
                self.M.append(np.zeros(n, np.float32))
            self.G.append(self.grad(i, step))
        self.dW = [torch_from(w, w_dtype) for w in self.W]
        self.dM = [torch_from(m, synth.F32) for m in self.M]
        self.dG = [torch_from(g, g_dtype) for g in self.G]

    def grad(self, i, step):
        r, c, k = self.shapes[i]
        return synth.tensor(self.seed, synth.stream_id(i, synth.ROLE_G), step, (k, r, c), self.g_sigma,
                            self.g_dtype)

    def new_grads(self, step):
        self.G = [self.grad(i, step) for i in range(len(self.shapes))]
        self.dG = [torch_from(g, self.g_dtype) for g in self.G]

    def plan_shapes(self):
        return [(r, c, k, 0) for (r, c, k) in self.shapes]


def check_step(wl: Workload, W_prev, M_prev, W_new, M_new, *, lr, mu, nesterov, wd, ns_steps,
               coeffs=oracle.DEFAULT_COEFFS, eps=1e-7, form="ema", tol=TOL_BF16, sample=None,
               bf16_max_bound=None, method="standard"):
    """Teacher-forced comparison of one GPU step against the oracle, per logical matrix.

    W_prev/M_prev are the host copies of the state the GPU started from; W_new/M_new
    what it produced.  Returns the worst (ulp, rel) seen; asserts the tolerances.
    bf16 weights: ``bf16_max_bound`` also asserts that the bound applied stays
    within that fraction of ||dW|| (the test discriminates), and rel is then the
    measured error over ||dW||.
    """
    mu32, omu = oracle_constants(mu, form)
    c32 = f32_coeffs(coeffs)
    worst_ulp, worst_rel = 0, 0.0
    for i, (r, c, k) in enumerate(wl.shapes):
        idx = range(k) if sample is None else sample(i, k)
        for j in idx:
            Wp = widen(W_prev[i][j], wl.w_dtype)
            Mp = M_prev[i][j]
            G = widen(wl.G[i][j], wl.g_dtype)
            Wo, Mo, U = oracle.muon_matrix_step(Wp, Mp, G, f32(lr), mu32, nesterov, f32(wd), ns_steps,
                                                c32, f32(eps), form, one_minus_mu=omu, method=method)
            ulp = int(ulp_distance(M_new[i][j], Mo).max())
            assert ulp <= 1, f"tensor {i} matrix {j}: momentum differs by {ulp} ulp"
            if wl.w_dtype == synth.BF16:
                rel = bf16_weight_check(W_new[i][j], Wo, Wp, tol, bf16_max_bound)
                if bf16_max_bound is None:
                    rel = 0.0
            else:
                rel = rel_fro(widen(W_new[i][j], wl.w_dtype) - Wp, Wo - Wp)
                assert rel <= tol, f"tensor {i} matrix {j} ({r}x{c}): rel update error {rel:.3e} > {tol:.1e}"
            worst_ulp = max(worst_ulp, ulp)
            worst_rel = max(worst_rel, rel)
    return worst_ulp, worst_rel


def bf16_weight_check(W_new_bits, Wo, Wp, tol, max_bound=None):
    """bf16 weights: W_new = bf16(W_or + d) with ||d|| <= tol ||dW_or||, so
    ||W_new - W_or|| <= tol ||dW_or|| + || |W_or| 2^-8 || (a bf16 half-ulp is at most
    2^-8 of the value).  Returns the measured left side over ||dW_or||.
    ``max_bound``: also assert that the bound is at most that fraction of
    ||dW_or||, i.e. that the rounding allowance does not swamp the tolerance."""
    err = np.linalg.norm(synth.as_f64(W_new_bits, synth.BF16) - Wo)
    den = max(np.linalg.norm(Wo - Wp), 1e-30)
    bound = tol * den + np.linalg.norm(np.abs(Wo) * 2.0 ** -8)
    assert err <= bound, f"bf16 weights: error {err:.3e} above the bound {bound:.3e}"
    if max_bound is not None:
        assert bound <= max_bound * den, \
            f"bf16 weights: the bound {bound / den:.3e} of ||dW|| is looser than {max_bound:.1e}"
    return float(err / den)


def run_steps(m, wl, *, lr=0.02, mu=0.95, nesterov=True, wd=0.0, ns_steps=5, cap=512 << 20, cfg=None,
              steps=1, form="ema", coeffs=oracle.DEFAULT_COEFFS, sample=None, tol=TOL_BF16,
              schedule=None, bf16_max_bound=None, method="standard"):
    """Run `steps` GPU Muon steps on a Workload, checking each against the oracle.
    ``schedule``: per-iteration (a, b, c) set on the plan (and used by the oracle)
    in place of ``coeffs``."""
    import torch
    cfg = cfg or m.muon_config_default()
    cfg.grad_dtype = wl.g_dtype
    cfg.param_dtype = wl.w_dtype
    cfg.momentum_form = m.MUON_MOMENTUM_SGD if form == "sgd" else m.MUON_MOMENTUM_EMA
    cfg.ns_a, cfg.ns_b, cfg.ns_c = coeffs
    plan = m.muon_plan(wl.plan_shapes(), bucket_cap_bytes=cap, config=cfg)
    m.allocate_workspace(plan)
    if schedule is not None:
        m.muon_set_ns_schedule(plan, schedule)
        coeffs = schedule
    worst = (0, 0.0)
    for step in range(steps):
        if step > 0:
            wl.new_grads(step)
        W_prev = [to_numpy(t, wl.w_dtype) for t in wl.dW]
        M_prev = [to_numpy(t, synth.F32) for t in wl.dM]
        m.muon_step(plan, wl.dW, wl.dG, wl.dM, lr, mu, nesterov, wd, ns_steps)
        st, nf = m.muon_sync(plan)
        assert st == m.MUON_OK and nf == 0
        torch.cuda.synchronize()
        W_new = [to_numpy(t, wl.w_dtype) for t in wl.dW]
        M_new = [to_numpy(t, synth.F32) for t in wl.dM]
        u, r = check_step(wl, W_prev, M_prev, W_new, M_new, lr=lr, mu=mu, nesterov=nesterov, wd=wd,
                          ns_steps=ns_steps, coeffs=coeffs, form=form, sample=sample, tol=tol,
                          bf16_max_bound=bf16_max_bound, method=method)
        worst = (max(worst[0], u), max(worst[1], r))
    return worst


def device_tensor(shape, dtype_code, seed, stream, step, sigma):
    """A seeded tensor filled on the device (bit-identical to synth.tensor)."""
    import torch
    dt = torch.bfloat16 if dtype_code == synth.BF16 else torch.float32
    t = torch.empty(shape, dtype=dt, device="cuda")
    if sigma > 0:
        synth.fill_normal_cuda(t, seed, stream, step, sigma)
    else:
        t.zero_()
    return t


def host_matrix(shape_rc, index, dtype_code, seed, stream, step, sigma):
    """Matrix `index` of a [count, rows, cols] seeded tensor, generated on the CPU."""
    r, c = shape_rc
    if sigma <= 0:
        return np.zeros((r, c), np.uint16 if dtype_code == synth.BF16 else np.float32)
    return synth.tensor(seed, stream, step, (r, c), sigma, dtype_code, start=index * r * c)


def check_matrix(W_prev, M_prev, G, W_new, M_new, *, w_dtype, g_dtype, lr, mu, nesterov=True, wd=0.0,
                 ns_steps=5, form="ema", tol=TOL_BF16, bf16_max_bound=None):
    """Teacher-forced oracle comparison of one logical matrix; returns (ulp, rel)."""
    mu32, omu = oracle_constants(mu, form)
    c32 = tuple(f32(v) for v in oracle.DEFAULT_COEFFS)
    Wp = widen(W_prev, w_dtype)
    Wo, Mo, _ = oracle.muon_matrix_step(Wp, M_prev, widen(G, g_dtype), f32(lr), mu32, nesterov, f32(wd),
                                        ns_steps, c32, f32(1e-7), form, one_minus_mu=omu)
    ulp = int(ulp_distance(M_new, Mo).max())
    assert ulp <= 1, f"momentum differs by {ulp} ulp"
    if w_dtype == synth.BF16:
        rel = bf16_weight_check(W_new, Wo, Wp, tol, bf16_max_bound)
        return ulp, (rel if bf16_max_bound is not None else 0.0)
    rel = rel_fro(widen(W_new, w_dtype) - Wp, Wo - Wp)
    assert rel <= tol, f"rel update error {rel:.3e} > {tol:.2e}"
    return ulp, rel
