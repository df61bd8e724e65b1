"""Helpers of the GPU parity tests: seeded inputs on both sides, teacher-forced oracle
comparison per logical matrix, and the error measures the tolerances apply to."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# per-matrix tolerances (relative Frobenius error of the update)
TOL_BF16 = 3e-2
TOL_TF32X3 = 1e-4


def nsm():
    import newton_schulz_muon_gb300.build as b
    b.build()
    import newton_schulz_muon_gb300 as m
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
               coeffs=oracle.DEFAULT_COEFFS, eps=1e-7, form="ema", tol=TOL_BF16, sample=None):
    """Teacher-forced comparison of one GPU step against the oracle, per logical matrix.

    W_prev/M_prev are the host copies of the state the GPU started from; W_new/M_new
    what it produced.  Returns the worst (ulp, rel) seen; asserts the tolerances.
    """
    mu32, omu = oracle_constants(mu, form)
    c32 = tuple(f32(v) for v in coeffs)
    worst_ulp, worst_rel = 0, 0.0
    for i, (r, c, k) in enumerate(wl.shapes):
        idx = range(k) if sample is None else sample(i, k)
        for j in idx:
            Wp = widen(W_prev[i][j], wl.w_dtype)
            Mp = M_prev[i][j]
            G = widen(wl.G[i][j], wl.g_dtype)
            Wo, Mo, U = oracle.muon_matrix_step(Wp, Mp, G, f32(lr), mu32, nesterov, f32(wd), ns_steps,
                                                c32, f32(eps), form, one_minus_mu=omu)
            ulp = int(ulp_distance(M_new[i][j], Mo).max())
            assert ulp <= 1, f"tensor {i} matrix {j}: momentum differs by {ulp} ulp"
            dW_gpu = widen(W_new[i][j], wl.w_dtype) - Wp
            dW_or = Wo - Wp
            rel = rel_fro(dW_gpu, dW_or)
            allowed = tol
            if wl.w_dtype == synth.BF16:
                # the stored weight is rounded to bf16: half an ulp of bf16 per element
                ulp16 = np.abs(Wo) * 2.0 ** -8
                allowed = tol + float(np.linalg.norm(0.5 * ulp16) / max(np.linalg.norm(dW_or), 1e-30))
            assert rel <= allowed, f"tensor {i} matrix {j} ({r}x{c}): rel update error {rel:.3e} > {allowed:.1e}"
            worst_ulp = max(worst_ulp, ulp)
            worst_rel = max(worst_rel, rel)
    return worst_ulp, worst_rel
