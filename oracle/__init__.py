"""Plain fp64 CPU oracle of the Muon optimizer step (momentum -> Newton-Schulz -> apply).

TEST INFRASTRUCTURE.  Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU
baseline may import this package; the CUDA path never does, and this package
shares no code, table or constant generator with it.  Inputs come from the
seeded generator in ``synth`` (which holds none of the method's arithmetic).

Every function works on one logical 2-D matrix in float64 with numpy, using
``@`` (a library matmul) as the only primitive beyond elementwise arithmetic,
and follows the steps in the order the sources give them:

* core update -- "Muon Optimizer + FSDP", section 背景 (background):
  M_t = momentum_update(grad); U_t = NewtonSchulz(M_t); W_t = W_t - lr * U_t,
  applied to each full 2-D logical matrix, never to a row shard of it.
* Newton-Schulz -- DeepSpeed issue "[RFC] Enable Correct and High-Performance Muon
  Optimizer under ZeRO CPU Offload", section 2 (root cause): 5-6 quintic
  iterations on the full 2-D matrix.  The pages print neither the coefficients
  nor the iteration body; the reading used here, and stated where the
  workload is defined, is X <- a X + (b A + c A A) X with A = X X^T,
  (a, b, c) = (3.4445, -4.7750, 2.0315), after dividing by (||V||_F + eps),
  eps = 1e-7, on the wide orientation (transpose when rows > cols).
* momentum -- named but not written out on the pages ("momentum_update",
  "first-order momentum tracking"); the reading is the EMA form
  M <- mu M + (1 - mu) G with Nesterov blend V = (1 - mu) G + mu M_new,
  and the SGD form M <- mu M + G, V = G + mu M_new as an option.
* per-iteration coefficients -- DeepSpeed issue "[RFC] Enable Correct and
  High-Performance Muon Optimizer under ZeRO CPU Offload", follow-up list
  ("Polar Express" as an ns_method): iteration k may use its own (a_k, b_k, c_k);
  ``polar_express_schedule`` builds them by fitting, at each iteration, the odd
  quintic closest to 1 in the max norm on the interval holding the singular
  values, then carrying the interval forward (the pages give no coefficients).
* apply -- W <- W - lr (sqrt(max(1, rows/cols)) U + wd W), decoupled weight
  decay on the old W.
* fused tensors -- "Muon Optimizer + FSDP", section 分块通信 (chunked
  communication): qkv = [Q; K; V] and experts [E, out, in] are split into
  logical matrices before Muon; DeepSpeed issue #8463 section 4.D: per-head
  Muon on interleaved [Q0, K0, V0, Q1, ...] layouts runs one Newton-Schulz per
  head slice.

Pins (tests/test_oracle_pins.py, tests/test_oracle_schedule_pins.py) tie these
functions to mathematics that does not go through them: the SVD closed form of an odd matrix polynomial,
orthogonal equivariance, scale and transpose identities, per-shard vs whole
matrix, and closed forms of the momentum recursion.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Sequence, Tuple

import numpy as np

DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)
DEFAULT_EPS = 1e-7
DEFAULT_NS_STEPS = 5


# ---------------------------------------------------------------------------
# momentum ("Muon Optimizer + FSDP", 背景: M_t = momentum_update(grad))
# ---------------------------------------------------------------------------

def momentum_update(M, G, mu: float, form: str = "ema", one_minus_mu: float | None = None):
    """New fp32 momentum state.

    EMA form: M_new = mu * M + (1 - mu) * G; SGD form: M_new = mu * M + G.
    The sum is formed in float64 and stored as float32 (round to nearest even),
    because the momentum buffer is fp32 state.  ``one_minus_mu`` lets a caller
    give (1 - mu) as the exact constant another implementation uses.
    """
    M = np.asarray(M, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    mu = float(mu)
    if form == "ema":
        w = (1.0 - mu) if one_minus_mu is None else float(one_minus_mu)
        M_new = mu * M + w * G
    elif form == "sgd":
        M_new = mu * M + G
    else:
        raise ValueError(f"unknown momentum form {form!r}")
    return M_new.astype(np.float32)


def nesterov_blend(M_new, G, mu: float, nesterov: bool, form: str = "ema",
                   one_minus_mu: float | None = None) -> np.ndarray:
    """The matrix handed to Newton-Schulz, in float64.

    Without Nesterov it is the new momentum itself.  With Nesterov it looks one
    step ahead: (1 - mu) G + mu M_new (EMA form) or G + mu M_new (SGD form).
    """
    M_new = np.asarray(M_new, dtype=np.float64)
    if not nesterov:
        return M_new
    G = np.asarray(G, dtype=np.float64)
    mu = float(mu)
    if form == "ema":
        w = (1.0 - mu) if one_minus_mu is None else float(one_minus_mu)
        return w * G + mu * M_new
    if form == "sgd":
        return G + mu * M_new
    raise ValueError(f"unknown momentum form {form!r}")


# ---------------------------------------------------------------------------
# Newton-Schulz (DeepSpeed #8463 section 2; "Muon Optimizer + FSDP" 背景)
# ---------------------------------------------------------------------------

def orient(V: np.ndarray) -> Tuple[np.ndarray, bool]:
    """Wide orientation: transpose a tall matrix (rows > cols) so that rows <= cols."""
    V = np.asarray(V, dtype=np.float64)
    if V.shape[0] > V.shape[1]:
        return V.T, True
    return V, False


def frobenius_normalize(V: np.ndarray, eps: float = DEFAULT_EPS) -> np.ndarray:
    """X0 = V / (||V||_F + eps), the Frobenius norm summed over every element."""
    V = np.asarray(V, dtype=np.float64)
    norm = math.sqrt(float(np.sum(V * V)))
    return V / (norm + eps)


def ns_iteration(X: np.ndarray, a: float, b: float, c: float) -> np.ndarray:
    """One quintic step: A = X X^T, B = b A + c A A, X' = a X + B X."""
    A = X @ X.T
    B = b * A + c * (A @ A)
    return a * X + B @ X


def coefficient_schedule(coeffs, steps: int) -> List[Tuple[float, float, float]]:
    """The (a, b, c) of each of ``steps`` iterations: one triple used every time,
    or a per-iteration list of triples whose last entry repeats past its end."""
    flat = list(coeffs)
    if flat and not isinstance(flat[0], (tuple, list, np.ndarray)):
        triples = [tuple(float(v) for v in flat)]
    else:
        triples = [tuple(float(v) for v in t) for t in flat]
    if any(len(t) != 3 for t in triples) or not triples:
        raise ValueError("coefficients are (a, b, c) triples")
    return [triples[min(k, len(triples) - 1)] for k in range(int(steps))]


def newton_schulz(V, steps: int = DEFAULT_NS_STEPS, coeffs=DEFAULT_COEFFS,
                  eps: float = DEFAULT_EPS) -> np.ndarray:
    """Approximate orthogonal polar factor of the whole 2-D matrix V (fp64).

    Orient wide, normalise by the Frobenius norm, run ``steps`` quintic
    iterations, and undo the orientation.  ``coeffs`` is one (a, b, c) for every
    iteration or a per-iteration schedule (see ``coefficient_schedule``).
    """
    X, transposed = orient(V)
    X = frobenius_normalize(X, eps)
    for a, b, c in coefficient_schedule(coeffs, steps):
        X = ns_iteration(X, a, b, c)
    return X.T if transposed else X


# ---------------------------------------------------------------------------
# the "gram" Newton-Schulz method (DeepSpeed PR "[Muon] CPU offload: pin the
# momentum and overlap the host writeback", section Tests: per-head shard tests
# parametrised over "gram" and "standard"; DeepSpeed issue "[RFC] ... ZeRO CPU
# Offload", follow-up list: the gram method gives results that differ from the
# quintic iteration's in floating point)
# ---------------------------------------------------------------------------
# The pages name the method and say only that its results differ in floating
# point.  The reading taken here is the iteration rewritten on the Gram matrix:
# with X_{k+1} = Q_k X_k and Q_k = a I + b A_k + c A_k^2, A_k = X_k X_k^T, one has
# A_{k+1} = Q_k A_k Q_k (Q_k is symmetric) and X_K = (Q_{K-1} ... Q_0) X_0, so the
# whole iteration runs on m x m matrices between one product X_0 X_0^T and one
# final product R X_0.  In exact arithmetic it is the quintic iteration itself.
# A restart at iteration r forms X_r = R_r X_0 and A_r = X_r X_r^T afresh.

def newton_schulz_gram(V, steps: int = DEFAULT_NS_STEPS, coeffs=DEFAULT_COEFFS,
                       eps: float = DEFAULT_EPS, restarts=()) -> np.ndarray:
    """The Gram-form Newton-Schulz iteration of the whole 2-D matrix V (fp64).

    Orient wide, normalise by the Frobenius norm, A = X X^T, R = I; per iteration
    (a restart first when k is in ``restarts``: X = R X, A = X X^T, R = I)
    Q = a I + b A + c A A, A = Q A Q, R = Q R; finally U = R X, un-oriented."""
    X, transposed = orient(V)
    X = frobenius_normalize(X, eps)
    m = X.shape[0]
    A = X @ X.T
    R = np.eye(m)
    for k, (a, b, c) in enumerate(coefficient_schedule(coeffs, steps)):
        if k in restarts:
            X = R @ X
            A = X @ X.T
            R = np.eye(m)
        Q = a * np.eye(m) + b * A + c * (A @ A)
        A = Q @ A @ Q
        R = Q @ R
    U = R @ X
    return U.T if transposed else U


# ---------------------------------------------------------------------------
# per-iteration coefficients (DeepSpeed issue "[RFC] Enable Correct and
# High-Performance Muon Optimizer under ZeRO CPU Offload", follow-up list:
# Newton-Schulz with per-iteration optimised coefficients, "Polar Express",
# arXiv:2505.16932, as an ns_method option)
# ---------------------------------------------------------------------------
# The pages name the method and its aim -- fewer iterations to the same polar
# accuracy -- but print no coefficients.  The construction taken here is the
# plainest reading of "per-iteration optimised": iteration k uses the odd quintic
# p_k(x) = a x + b x^3 + c x^5 that minimises max |1 - p_k(x)| over the interval
# [l_k, u_k] known to hold the singular values, and the next interval is the
# image [1 - E_k, 1 + E_k] of that one (E_k the minimised error).  After the
# Frobenius normalisation u_0 = 1; l_0 is an assumed lower bound.

def minimax_odd_quintic(lo: float, hi: float, grid_points: int = 200001, max_iter: int = 60):
    """(a, b, c, E): the odd quintic closest to 1 in the max norm on [lo, hi].

    Exchange iteration on the three-function basis x, x^3, x^5: on a reference of
    four points solve p(x_i) + (-1)^i E = 1, then move the reference to the
    extrema of the error 1 - p found on a dense grid, until the largest error on
    the grid equals |E|.  E > 0 means the error is +|E| at ``lo``.
    """
    lo, hi = float(lo), float(hi)
    if not 0.0 < lo <= hi:
        raise ValueError("need 0 < lo <= hi")
    x = np.linspace(lo, hi, grid_points)
    if hi - lo < 1e-4:
        # the three basis functions are nearly dependent on so short an interval
        # (fits differ in their coefficients, not in their ~1e-13 errors); the
        # minimax quintic there tends to the one flat to third order at 1,
        # p(x) = (15 x - 10 x^3 + 3 x^5) / 8 (p(1) = 1, p'(1) = p''(1) = 0), whose
        # error on [1 - d, 1 + d] is about 2.5 d^3
        a, b, c = 15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0
        err = 1.0 - (a * x + b * x ** 3 + c * x ** 5)
        return a, b, c, float(err[np.argmax(np.abs(err))])
    ref = lo + (hi - lo) * (1.0 - np.cos(np.pi * np.arange(4) / 3.0)) / 2.0
    sign = (-1.0) ** np.arange(4)
    for _ in range(max_iter):
        sol = np.linalg.solve(np.column_stack([ref, ref ** 3, ref ** 5, sign]), np.ones(4))
        a, b, c, E = (float(v) for v in sol)
        err = 1.0 - (a * x + b * x ** 3 + c * x ** 5)
        # the error's local extrema on the grid, ends included
        d = np.diff(err)
        turn = np.where(np.sign(d[1:]) != np.sign(d[:-1]))[0] + 1
        idx = np.concatenate([[0], turn, [len(x) - 1]])
        # keep one point per run of equal sign: the largest magnitude
        pts = []
        for i in idx:
            if pts and np.sign(err[i]) == np.sign(err[pts[-1]]):
                if abs(err[i]) > abs(err[pts[-1]]):
                    pts[-1] = i
            else:
                pts.append(i)
        while len(pts) > 4:  # drop the smaller end
            pts.pop(0 if abs(err[pts[0]]) < abs(err[pts[-1]]) else -1)
        if len(pts) < 4:
            raise RuntimeError("the error does not alternate four times")
        # sharpen interior extrema with Newton steps on p'(x) = a + 3 b x^2 + 5 c x^4
        ref = x[pts].copy()
        for i in range(1, 3):
            t = ref[i]
            for _ in range(8):
                d1 = a + 3 * b * t * t + 5 * c * t ** 4
                d2 = 6 * b * t + 20 * c * t ** 3
                if d2 == 0.0:
                    break
                t = min(max(t - d1 / d2, lo), hi)
            ref[i] = t
        e_ref = 1.0 - (a * ref + b * ref ** 3 + c * ref ** 5)
        sign = np.sign(e_ref)
        worst = max(float(np.max(np.abs(err))), float(np.max(np.abs(e_ref))))
        if worst - abs(E) <= 1e-14 * max(1.0, abs(E)):
            break
    # report the largest error actually reached, so that the next interval holds
    # the image of this one
    return a, b, c, math.copysign(worst, E)


def polar_express_schedule(n_iters: int, lower: float = 1e-3, safety: float = 1.0):
    """Per-iteration (a, b, c) for ``n_iters`` iterations and the bound E_k after
    each: iteration k fits [l_k, u_k * safety] (safety >= 1 leaves room for
    rounding that pushes a singular value past u_k); then [l, u] = [1 - E, 1 + E]."""
    lo, hi = float(lower), 1.0
    coeffs, errs = [], []
    for _ in range(int(n_iters)):
        a, b, c, E = minimax_odd_quintic(lo, hi * float(safety))
        coeffs.append((a, b, c))
        errs.append(abs(E))
        lo, hi = 1.0 - abs(E), 1.0 + abs(E)
    return coeffs, errs


# ---------------------------------------------------------------------------
# apply ("Muon Optimizer + FSDP", 背景: W_t = W_t - lr * U_t)
# ---------------------------------------------------------------------------

def shape_scale(rows: int, cols: int) -> float:
    """sqrt(max(1, rows / cols)) for the ORIGINAL (un-oriented) logical shape."""
    return math.sqrt(max(1.0, float(rows) / float(cols)))


def apply_update(W, U, lr: float, wd: float = 0.0) -> np.ndarray:
    """W - lr * (sqrt(max(1, rows/cols)) * U + wd * W), with the old W in the decay term."""
    W = np.asarray(W, dtype=np.float64)
    U = np.asarray(U, dtype=np.float64)
    rows, cols = W.shape
    return W - float(lr) * (shape_scale(rows, cols) * U + float(wd) * W)


def offload_update(U, rows: int, cols: int) -> np.ndarray:
    """The update sent back to the host in the offload layout: sqrt(max(1, rows/cols)) * U."""
    return shape_scale(rows, cols) * np.asarray(U, dtype=np.float64)


def muon_matrix_step(W, M, G, lr: float, mu: float, nesterov: bool = True, wd: float = 0.0,
                     ns_steps: int = DEFAULT_NS_STEPS, coeffs: Sequence[float] = DEFAULT_COEFFS,
                     eps: float = DEFAULT_EPS, form: str = "ema",
                     one_minus_mu: float | None = None, method: str = "standard"):
    """One Muon step of one logical matrix.

    Returns (W_new fp64, M_new fp32, U fp64).  The caller rounds W_new to the
    storage dtype of its weights.  ``method``: "standard" (the quintic iteration on
    X) or "gram" (the same iteration on the Gram matrix, newton_schulz_gram).
    """
    M_new = momentum_update(M, G, mu, form, one_minus_mu)
    V = nesterov_blend(M_new, G, mu, nesterov, form, one_minus_mu)
    if method == "gram":
        U = newton_schulz_gram(V, ns_steps, coeffs, eps)
    elif method == "standard":
        U = newton_schulz(V, ns_steps, coeffs, eps)
    else:
        raise ValueError(f"unknown Newton-Schulz method {method!r}")
    W_new = apply_update(W, U, lr, wd)
    return W_new, M_new, U


# ---------------------------------------------------------------------------
# logical matrices of fused tensors ("Muon Optimizer + FSDP", 分块通信;
# DeepSpeed #8463 section 4.D)
# ---------------------------------------------------------------------------

def logical_matrices(flat: np.ndarray, rows: int, cols: int, count: int,
                     stride: int | None = None) -> List[np.ndarray]:
    """Views of ``count`` logical rows x cols matrices laid out ``stride`` elements apart."""
    flat = np.asarray(flat).reshape(-1)
    stride = rows * cols if not stride else int(stride)
    return [flat[i * stride: i * stride + rows * cols].reshape(rows, cols) for i in range(count)]


def split_experts(T: np.ndarray) -> List[np.ndarray]:
    """[E, out, in] expert tensor -> E separate out x in matrices."""
    return [T[e] for e in range(T.shape[0])]


def split_heads(T: np.ndarray, head_rows: int) -> List[np.ndarray]:
    """Fused [H * head_rows, in] projection -> H head slices of head_rows rows each."""
    if T.shape[0] % head_rows:
        raise ValueError("rows are not a whole number of heads")
    return [T[h * head_rows:(h + 1) * head_rows] for h in range(T.shape[0] // head_rows)]


def interleaved_qkv_labels(n_kv_groups: int, q_per_group: int) -> List[str]:
    """Head labels of the interleaved layout [Q0..Q(g-1), K0, V0, Qg.., K1, V1, ...]."""
    labels = []
    for g in range(n_kv_groups):
        labels += [f"Q{g * q_per_group + i}" for i in range(q_per_group)]
        labels += [f"K{g}", f"V{g}"]
    return labels


def per_head_newton_schulz(T: np.ndarray, head_rows: int, **ns_kwargs) -> np.ndarray:
    """Per-head Muon: one Newton-Schulz per head slice, reassembled in place."""
    return np.concatenate([newton_schulz(h, **ns_kwargs) for h in split_heads(T, head_rows)], 0)


def muon_step(params: Iterable[np.ndarray], grads: Iterable[np.ndarray],
              momenta: Iterable[np.ndarray], shapes: Iterable[Tuple[int, int, int, int]],
              lr: float, mu: float, nesterov: bool = True, wd: float = 0.0,
              ns_steps: int = DEFAULT_NS_STEPS, coeffs: Sequence[float] = DEFAULT_COEFFS,
              eps: float = DEFAULT_EPS, form: str = "ema"):
    """Muon step over tensors, each holding ``count`` logical matrices.

    params/grads/momenta are flat float arrays (fp64-widened by the caller);
    shapes are (rows, cols, count, stride).  Returns new (params fp64, momenta fp32)
    lists.  Matrices are independent, so the order of this loop changes nothing.
    """
    out_w, out_m = [], []
    for W, G, M, (rows, cols, count, stride) in zip(params, grads, momenta, shapes):
        Wn = np.array(W, dtype=np.float64).reshape(-1)
        Mn = np.array(M, dtype=np.float32).reshape(-1)
        stride = rows * cols if not stride else stride
        for i in range(count):
            sl = slice(i * stride, i * stride + rows * cols)
            w_new, m_new, _ = muon_matrix_step(
                Wn[sl].reshape(rows, cols), Mn[sl].reshape(rows, cols),
                np.asarray(G, dtype=np.float64).reshape(-1)[sl].reshape(rows, cols),
                lr, mu, nesterov, wd, ns_steps, coeffs, eps, form)
            Wn[sl] = w_new.reshape(-1)
            Mn[sl] = m_new.reshape(-1)
        out_w.append(Wn)
        out_m.append(Mn)
    return out_w, out_m
