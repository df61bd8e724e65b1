"""Pins of the fp64 oracle to mathematics that does not go through it.

Each test would fail on a plausible mistake in the oracle: a dropped or
mis-signed polynomial term, a transposed operand, the wrong orientation rule,
eps in the wrong place, a wrong scale, or a momentum recursion off by a factor.
"""
import math

import numpy as np
import pytest

import oracle

# Coefficients and eps as stated for the 256x512 single-matrix workload
# (quintic (a, b, c) after Frobenius normalisation with eps 1e-7).
A_, B_, C_ = 3.4445, -4.7750, 2.0315
EPS = 1e-7


def _p_iter(x, steps):
    """Scalar odd quintic applied `steps` times (acts on singular values)."""
    for _ in range(steps):
        x = A_ * x + B_ * x ** 3 + C_ * x ** 5
    return x


def _closed_form(V, steps=5, eps=EPS):
    """NS via the SVD: X = P diag(s) Q^T  ->  P diag(p^steps(s / (||s||_2 + eps))) Q^T."""
    P, s, Qt = np.linalg.svd(V, full_matrices=False)
    fro = math.sqrt(float(np.sum(s ** 2)))
    return (P * _p_iter(s / (fro + eps), steps)) @ Qt


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _orthogonal(n, seed):
    q, r = np.linalg.qr(_rand((n, n), seed))
    return q * np.sign(np.diag(r))


@pytest.mark.parametrize("shape", [(3, 5), (8, 8), (17, 4), (64, 128), (1, 7), (9, 1), (40, 24)])
@pytest.mark.parametrize("steps", [0, 1, 5])
def test_svd_closed_form(shape, steps):
    V = _rand(shape, 100 + shape[0] * 7 + shape[1])
    U = oracle.newton_schulz(V, steps=steps, coeffs=(A_, B_, C_), eps=EPS)
    assert U.shape == V.shape
    assert _rel(U, _closed_form(V, steps)) < 1e-12


def test_closed_form_with_eps_on_the_norm_not_its_square():
    # tiny matrix: eps is not negligible against the norm, so where eps sits matters
    V = 1e-6 * _rand((4, 6), 3)
    U = oracle.newton_schulz(V)
    assert _rel(U, _closed_form(V)) < 1e-12
    P, s, Qt = np.linalg.svd(V, full_matrices=False)
    wrong = (P * _p_iter(s / math.sqrt(float(np.sum(s ** 2)) + EPS ** 2), 5)) @ Qt
    assert _rel(U, wrong) > 1e-3


def test_polar_band():
    # prescribed normalised singular values >= 0.01 land in the band the quintic reaches
    m, n = 6, 20
    s = np.array([1.0, 0.7, 0.4, 0.2, 0.1, 0.05])
    P, Q = _orthogonal(m, 1), _orthogonal(n, 2)[:m]
    V = (P * s) @ Q
    x = s / np.linalg.norm(s)
    assert x.min() >= 0.01
    sv = np.linalg.svd(oracle.newton_schulz(V), compute_uv=False)
    assert sv.min() >= 0.68 and sv.max() <= 1.135


@pytest.mark.parametrize("c", [1e-3, 7.0, 1e4])
def test_scale_invariance(c):
    V = _rand((12, 30), 5)
    assert _rel(oracle.newton_schulz(c * V, eps=0.0), oracle.newton_schulz(V, eps=0.0)) < 1e-12
    # with eps the difference is of order eps / ||V||
    d = _rel(oracle.newton_schulz(c * V), oracle.newton_schulz(V))
    assert d < 1e-5 * max(1.0, 1.0 / c)


@pytest.mark.parametrize("shape", [(10, 10), (7, 19), (19, 7)])
def test_transpose_identity(shape):
    V = _rand(shape, 9)
    assert _rel(oracle.newton_schulz(V.T), oracle.newton_schulz(V).T) < 1e-12


def test_row_and_column_permutation_equivariance():
    V = _rand((11, 23), 10)
    rp = np.random.default_rng(11).permutation(11)
    cp = np.random.default_rng(12).permutation(23)
    U = oracle.newton_schulz(V)
    assert _rel(oracle.newton_schulz(V[rp]), U[rp]) < 1e-12
    assert _rel(oracle.newton_schulz(V[:, cp]), U[:, cp]) < 1e-12


def test_orthogonal_equivariance():
    V = _rand((9, 14), 13)
    Q1, Q2 = _orthogonal(9, 14), _orthogonal(14, 15)
    assert _rel(oracle.newton_schulz(Q1 @ V @ Q2), Q1 @ oracle.newton_schulz(V) @ Q2) < 1e-11


def test_per_shard_is_not_whole_matrix():
    # NS([W_top; W_bottom]) != [NS(W_top); NS(W_bottom)]: block-wise Muon is another optimizer
    V = _rand((16, 40), 20)
    whole = oracle.newton_schulz(V)
    blocks = np.concatenate([oracle.newton_schulz(V[:8]), oracle.newton_schulz(V[8:])], 0)
    assert _rel(blocks, whole) > 0.05
    # a fused [Q; K; V] tensor split into its logical matrices is not the fused NS either
    qkv = _rand((24, 40), 21)
    split = np.concatenate([oracle.newton_schulz(t) for t in oracle.split_heads(qkv, 8)], 0)
    assert _rel(split, oracle.newton_schulz(qkv)) > 0.05


def test_per_head_on_a_shard_is_the_shard_of_per_head():
    T = _rand((6 * 4, 12), 22)           # 6 heads of 4 rows
    full = oracle.per_head_newton_schulz(T, 4)
    shard = T[8:16]                        # heads 2 and 3, whole heads only
    assert np.array_equal(oracle.per_head_newton_schulz(shard, 4), full[8:16])


def test_orthonormal_rows_special_case():
    m, n, k = 5, 12, 3.0
    Q = _orthogonal(n, 30)[:m]             # Q Q^T = I
    U = oracle.newton_schulz(k * Q)
    x = k / (k * math.sqrt(m) + EPS)
    assert _rel(U, _p_iter(x, 5) * Q) < 1e-13


def test_single_row():
    v = _rand((1, 33), 31)
    nv = float(np.sqrt(np.sum(v ** 2)))
    U = oracle.newton_schulz(v)
    assert _rel(U, _p_iter(nv / (nv + EPS), 5) * v / nv) < 1e-13


def test_zero_matrix():
    U = oracle.newton_schulz(np.zeros((4, 9)))
    assert np.all(U == 0.0)


def test_brute_force_one_iteration_tiny():
    X = np.array([[1.0, 2.0, -1.0], [0.5, 0.0, 3.0]])
    m, n = X.shape
    A = [[sum(X[i, k] * X[j, k] for k in range(n)) for j in range(m)] for i in range(m)]
    AA = [[sum(A[i][k] * A[k][j] for k in range(m)) for j in range(m)] for i in range(m)]
    B = [[B_ * A[i][j] + C_ * AA[i][j] for j in range(m)] for i in range(m)]
    ref = np.array([[A_ * X[i, j] + sum(B[i][k] * X[k, j] for k in range(m))
                     for j in range(n)] for i in range(m)])
    assert _rel(oracle.ns_iteration(X, A_, B_, C_), ref) < 1e-14


def test_p_of_one():
    # the quintic's value at 1 with these coefficients
    assert abs(_p_iter(1.0, 1) - 0.701) < 1e-12
    U = oracle.newton_schulz(np.array([[1.0]]), steps=1, eps=0.0)
    assert abs(U[0, 0] - 0.701) < 1e-12


# --- momentum -------------------------------------------------------------

@pytest.mark.parametrize("mu", [0.95, 0.9, 0.5])
def test_momentum_constant_gradient_from_zero(mu):
    G = _rand((3, 7), 40).astype(np.float32)
    M = np.zeros_like(G)
    Ms = np.zeros_like(G)
    for k in range(1, 8):
        M = oracle.momentum_update(M, G, mu, "ema")
        Ms = oracle.momentum_update(Ms, G, mu, "sgd")
        assert _rel(M.astype(np.float64), (1 - mu ** k) * G.astype(np.float64)) < 1e-6
        assert _rel(Ms.astype(np.float64), (1 - mu ** k) / (1 - mu) * G.astype(np.float64)) < 1e-6
    assert M.dtype == np.float32


def test_momentum_zero_gradient_decays_geometrically():
    M0 = _rand((4, 4), 41).astype(np.float32)
    M = M0
    for k in range(1, 6):
        M = oracle.momentum_update(M, np.zeros_like(M0), 0.95)
        assert _rel(M.astype(np.float64), 0.95 ** k * M0.astype(np.float64)) < 1e-6


def test_nesterov_blend_values():
    G = np.full((2, 2), 2.0)
    Mn = np.full((2, 2), 4.0, dtype=np.float32)
    assert np.allclose(oracle.nesterov_blend(Mn, G, 0.9, True, "ema"), 0.1 * 2 + 0.9 * 4)
    assert np.allclose(oracle.nesterov_blend(Mn, G, 0.9, True, "sgd"), 2 + 0.9 * 4)
    assert np.allclose(oracle.nesterov_blend(Mn, G, 0.9, False, "ema"), 4.0)


def test_ema_and_sgd_forms_give_the_same_weights_from_zero_init():
    # V_ema = (1 - mu) V_sgd by induction, and NS is scale invariant up to eps
    W0 = 0.02 * _rand((6, 10), 50)
    We, Ws = W0.copy(), W0.copy()
    Me = np.zeros((6, 10), np.float32)
    Msg = np.zeros((6, 10), np.float32)
    for step in range(3):
        G = _rand((6, 10), 60 + step).astype(np.float32)
        We, Me, _ = oracle.muon_matrix_step(We, Me, G, 0.02, 0.95, True, 0.0, form="ema")
        Ws, Msg, _ = oracle.muon_matrix_step(Ws, Msg, G, 0.02, 0.95, True, 0.0, form="sgd")
    assert _rel(We - W0, Ws - W0) < 1e-5


# --- apply ------------------------------------------------------------------

def test_shape_scale_uses_original_shape():
    assert oracle.shape_scale(9728, 2560) == pytest.approx(1.949358868961793, abs=1e-15)
    assert oracle.shape_scale(2048, 768) == pytest.approx(1.632993161855452, abs=1e-15)
    assert oracle.shape_scale(2560, 9728) == 1.0
    assert oracle.shape_scale(64, 64) == 1.0


def test_apply_update_terms():
    W = np.full((4, 2), 2.0)               # tall: scale sqrt(2)
    U = np.full((4, 2), 0.5)
    out = oracle.apply_update(W, U, lr=0.1, wd=0.0)
    assert np.allclose(out, 2.0 - 0.1 * math.sqrt(2.0) * 0.5, rtol=0, atol=1e-15)
    out = oracle.apply_update(W, U, lr=0.1, wd=0.3)
    assert np.allclose(out, 2.0 - 0.1 * (math.sqrt(2.0) * 0.5 + 0.3 * 2.0), rtol=0, atol=1e-15)


def test_offload_update_on_a_tall_matrix():
    # the offload writeback U' = sqrt(max(1, rows/cols)) U: a 32 x 8 matrix (rows =
    # 4 cols) takes the factor 2, its 8 x 32 transpose and a square one take 1; the
    # singular values of U' of a tall V are 2 p^5(s / (||s|| + eps)) (SVD closed
    # form); and the host applying W - lr (U' + wd W) lands where apply_update does
    V = _rand((32, 8), 80)
    U = oracle.newton_schulz(V)
    Up = oracle.offload_update(U, 32, 8)
    assert np.array_equal(Up, 2.0 * U)
    assert np.array_equal(oracle.offload_update(U.T, 8, 32), U.T)
    Q = _rand((6, 6), 81)
    assert np.array_equal(oracle.offload_update(Q, 6, 6), Q)
    s = np.linalg.svd(V, compute_uv=False)
    want = 2.0 * _p_iter(s / (math.sqrt(float(np.sum(s ** 2))) + EPS), 5)
    got = np.linalg.svd(Up, compute_uv=False)
    assert np.allclose(np.sort(got), np.sort(np.abs(want)), rtol=1e-12, atol=0)
    W = 0.02 * _rand((32, 8), 82)
    lr, wd = 0.02, 0.1
    host = W - lr * (Up + wd * W)
    assert _rel(host, oracle.apply_update(W, U, lr, wd)) < 1e-15
    assert _rel(host, W - lr * (2.0 * U + wd * W)) < 1e-15


def test_full_step_composes_the_parts():
    W = 0.02 * _rand((5, 8), 70)
    M = 0.02 * _rand((5, 8), 71).astype(np.float32)
    G = _rand((5, 8), 72).astype(np.float32)
    W1, M1, U = oracle.muon_matrix_step(W, M, G, 0.02, 0.95, True, 0.01)
    M_ref = (0.95 * M.astype(np.float64) + (1 - 0.95) * G.astype(np.float64)).astype(np.float32)
    assert np.array_equal(M1, M_ref)
    V = (1 - 0.95) * G.astype(np.float64) + 0.95 * M_ref.astype(np.float64)
    assert _rel(U, _closed_form(V)) < 1e-12
    assert _rel(W1, W - 0.02 * (U + 0.01 * W)) < 1e-15


# --- fused tensors ----------------------------------------------------------

def test_split_experts_and_logical_views():
    T = np.arange(3 * 4 * 5, dtype=np.float64).reshape(3, 4, 5)
    ex = oracle.split_experts(T)
    views = oracle.logical_matrices(T.reshape(-1), 4, 5, 3)
    for e in range(3):
        assert np.array_equal(ex[e], T[e]) and np.array_equal(views[e], T[e])
    strided = oracle.logical_matrices(np.arange(50.0), 2, 3, 4, stride=12)
    assert np.array_equal(strided[2], np.arange(24.0, 30.0).reshape(2, 3))


def test_interleaved_qkv_labels():
    lab = oracle.interleaved_qkv_labels(8, 4)
    assert len(lab) == 48
    assert lab[:6] == ["Q0", "Q1", "Q2", "Q3", "K0", "V0"]
    assert lab[6:12] == ["Q4", "Q5", "Q6", "Q7", "K1", "V1"]
    assert lab[-2:] == ["K7", "V7"]


def test_muon_step_over_tensors_matches_per_matrix():
    rows, cols, count = 3, 6, 4
    W = 0.02 * _rand((count * rows * cols,), 80)
    M = np.zeros(count * rows * cols, np.float32)
    G = _rand((count * rows * cols,), 81).astype(np.float32)
    (Wn,), (Mn,) = oracle.muon_step([W], [G], [M], [(rows, cols, count, 0)], 0.02, 0.95)
    for i in range(count):
        sl = slice(i * rows * cols, (i + 1) * rows * cols)
        w1, m1, _ = oracle.muon_matrix_step(W[sl].reshape(rows, cols), M[sl].reshape(rows, cols),
                                            G[sl].reshape(rows, cols), 0.02, 0.95)
        assert np.array_equal(Wn[sl], w1.reshape(-1))
        assert np.array_equal(Mn[sl], m1.reshape(-1))


# --- the "gram" Newton-Schulz method ------------------------------------------

@pytest.mark.parametrize("shape", [(3, 5), (8, 8), (17, 4), (64, 128), (1, 7), (9, 1), (40, 24)])
@pytest.mark.parametrize("steps", [0, 1, 5])
def test_gram_method_svd_closed_form(shape, steps):
    # the Gram-form iteration is the quintic iteration rewritten on X X^T: its
    # result is P p^steps(s / (||s|| + eps)) Q^T like the standard form's
    V = _rand(shape, 90 + steps)
    assert _rel(oracle.newton_schulz_gram(V, steps), _closed_form(V, steps)) < 1e-10


@pytest.mark.parametrize("restarts", [(), (2,), (1, 3), (0, 4)])
def test_gram_method_restarts_change_nothing_in_exact_arithmetic(restarts):
    V = _rand((24, 70), 91)
    assert _rel(oracle.newton_schulz_gram(V, 5, restarts=restarts), oracle.newton_schulz(V, 5)) < 1e-10


def test_gram_method_with_a_schedule_and_transpose():
    co = [(3.0, -3.2, 1.2), (2.5, -2.0, 0.6), (15 / 8, -10 / 8, 3 / 8)]
    V = _rand((50, 20), 92)                       # tall: transposed and back
    assert _rel(oracle.newton_schulz_gram(V, 4, co), oracle.newton_schulz(V, 4, co)) < 1e-10
    assert _rel(oracle.newton_schulz_gram(V.T, 4, co), oracle.newton_schulz_gram(V, 4, co).T) < 1e-13


def test_gram_method_brute_force_one_iteration():
    # one iteration written out with explicit loops on a 2 x 3 matrix:
    # A = X X^T, Q = a I + b A + c A A, U = Q X
    V = np.array([[1.0, -2.0, 0.5], [0.25, 3.0, -1.0]])
    fro = math.sqrt(sum(v * v for v in V.ravel()))
    X = V / (fro + EPS)
    A = [[sum(X[i][k] * X[j][k] for k in range(3)) for j in range(2)] for i in range(2)]
    AA = [[sum(A[i][k] * A[k][j] for k in range(2)) for j in range(2)] for i in range(2)]
    Q = [[A_ * (i == j) + B_ * A[i][j] + C_ * AA[i][j] for j in range(2)] for i in range(2)]
    U = np.array([[sum(Q[i][k] * X[k][j] for k in range(2)) for j in range(3)] for i in range(2)])
    assert _rel(oracle.newton_schulz_gram(V, 1), U) < 1e-14


def test_gram_method_differs_from_the_standard_form_only_by_rounding():
    # in float32 the two forms round different operations, so they do not agree
    # bit for bit; in float64 they agree to 1e-10 (the pins above)
    V = _rand((32, 256), 93)

    def f32_standard(V):
        X = (V / np.linalg.norm(V)).astype(np.float32)
        for _ in range(5):
            A = X @ X.T
            X = np.float32(A_) * X + (np.float32(B_) * A + np.float32(C_) * (A @ A)) @ X
        return X

    def f32_gram(V):
        X = (V / np.linalg.norm(V)).astype(np.float32)
        A, R, I = X @ X.T, np.eye(32, dtype=np.float32), np.eye(32, dtype=np.float32)
        for _ in range(5):
            Q = np.float32(A_) * I + np.float32(B_) * A + np.float32(C_) * (A @ A)
            A, R = Q @ A @ Q, Q @ R
        return R @ X

    s, g = f32_standard(V), f32_gram(V)
    assert 0 < _rel(g, s) < 1e-4
    assert _rel(g, oracle.newton_schulz(V)) < 1e-4 and _rel(s, oracle.newton_schulz(V)) < 1e-4


def test_full_step_gram_method():
    W = 0.02 * _rand((6, 9), 94)
    M = (0.02 * _rand((6, 9), 95)).astype(np.float32)
    G = _rand((6, 9), 96).astype(np.float32)
    Ws, Ms, Us = oracle.muon_matrix_step(W, M, G, 0.02, 0.95, True, 0.01)
    Wg, Mg, Ug = oracle.muon_matrix_step(W, M, G, 0.02, 0.95, True, 0.01, method="gram")
    assert np.array_equal(Ms, Mg) and _rel(Ug, Us) < 1e-10 and _rel(Wg, Ws) < 1e-12
    with pytest.raises(ValueError):
        oracle.muon_matrix_step(W, M, G, 0.02, 0.95, method="cubic")
