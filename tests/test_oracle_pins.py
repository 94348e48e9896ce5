"""Pins the float64 oracle to what the paper and mathematics fix, independent of the oracle itself.

Sources ("Ask Self, Ask Others: Relation Is All You Need"):
  Sec. 3.1 eq.(1)-(3), Appendix A.1.1  construction of U, S, E, R and F
  Appendix A.1.2-A.1.4, eq.(6)-(9)     Self/Exchange factorisation, F_ii + g_i = 1
  eq.(10), eq.(11), Appendix A.1.5    log-odds identity; lambda cancels inside Exchange
  Appendix A.1.7                      first token: F_11 = 1, Y_1 = I~_1
  Sec. 5.1 eq.(12)-(14), Appendix A.3  FlashRelation equals Full Relation
Each test is chosen so that a plausible slip in the oracle (a dropped 1/sqrt(d) or
1/tau_S, a zero-based log i, a wrong sign of lambda, P1 and P2 swapped, a wrong
derivative) fails at least one of them.
"""
import math
import os

import mpmath
import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _flow(P1, P2, tau, lam, causal=True):
    """F via V = identity (d = T): then Y_i = sum_j F_ij e_j = F_i."""
    T = P1.shape[2]
    assert P1.shape[3] == T
    V = np.broadcast_to(np.eye(T), P1.shape).copy()
    Y, L = oracle.fwd(P1, P2, V, tau, lam, causal)
    return Y, L


# ---------------------------------------------------------------- boundary (A.1.7)
@pytest.mark.parametrize("tau,lam,causal", [(1.0, 0.5, True), (0.5, -1.3, True), (2.0, 0.0, False), (0.7, 3.0, True)])
def test_single_token_returns_information(tau, lam, causal):
    P1, P2, V = _rand((2, 3, 1, 8), 1, 4.0), _rand((2, 3, 1, 8), 2, 4.0), _rand((2, 3, 1, 8), 3)
    Y, L = oracle.fwd(P1, P2, V, tau, lam, causal)
    assert np.array_equal(Y, V)  # F_11 = 1 exactly
    u = np.einsum("bhtc,bhtc->bht", P1, P2) / math.sqrt(8)
    assert np.allclose(L, 1.0 / (1.0 + np.exp(-u / tau)), rtol=0, atol=1e-15)  # L_1 = S_1


def test_first_row_is_its_own_information_in_longer_sequences():
    P1, P2, V = _rand((1, 2, 9, 4), 4, 3.0), _rand((1, 2, 9, 4), 5, 3.0), _rand((1, 2, 9, 4), 6)
    Y, _ = oracle.fwd(P1, P2, V, 1.0, 0.5, True)
    assert np.array_equal(Y[:, :, 0], V[:, :, 0])


# ------------------------------------------------- closed forms from constant evidence
def _diag_weight_closed_form(S, E, n_hist, lam, c):
    """F_ii = e^S / (e^S + n_hist * c^-lam * e^E)  (Appendix A.1.2-A.1.3 with all E_ij = E)."""
    S, E = mpmath.mpf(S), mpmath.mpf(E)
    a = mpmath.exp(S)
    b = n_hist * mpmath.power(c, -lam) * mpmath.exp(E)
    return float(a / (a + b))


def test_golden_u_zero_fixture_matches_closed_form_and_oracle():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "u_zero_diag_weights.txt")) if not ln.startswith("#")]
    T = 128
    P1 = np.zeros((1, 1, T, T))
    P2 = _rand((1, 1, T, T), 7)
    for lam in (0.0, 0.5):
        F, _ = _flow(P1, P2, 1.0, lam)
        for lam_s, i_s, f_s in rows:
            if float(lam_s) != lam:
                continue
            i = int(i_s)
            closed = _diag_weight_closed_form(0.5, 0.0, i - 1, lam, i)
            assert abs(float(f_s) - closed) < 1e-15, (lam, i)
            assert abs(F[0, 0, i - 1, i - 1] - float(f_s)) < 1e-15, (lam, i)
    # the four values quoted for lambda = 0 (e^0.5/(e^0.5 + i - 1)) at i = 2, 3, 10, 128
    F0, _ = _flow(P1, P2, 1.0, 0.0)
    for i, v in [(2, 0.622459), (3, 0.451863), (10, 0.154828), (128, 0.0128157)]:
        assert abs(F0[0, 0, i - 1, i - 1] - v) < 5e-7


@pytest.mark.parametrize("lam", [0.0, 0.5])
def test_u_zero_output_is_self_plus_uniform_history(lam):
    T, d = 40, 16
    P1 = np.zeros((1, 2, T, d))
    P2 = _rand((1, 2, T, d), 8)
    V = _rand((1, 2, T, d), 9)
    Y, _ = oracle.fwd(P1, P2, V, 1.3, lam, True)
    for i in range(1, T + 1):
        f = _diag_weight_closed_form(0.5, 0.0, i - 1, lam, i)
        hist = V[:, :, : i - 1].mean(axis=2) if i > 1 else 0.0
        expect = f * V[:, :, i - 1] + (1 - f) * hist
        assert np.allclose(Y[:, :, i - 1], expect, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_row_constant_evidence_closed_form(causal):
    """P2 rows all equal b, P1 row i = a_i: U_ij = a_i.b/sqrt(d) = c_i for every j.

    Hits sigmoid saturation and both SiLU tails (c in +-8, +-20, +-60).  Swapping
    the roles of P1 and P2 would make U depend on the column instead and fail.
    """
    d = 4
    cs = np.array([0.3, -8.0, 8.0, -20.0, 20.0, -60.0, 60.0, 1.7, -1.27846, 5.0, -0.5, 12.0])
    T = cs.size
    b = np.array([2.0, 0.0, 0.0, 0.0])
    P2 = np.broadcast_to(b, (1, 1, T, d)).copy()
    P1 = np.zeros((1, 1, T, d))
    P1[0, 0, :, 0] = cs * math.sqrt(d) / 2.0
    tau, lam = 0.5, 0.5
    V = np.broadcast_to(np.eye(T), (1, 1, T, T)).copy()
    P1p = np.zeros((1, 1, T, T)); P1p[..., :d] = P1
    P2p = np.zeros((1, 1, T, T)); P2p[..., :d] = P2
    # d is now T for the identity trick; rescale so that U keeps the values c_i
    P1p[..., 0] *= math.sqrt(T) / math.sqrt(d)
    F, _ = oracle.fwd(P1p, P2p, V, tau, lam, causal)
    F = F[0, 0]
    for k, c in enumerate(cs):
        i = k + 1
        S = mpmath.mpf(1) / (1 + mpmath.exp(-mpmath.mpf(c) / tau))
        E = mpmath.mpf(c) / (1 + mpmath.exp(-mpmath.mpf(c)))
        n_hist, count = (i - 1, i) if causal else (T - 1, T)
        f = _diag_weight_closed_form(S, E, n_hist, lam, count)
        assert abs(F[k, k] - f) < 1e-13, (c, F[k, k], f)
        hist = [j for j in (range(k) if causal else range(T)) if j != k]
        if hist:
            assert np.allclose(F[k, hist], (1 - f) / len(hist), rtol=0, atol=1e-13)
        if causal:
            assert np.all(F[k, k + 1:] == 0.0)


# ------------------------------------------------------------------ invariants
def test_rows_sum_to_one_and_are_causal():
    T = 24
    P1, P2 = _rand((2, 2, T, T), 10, 2.0), _rand((2, 2, T, T), 11, 2.0)
    F, _ = _flow(P1, P2, 0.8, 0.5)
    assert np.allclose(F.sum(-1), 1.0, rtol=0, atol=1e-13)
    assert np.all(np.triu(F, 1) == 0.0)
    assert np.all(F >= 0.0)


def test_exchange_allocation_does_not_depend_on_lambda_and_log_odds_shift():
    """eq.(11): pi^E is lambda-free.  eq.(10): log(g_i/F_ii) moves by -(l1-l2) log i."""
    T = 20
    P1, P2 = _rand((1, 3, T, T), 12, 1.5), _rand((1, 3, T, T), 13, 1.5)
    l1, l2 = 0.5, -0.25
    F1, _ = _flow(P1, P2, 1.0, l1)
    F2, _ = _flow(P1, P2, 1.0, l2)
    for i in range(2, T + 1):
        k = i - 1
        g1 = F1[..., k, :k].sum(-1)
        g2 = F2[..., k, :k].sum(-1)
        assert np.allclose(F1[..., k, k] + g1, 1.0, atol=1e-13)  # eq.(7)
        pi1 = F1[..., k, :k] / g1[..., None]
        pi2 = F2[..., k, :k] / g2[..., None]
        assert np.allclose(pi1, pi2, rtol=1e-11, atol=1e-14)  # eq.(8), (11)
        shift = np.log(g1 / F1[..., k, k]) - np.log(g2 / F2[..., k, k])
        assert np.allclose(shift, -(l1 - l2) * math.log(i), rtol=0, atol=1e-11)  # eq.(10)


def test_log_normaliser_matches_flow():
    T = 16
    P1, P2 = _rand((1, 1, T, T), 14), _rand((1, 1, T, T), 15)
    F, L = _flow(P1, P2, 1.0, 0.5)
    F_lam0, L_lam0 = _flow(P1, P2, 1.0, 0.0)
    # the diagonal entry has the same R_ii under both lambdas: F_ii = exp(S_i - L_i)
    assert np.allclose(np.log(np.diagonal(F[0, 0])) - np.log(np.diagonal(F_lam0[0, 0])),
                       -(L[0, 0] - L_lam0[0, 0]), atol=1e-12)


@pytest.mark.parametrize("tiles", [[1], [3, 7, 2], [16], [5, 1, 128]])
@pytest.mark.parametrize("tau,lam", [(1.0, 0.5), (0.5, 0.0), (2.0, -0.7)])
def test_flash_relation_equals_full_relation(tiles, tau, lam):
    """Appendix A.3.5: the tiled Exchange scan reproduces the Full Relation row exactly."""
    P1, P2, V = _rand((2, 2, 37, 8), 16, 2.0), _rand((2, 2, 37, 8), 17, 2.0), _rand((2, 2, 37, 8), 18)
    Y, L = oracle.fwd(P1, P2, V, tau, lam, True)
    Yf, Lf = oracle.flash_fwd(P1, P2, V, tau, lam, tiles)
    assert np.max(np.abs(Y - Yf)) < 1e-12
    assert np.max(np.abs(L - Lf)) < 1e-12


# ------------------------------------------------------------- brute force (mpmath)
mpmath.mp.dps = 50


def _mp_forward(P1, P2, V, tau, lam, causal):
    """Brute force at 50 digits, straight from eq.(1)-(3)."""
    T, d = len(P1), len(P1[0])
    tau, lam = mpmath.mpf(tau), mpmath.mpf(lam)
    Y = [[mpmath.mpf(0)] * d for _ in range(T)]
    L = [mpmath.mpf(0)] * T
    for i in range(T):
        vis = range(i + 1) if causal else range(T)
        count = (i + 1) if causal else T
        r = {}
        for j in vis:
            u = mpmath.fsum(mpmath.mpf(P1[i][c]) * mpmath.mpf(P2[j][c]) for c in range(d)) / mpmath.sqrt(d)
            if j == i:
                r[j] = 1 / (1 + mpmath.exp(-u / tau))
            else:
                r[j] = u / (1 + mpmath.exp(-u)) - lam * mpmath.log(count)
        Z = mpmath.fsum(mpmath.exp(x) for x in r.values())
        L[i] = mpmath.log(Z)
        for c in range(d):
            Y[i][c] = mpmath.fsum(mpmath.exp(r[j]) / Z * mpmath.mpf(V[j][c]) for j in vis)
    return Y, L


@pytest.mark.parametrize("T,d,causal,tau,lam", [(1, 3, True, 1.0, 0.5), (5, 4, True, 0.5, 0.5),
                                                (8, 2, True, 2.0, -0.3), (6, 3, False, 1.0, 0.5)])
def test_forward_matches_brute_force(T, d, causal, tau, lam):
    P1, P2, V = _rand((1, 1, T, d), 20, 2.0), _rand((1, 1, T, d), 21, 2.0), _rand((1, 1, T, d), 22)
    Y, L = oracle.fwd(P1, P2, V, tau, lam, causal)
    Ym, Lm = _mp_forward(P1[0, 0].tolist(), P2[0, 0].tolist(), V[0, 0].tolist(), tau, lam, causal)
    assert np.max(np.abs(Y[0, 0] - np.array(Ym, dtype=float))) < 1e-13
    assert np.max(np.abs(L[0, 0] - np.array(Lm, dtype=float))) < 1e-13


@pytest.mark.parametrize("causal", [True, False])
def test_backward_matches_brute_force_derivatives(causal):
    """Gradients of sum(dY * Y) at 50 digits by mpmath central differences of the brute force."""
    T, d, tau, lam = 4, 2, 0.7, 0.5
    P1, P2, V, dY = (_rand((1, 1, T, d), s, 1.5) for s in (30, 31, 32, 33))
    dP1, dP2, dV, dlam = oracle.bwd(P1, P2, V, dY, tau, lam, causal)
    base = [P1[0, 0].tolist(), P2[0, 0].tolist(), V[0, 0].tolist()]
    G = dY[0, 0].tolist()

    def loss(args, lam_v):
        Y, _ = _mp_forward(args[0], args[1], args[2], tau, lam_v, causal)
        return mpmath.fsum(Y[i][c] * G[i][c] for i in range(T) for c in range(d))

    h = mpmath.mpf("1e-20")
    for k, got in enumerate((dP1, dP2, dV)):
        for i in range(T):
            for c in range(d):
                plus = [[row[:] for row in a] for a in base]
                minus = [[row[:] for row in a] for a in base]
                plus[k][i][c] = mpmath.mpf(plus[k][i][c]) + h
                minus[k][i][c] = mpmath.mpf(minus[k][i][c]) - h
                ref = (loss(plus, lam) - loss(minus, lam)) / (2 * h)
                assert abs(got[0, 0, i, c] - float(ref)) < 1e-12, (k, i, c)
    ref = (loss(base, mpmath.mpf(lam) + h) - loss(base, mpmath.mpf(lam) - h)) / (2 * h)
    assert abs(dlam - float(ref)) < 1e-12


def test_backward_matches_finite_differences_fp64():
    T, d, tau, lam = 12, 6, 1.0, 0.5
    P1, P2, V, dY = (_rand((1, 2, T, d), s, 1.2) for s in (40, 41, 42, 43))
    dP1, dP2, dV, dlam = oracle.bwd(P1, P2, V, dY, tau, lam, True)

    def loss(a, b, v, lm):
        Y, _ = oracle.fwd(a, b, v, tau, lm, True)
        return float(np.sum(Y * dY))

    h = 1e-6
    rng = np.random.default_rng(44)
    for k, (arr, grad) in enumerate(((P1, dP1), (P2, dP2), (V, dV))):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, s)) for s in arr.shape)
            args = [P1.copy(), P2.copy(), V.copy()]
            args[k][idx] += h
            lp = loss(*args, lam)
            args[k][idx] -= 2 * h
            lm = loss(*args, lam)
            assert abs((lp - lm) / (2 * h) - grad[idx]) < 1e-7, (k, idx)
    num = (loss(P1, P2, V, lam + h) - loss(P1, P2, V, lam - h)) / (2 * h)
    assert abs(num - dlam) < 1e-7


# ---------------------------------------------- restricted entry points agree with full ones
@pytest.mark.parametrize("causal", [True, False])
def test_sampled_entry_points_agree_with_full_oracle(causal):
    B, H, T, d = 2, 2, 33, 8
    P1, P2, V, dY = (_rand((B, H, T, d), s) for s in (50, 51, 52, 53))
    tau, lam = 0.9, 0.5
    Y, L = oracle.fwd(P1, P2, V, tau, lam, causal)
    dP1, dP2, dV, _ = oracle.bwd(P1, P2, V, dY, tau, lam, causal)
    heads = np.array([0, 3, 1, 2, 3])
    rows = np.array([0, 32, 5, 17, 1])
    Ys, Ls = oracle.fwd_rows(P1, P2, V, tau, lam, causal, heads, rows)
    Yf, Lf = Y.reshape(B * H, T, d), L.reshape(B * H, T)
    assert np.allclose(Ys, Yf[heads, rows], atol=1e-14)
    assert np.allclose(Ls, Lf[heads, rows], atol=1e-14)
    head = 3
    Lh, Dh = oracle.row_stats(P1, P2, V, dY, tau, lam, causal, head)
    assert np.allclose(Lh, Lf[head], atol=1e-14)
    assert np.allclose(Dh, np.sum(Yf[head] * dY.reshape(B * H, T, d)[head], -1), atol=1e-13)
    cols = np.array([0, 5, 31, 32])
    g2, gv = oracle.bwd_cols(P1, P2, V, dY, tau, lam, causal, head, Lh, Dh, cols)
    assert np.allclose(g2, dP2.reshape(B * H, T, d)[head, cols], atol=1e-12)
    assert np.allclose(gv, dV.reshape(B * H, T, d)[head, cols], atol=1e-12)
    g1 = oracle.bwd_rows(P1, P2, V, dY, tau, lam, causal, head, cols)
    assert np.allclose(g1, dP1.reshape(B * H, T, d)[head, cols], atol=1e-12)


def test_oracle_rejects_bad_arguments():
    P = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.fwd(P, P, P, 0.0, 0.5, True)  # tau_S must be > 0
    with pytest.raises(ValueError):
        oracle.fwd(P, P, P, 1.0, float("nan"), True)
    with pytest.raises(ValueError):
        oracle.flash_fwd(P, P, P, 1.0, 0.5, [0])
