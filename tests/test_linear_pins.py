"""Pins of the Linear Relation oracle ("Ask Self, Ask Others", Sec. 5.2 eq.(15)-(17),
Appendix A.4) against what the pages and plain mathematics fix:
  - a hand-worked scalar example (d = 1), written out token by token;
  - full retention (alpha = 1): the masked-matrix closed form of unnormalised linear
    transport, E = Diag(S) (strict-lower(Q^ K^T) Diag(S)) I~;
  - the unrolled state of A.4.4 and the expanded historical exchange of A.4.5 (brute
    force over all earlier tokens with explicit retention products);
  - strict historical support (A.4.3): E_1 = 0 and E_t does not see I~_t or later tokens;
  - the write stores I~_t, not Y_t (A.4.6);
  - splitting the sequence and carrying the state equals one pass;
  - the backward by central finite differences on every input.
"""
import numpy as np
import pytest

from oracle import linear as lo

RNG = np.random.default_rng(11)


def _inputs(B, H, T, d, gscale=0.3, seed=0):
    r = np.random.default_rng(seed)
    P1 = r.standard_normal((B, H, T, d))
    P2 = r.standard_normal((B, H, T, d))
    I = r.standard_normal((B, H, T, d))
    G = -gscale * r.random((B, H, T, d))  # log-retention <= 0
    return P1, P2, I, G


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def test_scalar_worked_example():
    """d = 1: p^ = sign(p), the state is a number.  Three tokens by hand."""
    p1 = np.array([1.0, -2.0, 0.5])
    p2 = np.array([2.0, 1.0, -1.0])
    i = np.array([3.0, -1.0, 4.0])
    g = np.log(np.array([0.5, 0.25, 0.8]))
    tau = 2.0
    S = _sig(p1 * p2 / tau)                     # sqrt(d) = 1
    # t=1: C- = 0.5*0 = 0, E = 0, C = S1 * sign(p2_1) * i1
    C1 = S[0] * 1.0 * 3.0
    # t=2: C- = 0.25*C1, E = S2 * C- * sign(p1_2) = -S2 * 0.25 * C1
    E2 = S[1] * (0.25 * C1) * (-1.0)
    C2 = 0.25 * C1 + S[1] * 1.0 * (-1.0)
    # t=3: C- = 0.8*C2, E = S3 * C- * sign(p1_3)
    E3 = S[2] * (0.8 * C2) * 1.0
    C3 = 0.8 * C2 + S[2] * (-1.0) * 4.0
    Y, CT = lo.fwd(p1.reshape(1, 1, 3, 1), p2.reshape(1, 1, 3, 1), i.reshape(1, 1, 3, 1),
                   g.reshape(1, 1, 3, 1), tau)
    assert np.allclose(Y.ravel(), [3.0, -1.0 + E2, 4.0 + E3], rtol=1e-14, atol=1e-14)
    assert np.allclose(CT.ravel(), [C3], rtol=1e-14)


def test_full_retention_is_masked_linear_transport():
    B, H, T, d, tau = 2, 2, 23, 8, 1.5
    P1, P2, I, _ = _inputs(B, H, T, d)
    Y, _ = lo.fwd(P1, P2, I, np.zeros_like(P1), tau)
    for b in range(B):
        for h in range(H):
            n1 = P1[b, h] / np.linalg.norm(P1[b, h], axis=1, keepdims=True)
            n2 = P2[b, h] / np.linalg.norm(P2[b, h], axis=1, keepdims=True)
            S = _sig(np.sum(P1[b, h] * P2[b, h], axis=1) / (tau * np.sqrt(d)))
            W = np.tril(n1 @ n2.T, k=-1) * S[:, None] * S[None, :]
            assert np.allclose(Y[b, h], I[b, h] + W @ I[b, h], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gscale", [0.05, 1.0, 6.0])
def test_recurrence_equals_expanded_historical_exchange(gscale):
    P1, P2, I, G = _inputs(1, 3, 17, 6, gscale=gscale, seed=3)
    Y, _ = lo.fwd(P1, P2, I, G, 0.7)
    Yu = lo.fwd_unrolled(P1, P2, I, G, 0.7)
    assert np.allclose(Y, Yu, rtol=1e-12, atol=1e-13)


def test_final_state_equals_unrolled_state():
    """A.4.4: C_T = sum_j (prod_{u=j+1..T} D_u) S_j p^2_j I~_j^T."""
    P1, P2, I, G = _inputs(1, 1, 9, 5, gscale=0.8, seed=4)
    _, CT = lo.fwd(P1, P2, I, G, 1.0)
    T, d = 9, 5
    C = np.zeros((d, d))
    for j in range(T):
        S = _sig(P1[0, 0, j] @ P2[0, 0, j] / np.sqrt(d))
        k = P2[0, 0, j] / np.linalg.norm(P2[0, 0, j])
        decay = np.prod(np.exp(G[0, 0, j + 1:]), axis=0)
        C += (decay * S * k)[:, None] * I[0, 0, j][None, :]
    assert np.allclose(CT[0, 0], C, rtol=1e-12, atol=1e-13)


def test_strict_historical_support():
    P1, P2, I, G = _inputs(1, 2, 12, 4, seed=5)
    Y, _ = lo.fwd(P1, P2, I, G, 1.0)
    assert np.array_equal(Y[:, :, 0], I[:, :, 0])  # E_1 = 0 exactly
    t = 7
    I2, P12, P22, G2 = I.copy(), P1.copy(), P2.copy(), G.copy()
    I2[:, :, t:] += 5.0          # the token's own information and the future
    P22[:, :, t + 1:] *= -3.0    # future coordinates
    G2[:, :, t + 1:] -= 1.0      # future retention
    Y2, _ = lo.fwd(P12, P22, I2, G2, 1.0)
    assert np.allclose((Y2 - I2)[:, :, :t + 1], (Y - I)[:, :, :t + 1], rtol=0, atol=1e-14)


def test_write_stores_information_not_answer():
    """A.4.6: the state takes S_t p^2_t I~_t^T; with one earlier token, token 3 reads
    token 1 and token 2 only through their own I~, never through Y_2."""
    P1, P2, I, G = _inputs(1, 1, 3, 4, seed=6)
    G[:] = 0.0
    Y, _ = lo.fwd(P1, P2, I, G, 1.0)
    n1 = P1[0, 0] / np.linalg.norm(P1[0, 0], axis=1, keepdims=True)
    n2 = P2[0, 0] / np.linalg.norm(P2[0, 0], axis=1, keepdims=True)
    S = _sig(np.sum(P1[0, 0] * P2[0, 0], axis=1) / 2.0)
    E3 = S[2] * (S[0] * (n2[0] @ n1[2]) * I[0, 0, 0] + S[1] * (n2[1] @ n1[2]) * I[0, 0, 1])
    assert np.allclose(Y[0, 0, 2], I[0, 0, 2] + E3, rtol=1e-13)


def test_zero_coordinates_neither_read_nor_write():
    """A token whose p1 is zero reads nothing (E_t = 0); one whose p2 is zero writes
    nothing, so the later tokens see the same history as with that token's I~ zeroed."""
    P1, P2, I, G = _inputs(1, 1, 6, 4, seed=10)
    P1[0, 0, 2] = 0.0
    P2[0, 0, 3] = 0.0
    Y, _ = lo.fwd(P1, P2, I, G, 1.0)
    assert np.array_equal(Y[0, 0, 2], I[0, 0, 2])
    I0 = I.copy()
    I0[0, 0, 3] = 0.0
    Y0, _ = lo.fwd(P1, P2, I0, G, 1.0)
    assert np.allclose((Y - I)[0, 0, 4:], (Y0 - I0)[0, 0, 4:], rtol=0, atol=1e-15)


def test_split_sequence_carries_the_state():
    P1, P2, I, G = _inputs(2, 2, 20, 6, seed=7)
    Y, CT = lo.fwd(P1, P2, I, G, 1.3)
    Ya, Ca = lo.fwd(P1[:, :, :8], P2[:, :, :8], I[:, :, :8], G[:, :, :8], 1.3)
    Yb, Cb = lo.fwd(P1[:, :, 8:], P2[:, :, 8:], I[:, :, 8:], G[:, :, 8:], 1.3, C0=Ca)
    assert np.allclose(np.concatenate([Ya, Yb], axis=2), Y, rtol=1e-13, atol=1e-13)
    assert np.allclose(Cb, CT, rtol=1e-13, atol=1e-13)


def test_backward_by_finite_differences():
    B, H, T, d, tau = 1, 2, 7, 5, 0.9
    P1, P2, I, G = _inputs(B, H, T, d, gscale=0.6, seed=8)
    W = RNG.standard_normal((B, H, T, d))
    grads = lo.bwd(P1, P2, I, G, tau, W)
    args = [P1, P2, I, G]

    def loss(a):
        return float(np.sum(lo.fwd(*a, tau)[0] * W))

    h = 1e-6
    for which in range(4):
        for idx in [(0, 0, 0, 0), (0, 1, 3, 2), (0, 0, 6, 4), (0, 1, 5, 1), (0, 0, 2, 3)]:
            ap = [a.copy() for a in args]
            am = [a.copy() for a in args]
            ap[which][idx] += h
            am[which][idx] -= h
            fd = (loss(ap) - loss(am)) / (2 * h)
            assert abs(fd - grads[which][idx]) < 1e-6 * max(1.0, abs(fd)), (which, idx)


def test_retention_gradient_of_the_last_token():
    """alpha_T acts only on the read of token T (the later state is never read), so
    dG_T = alpha_T * S_T * p^1_T * (C_{T-1} dY_T), elementwise over channels."""
    B, H, T, d, tau = 1, 1, 5, 4, 1.0
    P1, P2, I, G = _inputs(B, H, T, d, seed=9)
    W = RNG.standard_normal((B, H, T, d))
    _, _, _, dG = lo.bwd(P1, P2, I, G, tau, W)
    _, C4 = lo.fwd(P1[:, :, :4], P2[:, :, :4], I[:, :, :4], G[:, :, :4], tau)
    S = _sig(P1[0, 0, 4] @ P2[0, 0, 4] / (tau * 2.0))
    q = P1[0, 0, 4] / np.linalg.norm(P1[0, 0, 4])
    a = np.exp(G[0, 0, 4])
    expect = a * S * q * (C4[0, 0] @ W[0, 0, 4])
    assert np.allclose(dG[0, 0, 4], expect, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------- retention gate
# Sec. 5.2 eq.(16) / Appendix A.4.1: g = -exp(A_log) * softplus(r + dt_bias), per
# head and channel, alpha = exp(g) in (0, 1].


def _gate_inputs(B=2, H=3, T=5, d=4, seed=3):
    r = np.random.default_rng(seed)
    R = 2.0 * r.standard_normal((B, H, T, d))
    A_log = 0.5 * r.standard_normal((H, d))
    dt_bias = r.standard_normal((H, d))
    return R, A_log, dt_bias


def test_gate_special_values():
    """softplus(0) = log 2; A_log = 0 gives exp(A_log) = 1; large arguments tend to -x e^A,
    very negative ones to -e^A e^x; alpha stays in (0, 1]."""
    R, A_log, dt_bias = _gate_inputs()
    zero = np.zeros((1, 2, 1, 3))
    G0 = lo.gate(zero, np.zeros((2, 3)), np.zeros((2, 3)))
    assert np.allclose(G0, -np.log(2.0), rtol=0, atol=1e-15)
    Gs = lo.gate(zero, np.log(np.array([[2.0, 3.0, 5.0]] * 2)), np.zeros((2, 3)))
    assert np.allclose(Gs[0, 0, 0], -np.array([2.0, 3.0, 5.0]) * np.log(2.0), atol=1e-14)
    big = lo.gate(np.full((1, 1, 1, 1), 40.0), np.array([[0.3]]), np.array([[1.0]]))
    assert abs(big[0, 0, 0, 0] + np.exp(0.3) * 41.0) < 1e-12
    small = lo.gate(np.full((1, 1, 1, 1), -40.0), np.array([[0.3]]), np.array([[1.0]]))
    assert abs(small[0, 0, 0, 0] / (-np.exp(0.3) * np.exp(-39.0)) - 1.0) < 1e-12
    G = lo.gate(R, A_log, dt_bias)
    assert np.all(G < 0.0) and np.all(np.exp(G) <= 1.0) and np.all(np.exp(G) > 0.0)
    # per-(head, channel) parameters: head h, channel c use A_log[h, c] and dt_bias[h, c]
    h, c = 2, 1
    x = R[1, h, 3, c] + dt_bias[h, c]
    assert abs(G[1, h, 3, c] + np.exp(A_log[h, c]) * np.log1p(np.exp(x))) < 1e-12


def test_gate_backward_by_finite_differences():
    R, A_log, dt_bias = _gate_inputs()
    dG = np.random.default_rng(9).standard_normal(R.shape)
    dR, dA, dB = lo.gate_bwd(R, A_log, dt_bias, dG)
    f = lambda R_, A_, b_: float(np.sum(lo.gate(R_, A_, b_) * dG))
    h = 1e-6
    for idx in [(0, 0, 0, 0), (1, 2, 4, 3), (0, 1, 2, 1)]:
        Rp, Rm = R.copy(), R.copy()
        Rp[idx] += h
        Rm[idx] -= h
        assert abs((f(Rp, A_log, dt_bias) - f(Rm, A_log, dt_bias)) / (2 * h) - dR[idx]) < 1e-6
    for idx in [(0, 0), (2, 3), (1, 2)]:
        Ap, Am = A_log.copy(), A_log.copy()
        Ap[idx] += h
        Am[idx] -= h
        assert abs((f(R, Ap, dt_bias) - f(R, Am, dt_bias)) / (2 * h) - dA[idx]) < 1e-6
        bp, bm = dt_bias.copy(), dt_bias.copy()
        bp[idx] += h
        bm[idx] -= h
        assert abs((f(R, A_log, bp) - f(R, A_log, bm)) / (2 * h) - dB[idx]) < 1e-6


def test_gated_linear_relation_chain_by_finite_differences():
    """The gated operator: Y = Linear(P1, P2, I~, gate(R)); its gradients w.r.t. R, A_log and
    dt_bias are the oracle's dG pushed through gate_bwd."""
    B, H, T, d, tau = 1, 2, 6, 3, 1.5
    P1, P2, I, _ = _inputs(B, H, T, d, seed=5)
    R, A_log, dt_bias = _gate_inputs(B, H, T, d, seed=6)
    dY = np.random.default_rng(7).standard_normal((B, H, T, d))
    _, _, _, dG = lo.bwd(P1, P2, I, lo.gate(R, A_log, dt_bias), tau, dY)
    dR, dA, dB = lo.gate_bwd(R, A_log, dt_bias, dG)
    f = lambda R_, A_, b_: float(np.sum(lo.fwd(P1, P2, I, lo.gate(R_, A_, b_), tau)[0] * dY))
    h = 1e-6
    for idx in [(0, 0, 3, 1), (0, 1, 5, 2)]:
        Rp, Rm = R.copy(), R.copy()
        Rp[idx] += h
        Rm[idx] -= h
        assert abs((f(Rp, A_log, dt_bias) - f(Rm, A_log, dt_bias)) / (2 * h) - dR[idx]) < 1e-6
    for idx in [(0, 0), (1, 2)]:
        Ap, Am = A_log.copy(), A_log.copy()
        Ap[idx] += h
        Am[idx] -= h
        assert abs((f(R, Ap, dt_bias) - f(R, Am, dt_bias)) / (2 * h) - dA[idx]) < 1e-6
        bp, bm = dt_bias.copy(), dt_bias.copy()
        bp[idx] += h
        bm[idx] -= h
        assert abs((f(R, A_log, bp) - f(R, A_log, bm)) / (2 * h) - dB[idx]) < 1e-6


def test_gate_pins_catch_a_dropped_exponential():
    """Planted mistake: -A_log instead of -exp(A_log) fails the special values."""
    zero = np.zeros((1, 1, 1, 1))
    wrong = -np.log(2.0) * np.log(np.array([[2.0]]))[None, :, None, :] * np.ones_like(zero)
    assert abs(lo.gate(zero, np.log(np.array([[2.0]])), np.zeros((1, 1)))[0, 0, 0, 0] - wrong[0, 0, 0, 0]) > 0.5
