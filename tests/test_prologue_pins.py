"""Pins of the prologue oracle (RoPE on P1/P2, Givens head-pair mixing of the information
states; "Ask Self, Ask Others", Sec. 3.1-3.2 eq.(4), Appendix A.2.2-A.2.3, B.3) against
closed forms, invariants, the pairing sets printed in Appendix A.2.3, and finite
differences for the backward.
"""
import numpy as np
import pytest

from oracle import prologue as po

RNG = np.random.default_rng(7)


def test_rope_position_zero_is_identity():
    X = RNG.standard_normal((2, 3, 1, 8))
    assert np.allclose(po.rope(X, 1e4), X, atol=0, rtol=0)


def test_rope_two_dimensional_closed_form():
    """d = 2: the only frequency is base^0 = 1, so position t rotates (x, y) by t radians."""
    t = np.arange(5, dtype=np.float64)
    X = np.tile(np.array([0.3, -1.7]), (1, 1, 5, 1))
    R = po.rope(X, 1e4)[0, 0]
    x, y = 0.3, -1.7
    assert np.allclose(R[:, 0], x * np.cos(t) - y * np.sin(t), atol=1e-15)
    assert np.allclose(R[:, 1], x * np.sin(t) + y * np.cos(t), atol=1e-15)


def test_rope_frequency_of_the_second_coordinate():
    """d = 4, base 100: coordinate c = 1 (paired with 3) turns by t * 100^(-2/4) = t / 10."""
    t = 7.0
    X = np.zeros((1, 1, 8, 4))
    X[0, 0, 7, 1] = 1.0  # unit vector on coordinate 1 at position 7
    R = po.rope(X, 100.0)[0, 0, 7]
    assert np.allclose(R, [0.0, np.cos(t / 10), 0.0, np.sin(t / 10)], atol=1e-15)


def test_rope_preserves_pair_norms():
    X = RNG.standard_normal((2, 2, 17, 64))
    R = po.rope(X, 1e4)
    n0 = X[..., :32] ** 2 + X[..., 32:] ** 2
    n1 = R[..., :32] ** 2 + R[..., 32:] ** 2
    assert np.allclose(n0, n1, rtol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    q = RNG.standard_normal((1, 1, 1, 48))
    k = RNG.standard_normal((1, 1, 1, 48))
    s1 = np.sum(po.rope(q, 1e4, pos0=[5]) * po.rope(k, 1e4, pos0=[2]))
    s2 = np.sum(po.rope(q, 1e4, pos0=[1005]) * po.rope(k, 1e4, pos0=[1002]))
    assert abs(s1 - s2) < 1e-10


def test_rope_backward_is_the_adjoint():
    X = RNG.standard_normal((2, 2, 9, 60))
    Y = RNG.standard_normal((2, 2, 9, 60))
    lhs = np.sum(po.rope(X, 1e4, pos0=[3, 11]) * Y)
    rhs = np.sum(X * po.rope_bwd(Y, 1e4, pos0=[3, 11]))
    assert abs(lhs - rhs) < 1e-10


def test_givens_pairings_match_appendix():
    """Appendix A.2.3 prints, for H = 8 (one-based): M_A = {(1,2),(3,4),(5,6),(7,8)},
    M_B = {(2,3),(4,5),(6,7),(8,1)}."""
    A = {(a + 1, b + 1) for a, b in po.givens_pairs(8, 0)}
    B = {(a + 1, b + 1) for a, b in po.givens_pairs(8, 1)}
    assert A == {(1, 2), (3, 4), (5, 6), (7, 8)}
    assert B == {(2, 3), (4, 5), (6, 7), (8, 1)}


def test_givens_special_angles_and_norms():
    I = RNG.standard_normal((2, 4, 5, 16))
    assert np.allclose(po.givens(I, [0.0, 0.0], 0), I, atol=0)
    G = po.givens(I, [np.pi / 2, np.pi / 2], 0)
    assert np.allclose(G[:, 0], -I[:, 1], atol=1e-15) and np.allclose(G[:, 1], I[:, 0], atol=1e-15)
    G = po.givens(I, [0.3, -1.1], 1)
    # Appendix A.2.2: ||I~a||^2 + ||I~b||^2 = ||Ia||^2 + ||Ib||^2 for every pair.
    for a, b in po.givens_pairs(4, 1):
        assert np.allclose(G[:, a] ** 2 + G[:, b] ** 2, I[:, a] ** 2 + I[:, b] ** 2, rtol=1e-13)


@pytest.mark.parametrize("pairing", [0, 1])
def test_givens_backward_by_finite_differences(pairing):
    H = 6
    I = RNG.standard_normal((2, H, 4, 8))
    W = RNG.standard_normal((2, H, 4, 8))
    theta = RNG.standard_normal(H // 2)
    It = po.givens(I, theta, pairing)
    dI, dth = po.givens_bwd(W, It, theta, pairing)
    h = 1e-6
    for k in range(H // 2):
        tp, tm = theta.copy(), theta.copy()
        tp[k] += h
        tm[k] -= h
        fd = (np.sum(W * po.givens(I, tp, pairing)) - np.sum(W * po.givens(I, tm, pairing))) / (2 * h)
        assert abs(fd - dth[k]) < 1e-7 * max(1.0, abs(fd))
    for idx in [(0, 0, 1, 2), (1, H - 1, 3, 7), (0, 3, 0, 0)]:
        Ip, Im = I.copy(), I.copy()
        Ip[idx] += h
        Im[idx] -= h
        fd = (np.sum(W * po.givens(Ip, theta, pairing)) - np.sum(W * po.givens(Im, theta, pairing))) / (2 * h)
        assert abs(fd - dI[idx]) < 1e-7 * max(1.0, abs(fd))
