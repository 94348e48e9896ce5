"""Float64 oracle of the operator's input prologue (TEST INFRASTRUCTURE ONLY).

"Ask Self, Ask Others: Relation Is All You Need":
  - RoPE on the relation coordinates P1, P2 (Sec. 3.1 below eq.(1); Appendix B.3:
    full head width, base 10^4; the information states stay unrotated).  The pages
    do not say how coordinates are paired; this oracle takes the half-split form:
    coordinate c in [0, d/2) is rotated with coordinate c + d/2 by the angle
    pos * base^(-2c/d), pos the zero-based token position.
  - Givens mixing of the information states of adjacent head pairs (Sec. 3.2
    eq.(4); Appendix A.2.2, A.2.3): for a pair (a, b) with angle theta,
        I~a = cos(theta) Ia - sin(theta) Ib,   I~b = sin(theta) Ia + cos(theta) Ib,
    with pairing A = {(1,2), (3,4), ..., (H-1,H)} and pairing B = {(2,3), (4,5),
    ..., (H,1)} (one-based heads), H/2 angles per layer.
Backward: both maps are rotations, so the input gradients are the transposed
rotations of the output gradients; d theta = sum (dI~b . I~a - dI~a . I~b).
Plain numpy in float64: one rotation per pair, written out.
"""
from __future__ import annotations

import numpy as np


def rope_angles(T: int, d: int, base: float, pos0=None, B: int = 1) -> np.ndarray:
    """Angles [B, T, d/2]: (pos0[b] + t) * base^(-2c/d)."""
    c = np.arange(d // 2, dtype=np.float64)
    inv_freq = base ** (-2.0 * c / d)
    p0 = np.zeros(B, dtype=np.float64) if pos0 is None else np.asarray(pos0, dtype=np.float64)
    t = p0[:, None] + np.arange(T, dtype=np.float64)[None, :]
    return t[:, :, None] * inv_freq[None, None, :]


def rope(X, base: float, pos0=None) -> np.ndarray:
    """X [B, H, T, d] -> rotated; coordinate c pairs with c + d/2."""
    X = np.asarray(X, dtype=np.float64)
    B, H, T, d = X.shape
    a = rope_angles(T, d, base, pos0, B)[:, None]  # [B, 1, T, d/2]
    cos, sin = np.cos(a), np.sin(a)
    x1, x2 = X[..., : d // 2], X[..., d // 2:]
    return np.concatenate([cos * x1 - sin * x2, sin * x1 + cos * x2], axis=-1)


def rope_bwd(dP, base: float, pos0=None) -> np.ndarray:
    """Gradient w.r.t. the unrotated input: the transposed rotation of dP."""
    dP = np.asarray(dP, dtype=np.float64)
    B, H, T, d = dP.shape
    a = rope_angles(T, d, base, pos0, B)[:, None]
    cos, sin = np.cos(a), np.sin(a)
    g1, g2 = dP[..., : d // 2], dP[..., d // 2:]
    return np.concatenate([cos * g1 + sin * g2, -sin * g1 + cos * g2], axis=-1)


def givens_pairs(H: int, pairing: int):
    """Zero-based head pairs (a, b); pair k uses angle theta[k]."""
    if H % 2:
        raise ValueError("Givens mixing needs an even number of heads")
    if pairing == 0:
        return [(2 * k, 2 * k + 1) for k in range(H // 2)]
    return [(2 * k + 1, (2 * k + 2) % H) for k in range(H // 2)]


def givens(I, theta, pairing: int) -> np.ndarray:
    I = np.asarray(I, dtype=np.float64)
    out = np.empty_like(I)
    for k, (a, b) in enumerate(givens_pairs(I.shape[1], pairing)):
        c, s = np.cos(float(theta[k])), np.sin(float(theta[k]))
        out[:, a] = c * I[:, a] - s * I[:, b]
        out[:, b] = s * I[:, a] + c * I[:, b]
    return out


def givens_bwd(dIt, It, theta, pairing: int):
    """Returns (dI, dtheta) given dI~ and the mixed states I~."""
    dIt = np.asarray(dIt, dtype=np.float64)
    It = np.asarray(It, dtype=np.float64)
    dI = np.empty_like(dIt)
    dtheta = np.zeros(len(theta), dtype=np.float64)
    for k, (a, b) in enumerate(givens_pairs(dIt.shape[1], pairing)):
        c, s = np.cos(float(theta[k])), np.sin(float(theta[k]))
        dI[:, a] = c * dIt[:, a] + s * dIt[:, b]
        dI[:, b] = -s * dIt[:, a] + c * dIt[:, b]
        dtheta[k] = float(np.sum(dIt[:, b] * It[:, a] - dIt[:, a] * It[:, b]))
    return dI, dtheta
