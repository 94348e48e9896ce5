"""Float64 oracle of Linear Relation (TEST INFRASTRUCTURE ONLY).

"Ask Self, Ask Others: Relation Is All You Need", Sec. 5.2 eq.(15)-(17) and
Appendix A.4, per head with P1, P2 (after RoPE), information states I~ and the
channel-wise log-retention g (alpha = exp(g) in (0, 1], Sec. 5.2 eq.(16); the
projection that produces g from the token is outside the operator):
    S_t  = sigmoid(p1_t . p2_t / (tau_S sqrt(d)))                          (15)
    p^1_t = p1_t / ||p1_t||,  p^2_t = p2_t / ||p2_t||   (a zero vector maps to zero)
    C-_t = Diag(alpha_t) C_{t-1},   C_0 = 0 (or a given initial state)
    E_t  = S_t (C-_t)^T p^1_t,  Y_t = I~_t + E_t,  C_t = C-_t + S_t p^2_t I~_t^T   (17)
The backward is the chain rule of this recurrence, run backwards in time with
the states kept from the forward.  Plain numpy, one token at a time.

gate()/gate_bwd() are the optional KDA-style retention of eq.(16) that produces
g from a per-token projection r_t: g = -exp(A_log) * softplus(r + dt_bias) per
head and channel, and its chain rule.
"""
from __future__ import annotations

import numpy as np


def _prep(p1, p2, tau):
    d = p1.shape[-1]
    n1, n2 = np.linalg.norm(p1), np.linalg.norm(p2)
    z = float(p1 @ p2) / (tau * np.sqrt(d))
    S = 1.0 / (1.0 + np.exp(-z))
    # A zero coordinate vector normalises to zero (the pages leave 0/0 open).
    q = p1 / n1 if n1 > 0 else np.zeros_like(p1)
    k = p2 / n2 if n2 > 0 else np.zeros_like(p2)
    return S, q, k, n1, n2


def fwd(P1, P2, I, G, tau: float, C0=None):
    """P1, P2, I, G: [B, H, T, d].  Returns Y [B, H, T, d] and the final states [B, H, d, d]."""
    P1, P2, I, G = (np.asarray(a, dtype=np.float64) for a in (P1, P2, I, G))
    B, H, T, d = P1.shape
    Y = np.empty_like(I)
    CT = np.empty((B, H, d, d))
    for b in range(B):
        for h in range(H):
            C = np.zeros((d, d)) if C0 is None else np.array(C0[b, h], dtype=np.float64)
            for t in range(T):
                S, q, k, _, _ = _prep(P1[b, h, t], P2[b, h, t], tau)
                a = np.exp(G[b, h, t])
                Cm = a[:, None] * C                       # Diag(alpha) C_{t-1}
                E = S * (Cm.T @ q)                        # read before the write
                Y[b, h, t] = I[b, h, t] + E
                C = Cm + S * np.outer(k, I[b, h, t])      # become Others
            CT[b, h] = C
    return Y, CT


def fwd_unrolled(P1, P2, I, G, tau: float):
    """Appendix A.4.5: E_t = S_t sum_{j<t} S_j (p^2_j . (prod_{u=j+1..t} alpha_u) p^1_t) I~_j."""
    P1, P2, I, G = (np.asarray(a, dtype=np.float64) for a in (P1, P2, I, G))
    B, H, T, d = P1.shape
    Y = np.array(I)
    for b in range(B):
        for h in range(H):
            pre = [_prep(P1[b, h, t], P2[b, h, t], tau) for t in range(T)]
            for t in range(T):
                St, q = pre[t][0], pre[t][1]
                E = np.zeros(d)
                for j in range(t):
                    decay = np.exp(np.sum(G[b, h, j + 1:t + 1], axis=0))  # prod of alpha_{j+1..t}
                    E += pre[j][0] * float(pre[j][2] @ (decay * q)) * I[b, h, j]
                Y[b, h, t] += St * E
    return Y


def bwd(P1, P2, I, G, tau: float, dY):
    """Gradients (dP1, dP2, dI, dG) of sum(Y * dY) from C_0 = 0."""
    P1, P2, I, G, dY = (np.asarray(a, dtype=np.float64) for a in (P1, P2, I, G, dY))
    B, H, T, d = P1.shape
    dP1, dP2, dI, dG = (np.zeros_like(P1) for _ in range(4))
    sq = np.sqrt(d)
    for b in range(B):
        for h in range(H):
            pre = [_prep(P1[b, h, t], P2[b, h, t], tau) for t in range(T)]
            Cs = [np.zeros((d, d))]  # C_0 .. C_T
            for t in range(T):
                S, q, k = pre[t][:3]
                a = np.exp(G[b, h, t])
                Cs.append(a[:, None] * Cs[-1] + S * np.outer(k, I[b, h, t]))
            dC = np.zeros((d, d))  # gradient w.r.t. C_t
            for t in range(T - 1, -1, -1):
                S, q, k, n1, n2 = pre[t]
                a = np.exp(G[b, h, t])
                Cprev = Cs[t]
                Cm = a[:, None] * Cprev
                g = dY[b, h, t]
                # write: C_t = C-_t + S k I^T
                dIt = g + S * (dC.T @ k)
                dk = S * (dC @ I[b, h, t])
                dS = float(k @ dC @ I[b, h, t])
                # read: E = S C-^T q
                dCm = dC + S * np.outer(q, g)
                dq = S * (Cm @ g)
                dS += float(q @ Cm @ g)
                # decay: C-_t = Diag(a) C_{t-1}
                da = np.sum(dCm * Cprev, axis=1)
                dC = a[:, None] * dCm
                dG[b, h, t] = da * a
                dI[b, h, t] = dIt
                # S = sigmoid(p1.p2 / (tau sqrt d)); p^ = p / ||p||
                dz = dS * S * (1.0 - S) / (tau * sq)
                p1, p2 = P1[b, h, t], P2[b, h, t]
                dP1[b, h, t] = dz * p2 + ((dq - q * float(q @ dq)) / n1 if n1 > 0 else 0.0)
                dP2[b, h, t] = dz * p1 + ((dk - k * float(k @ dk)) / n2 if n2 > 0 else 0.0)
    return dP1, dP2, dI, dG


def gate(R, A_log, dt_bias):
    """KDA-style retention of Sec. 5.2 eq.(16) (Appendix A.4.1), per head h and channel c:
    g = -exp(A_log[h, c]) * softplus(r + dt_bias[h, c]), alpha = exp(g) in (0, 1].
    R: [B, H, T, d] (the projection output r_t); A_log, dt_bias: [H, d].  Returns G [B, H, T, d]."""
    R = np.asarray(R, dtype=np.float64)
    A_log = np.asarray(A_log, dtype=np.float64)[None, :, None, :]
    dt_bias = np.asarray(dt_bias, dtype=np.float64)[None, :, None, :]
    return -np.exp(A_log) * np.logaddexp(0.0, R + dt_bias)


def gate_bwd(R, A_log, dt_bias, dG):
    """Chain rule of gate(): from dG = d loss / d g, returns dR [B, H, T, d] and dA_log, d_dt_bias
    [H, d] (summed over batches and tokens).  d softplus(x)/dx = sigmoid(x); d g / d A_log = g."""
    R, dG = np.asarray(R, dtype=np.float64), np.asarray(dG, dtype=np.float64)
    A = np.asarray(A_log, dtype=np.float64)[None, :, None, :]
    x = R + np.asarray(dt_bias, dtype=np.float64)[None, :, None, :]
    g = -np.exp(A) * np.logaddexp(0.0, x)
    sig = 1.0 / (1.0 + np.exp(-x))
    dR = dG * (-np.exp(A)) * sig
    return dR, np.sum(dG * g, axis=(0, 2)), np.sum(dR, axis=(0, 2))
