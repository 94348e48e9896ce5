"""GPU parity at the method's edge: sigmoid saturation and both SiLU tails.

The seeded Gaussian workloads keep |U| near 1 (std 1.125 even for the large-|U|
configuration at d = 64), so they never reach the regimes where the bf16
kernels' tanh-based sigmoid/SiLU and the lazily raised softmax maximum could
break.  These cases build the evidence directly:

* Row-constant evidence: row i of P1 is (c_i sqrt(d) / 2, 0, ..., 0) and row j
  of P2 is (2, 0, w_j) with w_j seeded Gaussian coordinates 2..d-1, so
  U_ij = c_i for every visible j.  (The w_j leave U unchanged but give dP1 a
  scale: without them dP1_i = (2/sqrt(d)) sum_j dU_ij e_0, and since
  sum_j dR_ij = 0 that is a cancellation residue whose size is set by the
  rounding of D_i = dY_i . Y_i, not by the method.)  Then
  ("Ask Self, Ask Others", Sec. 3.1 eq.(1)-(3); Appendix A.1.2-A.1.3) the Self
  weight is F_ii = e^S / (e^S + n c^-lambda e^E) with S = sigmoid(c/tau_S),
  E = SiLU(c), n visible history entries and count c (i causal, T otherwise),
  the history shares the rest uniformly, and
  L_i = log(e^S + n c^-lambda e^E).  With c in {+-8, +-20, +-60} the Self entry
  saturates and the Exchange entries sit in both SiLU tails.
* One Exchange entry of +60 among -60s in the last key tile of a row, so the
  running maximum jumps by 60 on the row's final tile and the rescale fires.

Every case is compared element by element with the float64 oracle and, where
the closed form applies, with the closed form.  Tolerances: Y <= 1e-2 max|V|
(bf16) / 1e-5 max|V| (fp32); L <= 1e-3 max(1, |L|) (bf16) /
1e-6 max(1, |L|) + T 2^-24 (fp32) -- relative above 1 because L reaches ~60
here and fp32 spaces numbers near 64 by 7.6e-6, plus the worst-case rounding
of a float32 sum of up to T terms (relative error below T 2^-24), which sets
log l when all of a row's terms are equal; gradients <= 2e-2 / 1e-4 of the
largest reference entry.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

Y_TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}
L_TOL = {torch.float32: 1e-6, torch.bfloat16: 1e-3}
G_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def _l_bound(dtype, T, L_ref):
    """Per-row L bound: relative above |L| = 1, plus float32 summation of T terms."""
    return L_TOL[dtype] * np.maximum(1.0, np.abs(L_ref)) + (T * 2.0 ** -24 if dtype == torch.float32 else 0.0)

EDGE_C = [8.0, -8.0, 20.0, -20.0, 60.0, -60.0, 0.3, -1.27846]


def _np(t):
    return t.detach().double().cpu().numpy()


def _row_constant(T, d, dtype, cs, H=2):
    """P1, P2 with U_ij = c_i (head h takes the list rotated by h), V, dY seeded.

    Coordinate 1 of P1 and P2 stays zero, free for a test to place one entry."""
    P1 = torch.zeros(1, H, T, d, dtype=torch.float64)
    for h in range(H):
        c = np.array([cs[(k + h) % len(cs)] for k in range(T)])
        P1[0, h, :, 0] = torch.from_numpy(c * math.sqrt(d) / 2.0)
    P2 = torch.zeros(1, H, T, d, dtype=torch.float64)
    P2[..., 0] = 2.0
    P2[..., 2:] = rin.gaussian((1, H, T, d - 2), 43).double()
    x = {
        "P1": P1.to(dtype),
        "P2": P2.to(dtype),
        "V": rin.gaussian((1, H, T, d), 44, 1.0, dtype),
        "dY": rin.gaussian((1, H, T, d), 45, 1.0, dtype),
    }
    # The evidence the kernels see: the stored (rounded) coordinates, in float64.
    c_act = x["P1"][0, :, :, 0].double().numpy() * 2.0 / math.sqrt(d)
    return x, c_act


def _closed_form(c, V, tau, lam, causal):
    """Y and L of one head whose evidence is constant along each row (c: [T])."""
    T = c.size
    i = np.arange(1, T + 1, dtype=np.float64)
    S = 1.0 / (1.0 + np.exp(-c / tau))
    E = c / (1.0 + np.exp(-c))
    n = (i - 1) if causal else np.full(T, T - 1.0)
    count = i if causal else np.full(T, float(T))
    # log of the history mass n c^-lambda e^E (absent when n = 0)
    with np.errstate(divide="ignore"):
        log_hist = np.where(n > 0, np.log(np.maximum(n, 1.0)) - lam * np.log(count) + E, -np.inf)
    L = np.logaddexp(S, log_hist)
    f_self = np.exp(S - L)
    if causal:
        csum = np.cumsum(V, axis=0)
        hist = np.zeros_like(V)
        hist[1:] = csum[:-1] / (i[1:, None] - 1)
    else:
        hist = (V.sum(axis=0)[None, :] - V) / (T - 1)
    Y = f_self[:, None] * V + (1.0 - f_self)[:, None] * hist
    return Y, L


def _run_fwd(x, tau, lam, causal):
    xd = {k: v.cuda() for k, v in x.items()}
    Y, L = rb.fwd(xd["P1"], xd["P2"], xd["V"], tau, lam, causal)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    return xd, Y, L


def _check_y_l(Yg, Lg, Yr, Lr, vmax, dtype, what):
    ey = float(np.max(np.abs(Yg - Yr)))
    el = float(np.max(np.abs(Lg - Lr) / _l_bound(dtype, Lr.shape[-1], Lr)))
    assert ey <= Y_TOL[dtype] * vmax, (what, "Y", ey, Y_TOL[dtype] * vmax)
    assert el <= 1.0, (what, "L error / bound", el)


CASES = [(dt, d, causal) for dt in (torch.bfloat16, torch.float32) for d in (64, 128) for causal in (True, False)]


@pytest.mark.parametrize("dtype,d,causal", CASES,
                         ids=[f"{'bf16' if dt == torch.bfloat16 else 'f32'}_d{d}_{'causal' if c else 'full'}"
                              for dt, d, c in CASES])
def test_row_constant_edge_forward(dtype, d, causal):
    """Saturated Self entries and both SiLU tails across three key tiles and a ragged tail."""
    T, tau, lam = 300, 0.5, 0.5
    x, c_act = _row_constant(T, d, dtype, EDGE_C)
    _, Y, L = _run_fwd(x, tau, lam, causal)
    Yg, Lg = _np(Y), _np(L)
    Yr, Lr = oracle.fwd(x["P1"], x["P2"], x["V"], tau, lam, causal)
    vmax = float(x["V"].abs().max())
    _check_y_l(Yg, Lg, Yr, Lr, vmax, dtype, "oracle")
    Vn = _np(x["V"])
    for h in range(c_act.shape[0]):
        Yc, Lc = _closed_form(c_act[h], Vn[0, h], tau, lam, causal)
        _check_y_l(Yg[0, h], Lg[0, h], Yc, Lc, vmax, dtype, f"closed form, head {h}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("cs", [[8.0, -8.0], EDGE_C], ids=["c_pm8", "c_edge"])
def test_row_constant_edge_backward(dtype, cs):
    """The backward in the saturated regime against the oracle's chain rule."""
    T, d, tau, lam = 300, 64, 0.5, 0.5
    x, _ = _row_constant(T, d, dtype, cs)
    xd, Y, L = _run_fwd(x, tau, lam, True)
    dP1, dP2, dV, dlam = rb.bwd(xd["P1"], xd["P2"], xd["V"], Y, L, xd["dY"], tau, lam, True)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    ref = oracle.bwd(x["P1"], x["P2"], x["V"], x["dY"], tau, lam, True)
    for got, exp, name in zip((dP1, dP2, dV), ref[:3], ("dP1", "dP2", "dV")):
        gmax = float(np.max(np.abs(exp)))
        err = float(np.max(np.abs(_np(got) - exp)))
        assert err <= G_TOL[dtype] * gmax, (name, err, gmax)
    derr = abs(float(dlam.item()) - ref[3])
    assert derr <= 5 * G_TOL[dtype] * max(1.0, abs(ref[3])), (float(dlam.item()), ref[3])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_late_maximum_jump_rescales(dtype):
    """Row 290 sees -60 everywhere except key 280 (+60), in its last key tile."""
    T, d, tau, lam = 300, 64, 1.0, 0.5
    x, _ = _row_constant(T, d, dtype, [-60.0], H=1)
    i0, j_star = 290, 280
    P1 = x["P1"].double()
    P2 = x["P2"].double()
    # U[i0, j*] = (P1[i0,0] * 2 + g * e) / 8 = (-480 + 960) / 8 = +60; every other
    # entry keeps -60 because no other P1 row has a second coordinate.
    P1[0, 0, i0, 1] = 32.0
    P2[0, 0, j_star, 1] = 30.0
    x["P1"], x["P2"] = P1.to(dtype), P2.to(dtype)
    _, Y, L = _run_fwd(x, tau, lam, True)
    Yg, Lg = _np(Y), _np(L)
    Yr, Lr = oracle.fwd(x["P1"], x["P2"], x["V"], tau, lam, True)
    vmax = float(x["V"].abs().max())
    _check_y_l(Yg, Lg, Yr, Lr, vmax, dtype, "oracle")
    # Closed form of row i0: Self sigmoid(-60), i0 - 1 Exchange entries, one at +60.
    i = i0 + 1
    S = 1.0 / (1.0 + math.exp(60.0 / tau))
    E_neg = -60.0 / (1.0 + math.exp(60.0))
    hist = [math.log(i - 2) - lam * math.log(i) + E_neg, -lam * math.log(i) + 60.0]
    L_row = float(np.logaddexp.reduce([S] + hist))
    assert abs(Lg[0, 0, i0] - L_row) <= _l_bound(dtype, T, L_row)
    # Nearly all of the row's weight sits on key j*.
    assert float(np.max(np.abs(Yg[0, 0, i0] - _np(x["V"])[0, 0, j_star]))) <= Y_TOL[dtype] * vmax + 1e-20
