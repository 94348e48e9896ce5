"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (from the arithmetic):
  Y  : fp32 path <= 1e-5 * max|V|;  bf16 path <= 1e-2 * max|V| (fp32 accumulation,
       flow weights rounded to bf16 before the second product, bf16 output).
  L  : fp32 path <= 1e-6 * max(1, |L|) + T 2^-24; bf16 path <= 1e-3 * max(1, |L|).
       The bf16 kernels use tanh.approx (relative error ~2^-11) for SiLU, so an
       Exchange logit of size |U| carries up to ~|U| 2^-12 of error; averaged over a
       row it stays far below 1e-3.  Above 1 the bound is relative: fp32 spaces
       numbers near |L| by |L| 2^-23, about eight spacings at any magnitude.  The
       fp32 term T 2^-24 is the worst-case relative rounding of a float32 sum of up
       to T terms, which becomes log l's error when a row's terms are all equal.
  dP1, dP2, dV : fp32 path <= 1e-4 * max|g_ref| per tensor; bf16 path <= 2e-2 * max|g_ref|.
Inputs come from the seeded generator (relation_token_mixing_gb300.inputs); the
oracle upcasts the same rounded tensors to float64.
"""
import json
import math
import os

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


_MARGIN_LOG = os.environ.get("RELATION_PARITY_LOG")


def _record(what, err, tol):
    """Appends (test, quantity, error, tolerance) to RELATION_PARITY_LOG when set."""
    if _MARGIN_LOG:
        test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        with open(_MARGIN_LOG, "a") as f:
            f.write(json.dumps({"test": test, "what": what, "err": err, "tol": tol}) + "\n")


def _dev(x):
    return {k: v.cuda() for k, v in x.items()}


def _gpu_fwd(x, w):
    Y, L = rb.fwd(x["P1"], x["P2"], x["V"], w.tau_S, w.lam, w.causal)
    assert rb.relation_last_launch_count() == 1
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    return Y, L


def _gpu_bwd(x, w, Y, L):
    g = rb.bwd(x["P1"], x["P2"], x["V"], Y, L, x["dY"], w.tau_S, w.lam, w.causal)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    return g


def _maxerr(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def _lerr(a, b, dtype, T):
    """Largest L error as a fraction of its bound (see the module docstring)."""
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    bound = L_TOL[dtype] * np.maximum(1.0, np.abs(b)) + (T * 2.0 ** -24 if dtype == torch.float32 else 0.0)
    return float(np.max(np.abs(a - b) / bound))


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _check_fwd_full(w, x_cpu):
    x = _dev(x_cpu)
    Y, L = _gpu_fwd(x, w)
    Yr, Lr = oracle.fwd(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], w.tau_S, w.lam, w.causal)
    vmax = float(np.max(np.abs(_np(x_cpu["V"]))))
    ey, el = _maxerr(_np(Y), Yr), _lerr(_np(L), Lr, w.dtype, w.T)
    _record("Y", ey, Y_TOL[w.dtype] * vmax)
    _record("L/bound", el, 1.0)
    assert ey <= Y_TOL[w.dtype] * vmax, (ey, vmax)
    assert el <= 1.0, el
    return Y, L


def _check_bwd_full(w, x_cpu, Y, L):
    x = _dev(x_cpu)
    dP1, dP2, dV, dlam = _gpu_bwd(x, w, Y, L)
    ref = oracle.bwd(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], x_cpu["dY"], w.tau_S, w.lam, w.causal)
    # A tensor whose reference is identically zero (dP1, dP2 at T = 1) is held to
    # the scale of the other gradients instead.
    floor = max(float(np.max(np.abs(e))) for e in ref[:3])
    for got, exp, name in zip((dP1, dP2, dV), ref[:3], ("dP1", "dP2", "dV")):
        gmax = float(np.max(np.abs(exp)))
        if gmax == 0.0:
            gmax = floor
        err = _maxerr(_np(got), exp)
        _record(name, err, G_TOL[w.dtype] * gmax)
        assert err <= G_TOL[w.dtype] * gmax, (name, err, gmax)
    scale = max(1.0, abs(ref[3]))
    derr = abs(float(dlam.item()) - ref[3])
    _record("dlambda", derr, 5 * G_TOL[w.dtype] * scale)
    assert derr <= 5 * G_TOL[w.dtype] * scale, (float(dlam.item()), ref[3])


# --------------------------------------------------------------- small cases
def _small(name, B, H, T, d, dtype, tau, lam, causal, p_scale=1.0):
    return rin.Workload(name, B, H, T, d, dtype, tau, lam, causal, p_scale, backward=True)


SMALL = [
    _small("f32_t128", 1, 1, 128, 64, torch.float32, 1.0, 0.5, True),
    _small("f32_t128_lam0", 1, 1, 128, 64, torch.float32, 1.0, 0.0, True),
    _small("f32_ragged_d128", 2, 2, 150, 128, torch.float32, 0.7, 0.5, True),
    _small("f32_noncausal", 1, 2, 97, 64, torch.float32, 1.0, 0.5, False),
    _small("bf16_ragged_d64", 2, 3, 300, 64, torch.bfloat16, 1.0, 0.5, True),
    _small("bf16_ragged_d128", 1, 3, 300, 128, torch.bfloat16, 1.0, 0.5, True),
    _small("bf16_large_u", 1, 4, 384, 64, torch.bfloat16, 0.5, 0.5, True, 3.0 / 64 ** 0.25),
    _small("bf16_lam0_tau2", 2, 2, 256, 64, torch.bfloat16, 2.0, 0.0, True),
    _small("bf16_neg_lam", 1, 2, 200, 64, torch.bfloat16, 1.0, -0.75, True),
    _small("bf16_noncausal_d64", 1, 2, 300, 64, torch.bfloat16, 1.0, 0.5, False),
    _small("bf16_noncausal_d128", 1, 2, 200, 128, torch.bfloat16, 1.0, 0.5, False),
    _small("bf16_t1", 2, 2, 1, 64, torch.bfloat16, 1.0, 0.5, True),
    _small("bf16_t2", 1, 1, 2, 64, torch.bfloat16, 1.0, 0.5, True),
    _small("bf16_t129", 1, 2, 129, 64, torch.bfloat16, 1.0, 0.5, True),
    _small("bf16_t640_d128", 1, 1, 640, 128, torch.bfloat16, 1.0, 0.5, True),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_forward_and_backward_match_oracle(w):
    x_cpu = rin.make(w)
    Y, L = _check_fwd_full(w, x_cpu)
    _check_bwd_full(w, x_cpu, Y, L)


def test_single_token_is_exact():
    w = _small("t1", 2, 3, 1, 64, torch.bfloat16, 1.0, 0.5, True)
    x = _dev(rin.make(w))
    Y, _ = _gpu_fwd(x, w)
    assert torch.equal(Y, x["V"])


@pytest.mark.parametrize("lam", [0.0, 0.5])
def test_zero_evidence_closed_form(lam):
    """P1 = 0: Self weight e^0.5 / (e^0.5 + (i-1) i^-lam), history uniform (Appendix A.1.2-A.1.3)."""
    B, H, T, d = 1, 2, 300, 64
    P1 = torch.zeros(B, H, T, d, dtype=torch.bfloat16)
    P2 = rin.gaussian((B, H, T, d), 43, 1.0, torch.bfloat16)
    V = rin.gaussian((B, H, T, d), 44, 1.0, torch.bfloat16)
    Y, _ = rb.fwd(P1.cuda(), P2.cuda(), V.cuda(), 1.0, lam, True)
    torch.cuda.synchronize()
    Vn = _np(V)
    i = np.arange(1, T + 1, dtype=np.float64)
    f = math.exp(0.5) / (math.exp(0.5) + (i - 1) * i ** (-lam))
    csum = np.cumsum(Vn, axis=2)
    hist = np.zeros_like(Vn)
    hist[:, :, 1:] = csum[:, :, :-1] / (i[1:, None] - 1)
    expect = f[None, None, :, None] * Vn + (1 - f)[None, None, :, None] * hist
    _record("Y(closed form)", _maxerr(_np(Y), expect), 1e-2 * np.max(np.abs(Vn)))
    assert _maxerr(_np(Y), expect) <= 1e-2 * np.max(np.abs(Vn))


def test_forward_is_deterministic_and_writes_in_bounds():
    w = _small("det", 2, 2, 333, 64, torch.bfloat16, 1.0, 0.5, True)
    x = _dev(rin.make(w))
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, True)
    n = x["V"].numel()
    guard = 4096
    buf = torch.full((n + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    Lbuf = torch.full((2 * 2 * 333 + 2 * guard,), 7.0, dtype=torch.float32, device="cuda")
    Y = buf[guard:guard + n].view_as(x["V"])
    L = Lbuf[guard:guard + 2 * 2 * 333].view(2, 2, 333)
    rb.relation_fwd(prob, x["P1"], x["P2"], x["V"], Y, L)
    first = Y.clone()
    rb.relation_fwd(prob, x["P1"], x["P2"], x["V"], Y, L)
    torch.cuda.synchronize()
    assert torch.equal(first, Y)
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + n:] == 7.0)
    assert torch.all(Lbuf[:guard] == 7.0) and torch.all(Lbuf[guard + 2 * 2 * 333:] == 7.0)


def test_backward_writes_in_bounds():
    w = _small("guard_bwd", 1, 2, 200, 64, torch.bfloat16, 1.0, 0.5, True)
    x = _dev(rin.make(w))
    Y, L = _gpu_fwd(x, w)
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, True)
    n = x["V"].numel()
    guard = 4096
    bufs = [torch.full((n + 2 * guard,), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    outs = [b[guard:guard + n].view_as(x["V"]) for b in bufs]
    ws_bytes = rb.relation_bwd_workspace_bytes(prob)
    wsbuf = torch.full((ws_bytes // 4 + 2 * guard,), 5.0, dtype=torch.float32, device="cuda")
    ws = wsbuf[guard:guard + ws_bytes // 4]
    dlam = torch.zeros(1, device="cuda")
    rb.relation_bwd(prob, x["P1"], x["P2"], x["V"], Y, L, x["dY"], *outs, dlam, ws)
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[:guard] == 3.0) and torch.all(b[guard + n:] == 3.0)
    assert torch.all(wsbuf[:guard] == 5.0) and torch.all(wsbuf[guard + ws_bytes // 4:] == 5.0)
    assert rb.relation_check_device_status() == 0


def test_backward_stages_equal_single_call():
    w = _small("stages", 1, 2, 260, 64, torch.bfloat16, 1.0, 0.5, True)
    x = _dev(rin.make(w))
    Y, L = _gpu_fwd(x, w)
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, True)
    ws = torch.empty(rb.relation_bwd_workspace_bytes(prob) // 4, device="cuda")
    a = [torch.empty_like(x["V"]) for _ in range(3)]
    b = [torch.empty_like(x["V"]) for _ in range(3)]
    la, lb = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    rb.relation_bwd(prob, x["P1"], x["P2"], x["V"], Y, L, x["dY"], *a, la, ws)
    assert rb.relation_last_launch_count() == 3
    for stage in (rb.relation_bwd_prepare, rb.relation_bwd_main, rb.relation_bwd_finish):
        stage(prob, x["P1"], x["P2"], x["V"], Y, L, x["dY"], *b, lb, ws)
    torch.cuda.synchronize()
    for u, v in zip(a[1:], b[1:]):  # dP2 and dV are written without atomics
        assert torch.equal(u, v)
    assert torch.allclose(a[0].float(), b[0].float(), atol=1e-2, rtol=1e-2)


# ------------------------------------------------ the five synthetic workloads
def test_workload_single_head_fp32():
    w = rin.WORKLOADS["single_head_fp32"]
    for lam in (0.0, 0.5):
        wl = rin.Workload(w.name, w.B, w.H, w.T, w.d, w.dtype, w.tau_S, lam, backward=True)
        x_cpu = rin.make(wl)
        Y, L = _check_fwd_full(wl, x_cpu)
        _check_bwd_full(wl, x_cpu, Y, L)


def test_workload_mhr_fwd_T1024_full():
    w = rin.WORKLOADS["mhr_fwd_T1024"]
    _check_fwd_full(w, rin.make(w))


def _sample_rows(T, BH, rng, n):
    fixed = [0, 1, 126, 127, 128, 129, T // 2, T - 129, T - 128, T - 2, T - 1]
    rows = np.array([r for r in fixed if 0 <= r < T] + list(rng.integers(0, T, n)), dtype=np.int64)
    heads = rng.integers(0, BH, rows.size).astype(np.int64)
    heads[: min(3, heads.size)] = [0, BH - 1, BH // 2][: min(3, heads.size)]
    return heads, rows


def _check_fwd_sampled(w, x_cpu, Y, L, n=200, seed=0):
    rng = np.random.default_rng(seed)
    BH = w.B * w.H
    heads, rows = _sample_rows(w.T, BH, rng, n)
    Yr, Lr = oracle.fwd_rows(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], w.tau_S, w.lam, w.causal, heads, rows)
    Yg = _np(Y).reshape(BH, w.T, w.d)[heads, rows]
    Lg = _np(L).reshape(BH, w.T)[heads, rows]
    vmax = float(np.max(np.abs(_np(x_cpu["V"]))))
    _record("Y(sampled)", _maxerr(Yg, Yr), Y_TOL[w.dtype] * vmax)
    _record("L/bound(sampled)", _lerr(Lg, Lr, w.dtype, w.T), 1.0)
    assert _maxerr(Yg, Yr) <= Y_TOL[w.dtype] * vmax
    assert _lerr(Lg, Lr, w.dtype, w.T) <= 1.0


def _check_bwd_sampled(w, x_cpu, grads, heads=(0,), ncols=24, seed=1):
    dP1, dP2, dV, _ = grads
    rng = np.random.default_rng(seed)
    BH = w.B * w.H
    T = w.T
    for h in heads:
        L, D = oracle.row_stats(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], x_cpu["dY"], w.tau_S, w.lam, w.causal, h)
        cols = np.unique(np.concatenate([[0, 1, 127, 128, T // 2, T - 1], rng.integers(0, T, ncols)])).astype(np.int64)
        g2, gv = oracle.bwd_cols(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], x_cpu["dY"], w.tau_S, w.lam, w.causal, h, L,
                                 D, cols)
        g1 = oracle.bwd_rows(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], x_cpu["dY"], w.tau_S, w.lam, w.causal, h, cols)
        for got, exp, name in ((dP1, g1, "dP1"), (dP2, g2, "dP2"), (dV, gv, "dV")):
            gg = _np(got).reshape(BH, T, w.d)[h, cols]
            # per-tensor scale: the largest reference magnitude among the sampled rows
            gmax = float(np.max(np.abs(exp)))
            _record(name + "(sampled)", _maxerr(gg, exp), G_TOL[w.dtype] * gmax)
            assert _maxerr(gg, exp) <= G_TOL[w.dtype] * gmax, (name, h, _maxerr(gg, exp), gmax)


def test_workload_mhr_fwd_T4096_large_u_sampled():
    w = rin.WORKLOADS["mhr_fwd_T4096_large_u"]
    x_cpu = rin.make(w)
    Y, L = _gpu_fwd(_dev(x_cpu), w)
    _check_fwd_sampled(w, x_cpu, Y, L)


def test_workload_mhr_fwd_bwd_T2048_sampled():
    w = rin.WORKLOADS["mhr_fwd_bwd_T2048"]
    x_cpu = rin.make(w)
    x = _dev(x_cpu)
    Y, L = _gpu_fwd(x, w)
    _check_fwd_sampled(w, x_cpu, Y, L)
    grads = _gpu_bwd(x, w, Y, L)
    _check_bwd_sampled(w, x_cpu, grads, heads=(0, w.B * w.H - 1))


def test_workload_mhr_fwd_bwd_T16384_d128_sampled():
    w = rin.WORKLOADS["mhr_fwd_bwd_T16384_d128"]
    x_cpu = rin.make(w)
    x = _dev(x_cpu)
    Y, L = _gpu_fwd(x, w)
    _check_fwd_sampled(w, x_cpu, Y, L, n=64)
    grads = _gpu_bwd(x, w, Y, L)
    _check_bwd_sampled(w, x_cpu, grads, heads=(w.B * w.H - 1,), ncols=8)


def test_headline_shape_fwd_bwd_sampled():
    w = rin.WORKLOADS["mhr_fwd_bwd_T4096"]
    x_cpu = rin.make(w)
    x = _dev(x_cpu)
    Y, L = _gpu_fwd(x, w)
    _check_fwd_sampled(w, x_cpu, Y, L, n=64)
    grads = _gpu_bwd(x, w, Y, L)
    _check_bwd_sampled(w, x_cpu, grads, heads=(5,), ncols=12)
