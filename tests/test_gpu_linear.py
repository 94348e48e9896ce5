"""GPU parity of Linear Relation ("Ask Self, Ask Others", Sec. 5.2 eq.(15)-(17),
Appendix A.4) against the float64 recurrent oracle, through the C ABI.

Tolerance (bf16 operands, fp32 state and accumulation): the state enters every chunk
as a bf16 tensor-core operand and the chunk operands (q . F, k . B, the intra-chunk
matrix) are rounded to bf16 (relative 2^-9 each), and Y is rounded to bf16 once, so
    max |Y - Y_ref| <= 1e-2 * max |Y_ref|;
the final fp32 state sums bf16-rounded products: max |C - C_ref| <= 1e-2 * max |C_ref|.
"""
import numpy as np
import pytest
import torch

from oracle import linear as lo
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

BHTD, BTHD = rb.RELATION_LAYOUT_BHTD, rb.RELATION_LAYOUT_BTHD
TOL = 1e-2


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _to(t, layout):
    return t.permute(0, 2, 1, 3).contiguous() if layout == BTHD else t.contiguous()


def _back(t, layout):
    return t.permute(0, 2, 1, 3) if layout == BTHD else t


def _run_fwd(x, tau, layout, want_state=True):
    dev = {k: _to(v, layout).cuda() for k, v in x.items()}
    Y, C = rb.linear_fwd(dev["P1"], dev["P2"], dev["I"], dev["G"], tau, layout=layout, want_state=want_state)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    return _np(_back(Y, layout)), (None if C is None else _np(C))


def _err(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))))


# name, B, H, T, d, layout, g_scale, tau
CASES = [
    ("d64_ragged", 2, 3, 100, 64, BHTD, 1.0, 2.0),
    ("d64_segments", 1, 2, 700, 64, BHTD, 1.0, 1.0),
    ("d60_bthd_segments", 1, 4, 333, 60, BTHD, 1.0, 2.0),
    ("d48", 2, 2, 150, 48, BHTD, 1.0, 0.5),
    ("d64_strong_decay", 1, 2, 200, 64, BHTD, 8.0, 2.0),
    ("d64_full_retention", 1, 2, 300, 64, BHTD, 0.0, 2.0),
    ("d64_T1", 2, 2, 1, 64, BHTD, 1.0, 2.0),
    ("d60_T17", 1, 3, 17, 60, BTHD, 1.0, 2.0),
]


@pytest.mark.parametrize("name,B,H,T,d,layout,gs,tau", CASES, ids=[c[0] for c in CASES])
def test_linear_forward_matches_oracle(name, B, H, T, d, layout, gs, tau):
    x = rin.make_linear(rin.LinearWorkload(name, B, H, T, d, tau, gs))
    Y, C = _run_fwd(x, tau, layout)
    xs = {k: _np(v) for k, v in x.items()}
    Yr, Cr = lo.fwd(xs["P1"], xs["P2"], xs["I"], xs["G"], tau)
    assert _err(Y, Yr) <= TOL * float(np.max(np.abs(Yr))), name
    assert _err(C, Cr) <= TOL * max(float(np.max(np.abs(Cr))), 1e-6), name


def test_linear_forward_first_token_is_its_information():
    """Strict historical support (Appendix A.4.3): Y_1 = I~_1 exactly."""
    x = rin.make_linear(rin.LinearWorkload("first", 2, 4, 40, 64))
    Y, _ = _run_fwd(x, 2.0, BHTD, want_state=False)
    assert np.array_equal(Y[:, :, 0], _np(x["I"])[:, :, 0])


def test_linear_forward_many_heads_sampled():
    """B*H large enough for one segment per head (the single-pass path); sampled heads."""
    B, H, T, d, tau = 48, 8, 96, 64, 2.0
    x = rin.make_linear(rin.LinearWorkload("many", B, H, T, d, tau))
    Y, C = _run_fwd(x, tau, BHTD)
    for b, h in [(0, 0), (17, 5), (47, 7)]:
        xs = {k: _np(v[b:b + 1, h:h + 1]) for k, v in x.items()}
        Yr, Cr = lo.fwd(xs["P1"], xs["P2"], xs["I"], xs["G"], tau)
        assert _err(Y[b:b + 1, h:h + 1], Yr) <= TOL * float(np.max(np.abs(Yr)))
        assert _err(C[b:b + 1, h:h + 1], Cr) <= TOL * float(np.max(np.abs(Cr)))


def test_linear_forward_zero_coordinates():
    x = rin.make_linear(rin.LinearWorkload("zero", 1, 2, 48, 64))
    x["P1"][0, 0, 5] = 0
    x["P2"][0, 1, 20:24] = 0
    Y, C = _run_fwd(x, 2.0, BHTD)
    xs = {k: _np(v) for k, v in x.items()}
    Yr, Cr = lo.fwd(xs["P1"], xs["P2"], xs["I"], xs["G"], 2.0)
    assert np.array_equal(Y[0, 0, 5], xs["I"][0, 0, 5])
    assert _err(Y, Yr) <= TOL * float(np.max(np.abs(Yr)))


def test_linear_rejects_unsupported():
    x = torch.zeros(1, 1, 8, 80, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(1, 1, 8, 80, dtype=torch.float32, device="cuda")
    with pytest.raises(rb.RelationError) as e:
        rb.linear_fwd(x, x, x, g, 1.0)
    assert e.value.code == 2
    xf = torch.zeros(1, 1, 8, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(rb.RelationError) as e:
        rb.linear_fwd(xf, xf, xf, xf, 1.0)
    assert e.value.code == 2


# Backward tolerance: every gradient is a sum of products of bf16-rounded operands
# (chunk operands, the bf16 inputs, the state as a bf16 tensor-core operand) with fp32
# accumulation, rounded to bf16 once (dG: float32), and dP1 / dP2 pass through one
# more bf16 rounding (the normalisation part stored, then the Self part added):
#     max |g - g_ref| <= 2e-2 * max |g_ref|   for g in dP1, dP2, dI, dG.
GTOL = 2e-2

BWD_CASES = [
    ("d64_ragged", 2, 3, 100, 64, BHTD, 1.0, 2.0),
    ("d64_segments", 1, 2, 700, 64, BHTD, 1.0, 1.0),
    ("d60_bthd_segments", 1, 4, 333, 60, BTHD, 1.0, 2.0),
    ("d48", 2, 2, 150, 48, BHTD, 1.0, 0.5),
    ("d64_strong_decay", 1, 2, 200, 64, BHTD, 8.0, 2.0),
    ("d64_full_retention", 1, 2, 300, 64, BHTD, 0.0, 2.0),
    ("d64_T1", 2, 2, 1, 64, BHTD, 1.0, 2.0),
    ("d60_T17", 1, 3, 17, 60, BTHD, 1.0, 2.0),
    ("d64_T32_even_chunks", 1, 1, 32, 64, BHTD, 1.0, 2.0),
]


@pytest.mark.parametrize("name,B,H,T,d,layout,gs,tau", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_linear_backward_matches_oracle(name, B, H, T, d, layout, gs, tau):
    x = rin.make_linear(rin.LinearWorkload(name, B, H, T, d, tau, gs, backward=True))
    dev = {k: _to(v, layout).cuda() for k, v in x.items()}
    grads = rb.linear_bwd(dev["P1"], dev["P2"], dev["I"], dev["G"], dev["dY"], tau, layout=layout)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    xs = {k: _np(v) for k, v in x.items()}
    refs = lo.bwd(xs["P1"], xs["P2"], xs["I"], xs["G"], tau, xs["dY"])
    for got, ref, label in zip(grads, refs, ("dP1", "dP2", "dI", "dG")):
        err = _err(_np(_back(got, layout)), ref)
        assert err <= GTOL * max(float(np.max(np.abs(ref))), 1e-6), (name, label, err, float(np.max(np.abs(ref))))


def test_linear_backward_many_heads_sampled():
    B, H, T, d, tau = 48, 8, 80, 64, 2.0
    x = rin.make_linear(rin.LinearWorkload("many", B, H, T, d, tau, backward=True))
    dev = {k: v.cuda() for k, v in x.items()}
    grads = [_np(g) for g in rb.linear_bwd(dev["P1"], dev["P2"], dev["I"], dev["G"], dev["dY"], tau)]
    for b, h in [(0, 0), (31, 2), (47, 7)]:
        xs = {k: _np(v[b:b + 1, h:h + 1]) for k, v in x.items()}
        refs = lo.bwd(xs["P1"], xs["P2"], xs["I"], xs["G"], tau, xs["dY"])
        for got, ref in zip(grads, refs):
            assert _err(got[b:b + 1, h:h + 1], ref) <= GTOL * float(np.max(np.abs(ref)))


@pytest.mark.parametrize("T", [700, 64])
def test_linear_backward_reusing_forward_states(T):
    """relation_linear_bwd with states_from_forward = 1 after relation_linear_fwd on the same
    workspace (segment-split path at T = 700, single segment at T = 64) equals the oracle."""
    B, H, d, tau = 1, 2, 64, 1.0
    x = rin.make_linear(rin.LinearWorkload("reuse", B, H, T, d, tau, backward=True))
    dev = {k: v.cuda() for k, v in x.items()}
    prob = rb.problem_for(dev["P1"], tau, 0.0, True)
    ws = rb.linear_workspace(prob, "cuda")
    rb.linear_fwd(dev["P1"], dev["P2"], dev["I"], dev["G"], tau, workspace=ws)
    grads = rb.linear_bwd(dev["P1"], dev["P2"], dev["I"], dev["G"], dev["dY"], tau, workspace=ws,
                          states_from_forward=True)
    torch.cuda.synchronize()
    xs = {k: _np(v) for k, v in x.items()}
    refs = lo.bwd(xs["P1"], xs["P2"], xs["I"], xs["G"], tau, xs["dY"])
    for got, ref in zip(grads, refs):
        assert _err(_np(got), ref) <= GTOL * float(np.max(np.abs(ref)))


@pytest.mark.parametrize("wname,heads", [("linear_d60_T2048", [(0, 0), (9, 5), (15, 7)]),
                                         ("linear_d60_T32768", [(0, 2), (0, 7)])])
def test_linear_benchmark_workloads_sampled_heads(wname, heads):
    """The benchmark's workloads at full size, in its launch configuration (forward, then the
    backward reusing the forward's segment states from the shared workspace); whole heads
    sampled against the oracle, forward and backward."""
    w = rin.LINEAR_WORKLOADS[wname]
    x = rin.make_linear(w)
    dev = {k: v.cuda() for k, v in x.items()}
    prob = rb.problem_for(dev["P1"], w.tau_S, 0.0, True)
    ws = rb.linear_workspace(prob, "cuda")
    Y, _ = rb.linear_fwd(dev["P1"], dev["P2"], dev["I"], dev["G"], w.tau_S, workspace=ws)
    grads = rb.linear_bwd(dev["P1"], dev["P2"], dev["I"], dev["G"], dev["dY"], w.tau_S, workspace=ws,
                          states_from_forward=True)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    for b, h in heads:
        xs = {k: _np(v[b:b + 1, h:h + 1]) for k, v in x.items()}
        Yr, _ = lo.fwd(xs["P1"], xs["P2"], xs["I"], xs["G"], w.tau_S)
        assert _err(_np(Y[b:b + 1, h:h + 1]), Yr) <= TOL * float(np.max(np.abs(Yr)))
        refs = lo.bwd(xs["P1"], xs["P2"], xs["I"], xs["G"], w.tau_S, xs["dY"])
        for got, ref in zip(grads, refs):
            assert _err(_np(got[b:b + 1, h:h + 1]), ref) <= GTOL * float(np.max(np.abs(ref)))


# The KDA-style retention gate fused into the kernels (Sec. 5.2 eq.(16); Appendix A.4.1):
# R, A_log, dt_bias in, g = -exp(A_log) softplus(R + dt_bias) computed as each chunk is read;
# the backward returns dR, dA_log, d dt_bias.  Reference: oracle.linear.gate / gate_bwd composed
# with the recurrent oracle.  Tolerances as above for Y and the per-token gradients; the
# parameter gradients get the bound that the per-token one propagates to through their sums.
GATE_CASES = [
    ("d64_ragged", 2, 3, 100, 64, BHTD, 1.0, 2.0),
    ("d60_bthd_segments", 1, 4, 333, 60, BTHD, 1.0, 2.0),
    ("d48_strong_decay", 2, 2, 150, 48, BHTD, 8.0, 0.5),
]


@pytest.mark.parametrize("name,B,H,T,d,layout,gs,tau", GATE_CASES, ids=[c[0] for c in GATE_CASES])
def test_linear_gate_matches_oracle(name, B, H, T, d, layout, gs, tau):
    x = rin.make_linear(rin.LinearWorkload(name, B, H, T, d, tau, gs, backward=True))
    R, A_log, dtb = rin.linear_gate_inputs(B, H, T, d, g_scale=gs)
    dev = {k: _to(v, layout).cuda() for k, v in x.items()}
    Rd = _to(R, layout).cuda()
    Y, dP1, dP2, dI, dR, dA, dB = rb.linear_gate_fwd_bwd(dev["P1"], dev["P2"], dev["I"], Rd, A_log.cuda(),
                                                          dtb.cuda(), dev["dY"], tau, layout=layout)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    xs = {k: _np(v) for k, v in x.items()}
    Gr = lo.gate(R.double().numpy(), A_log.double().numpy(), dtb.double().numpy())
    Yr, _ = lo.fwd(xs["P1"], xs["P2"], xs["I"], Gr, tau)
    assert _err(_np(_back(Y, layout)), Yr) <= TOL * float(np.max(np.abs(Yr))), name
    g1, g2, gI, gG = lo.bwd(xs["P1"], xs["P2"], xs["I"], Gr, tau, xs["dY"])
    gR, gA, gB = lo.gate_bwd(R.double().numpy(), A_log.double().numpy(), dtb.double().numpy(), gG)
    for got, ref, label in ((dP1, g1, "dP1"), (dP2, g2, "dP2"), (dI, gI, "dI")):
        err = _err(_np(_back(got, layout)), ref)
        assert err <= GTOL * max(float(np.max(np.abs(ref))), 1e-6), (name, label, err)
    # The gate's gradients are dG times d g / d (input), so the per-token bound on dG
    # (GTOL * max|dG|) propagates elementwise to dR (d g / d R = -exp(A_log) sigmoid(R + dt_bias),
    # up to 16 g_scale here) and, through the sums over all B*T tokens, to dA_log (d g / d A_log
    # = g) and d dt_bias (the same slope as R): GTOL * max|dG| * sum_t |d g / d parameter| per channel.
    x_in = R.double().numpy() + dtb.double().numpy()[None, :, None, :]
    slope_b = np.exp(A_log.double().numpy())[None, :, None, :] / (1.0 + np.exp(-x_in))
    gmax = float(np.max(np.abs(gG)))
    dR_err = np.abs(_np(_back(dR, layout)) - gR)
    assert np.all(dR_err <= GTOL * gmax * slope_b + 1e-6), (name, "dR", float(np.max(dR_err / (GTOL * gmax * slope_b))))
    for got, ref, w, label in ((dA, gA, np.abs(Gr), "dA_log"), (dB, gB, slope_b, "d_dt_bias")):
        bound = GTOL * gmax * w.sum(axis=(0, 2))
        assert np.all(np.abs(_np(got) - ref) <= bound), (name, label, float(np.max(np.abs(_np(got) - ref) / bound)))


def test_linear_gate_equals_ungated_with_its_retention():
    """The gated forward on (R, A_log, dt_bias) and the plain forward on G = gate(...) computed
    in float32 on the host agree to within the bf16 operand rounding."""
    B, H, T, d, tau = 1, 2, 200, 64, 2.0
    x = rin.make_linear(rin.LinearWorkload("eq", B, H, T, d, tau))
    R, A_log, dtb = rin.linear_gate_inputs(B, H, T, d)
    dev = {k: v.cuda() for k, v in x.items()}
    G32 = torch.from_numpy(lo.gate(R.double().numpy(), A_log.double().numpy(), dtb.double().numpy())).float().cuda()
    Y0, _ = rb.linear_fwd(dev["P1"], dev["P2"], dev["I"], G32, tau)
    prob = rb.problem_for(dev["P1"], tau, 0.0, True)
    ws = rb.linear_workspace(prob, "cuda")
    Y1 = torch.empty_like(dev["I"])
    rb.relation_linear_fwd_gate(prob, dev["P1"], dev["P2"], dev["I"], R.cuda(), A_log.cuda(), dtb.cuda(), Y1, None, ws)
    torch.cuda.synchronize()
    assert float((Y0.float() - Y1.float()).abs().max()) <= 1e-2 * float(Y0.float().abs().max())
