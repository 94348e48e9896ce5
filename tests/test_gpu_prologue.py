"""GPU parity of the input prologue (RoPE on P1/P2, Givens head-pair mixing of the
information states; "Ask Self, Ask Others", Sec. 3.1-3.2 eq.(4), Appendix A.2, B.3) and
of its backward, against the float64 prologue oracle; and of the whole chain prologue ->
operator -> operator backward -> prologue backward against the composed oracles.

Tolerances: fp32 outputs <= 2e-6 * max|x| (rotations by fp32 angles accurate to ~1e-6
rad, including at large positions); bf16 <= 1e-2 * max|x| (one bf16 rounding of the
output).  d theta sums many products: fp32 <= 1e-4, bf16 <= 1e-2, relative.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import prologue as po
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 2e-6, torch.bfloat16: 1e-2}
DTH_TOL = {torch.float32: 1e-4, torch.bfloat16: 1e-2}
BHTD, BTHD = rb.RELATION_LAYOUT_BHTD, rb.RELATION_LAYOUT_BTHD


def _to(t, layout):
    return t.permute(0, 2, 1, 3).contiguous() if layout == BTHD else t.contiguous()


def _back(t, layout):
    return t.permute(0, 2, 1, 3) if layout == BTHD else t


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _err(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


CASES = [
    ("f32_d64", 2, 4, 100, 64, torch.float32, 0, BHTD, None),
    ("f32_d60_bthd_B", 1, 6, 77, 60, torch.float32, 1, BTHD, [12345]),
    ("f32_d128_far", 2, 2, 50, 128, torch.float32, 1, BHTD, [1_000_000, 7]),
    ("bf16_d48", 2, 8, 130, 48, torch.bfloat16, 1, BHTD, None),
    ("bf16_d80_bthd", 1, 4, 64, 80, torch.bfloat16, 0, BTHD, [4090]),
    ("bf16_d64_bthd_B", 2, 2, 200, 64, torch.bfloat16, 1, BTHD, [3, 0]),
]


@pytest.mark.parametrize("name,B,H,T,d,dtype,pairing,layout,pos0", CASES, ids=[c[0] for c in CASES])
def test_prologue_forward_and_backward(name, B, H, T, d, dtype, pairing, layout, pos0):
    base = 1e4
    w = rin.Workload("pro", B, H, T, d, dtype, 1.0, 0.5, True, 1.0, backward=True)
    x = rin.make(w)  # P1, P2, V, dY as X1, X2, I and an upstream gradient
    g = torch.Generator().manual_seed(5)
    theta = (torch.rand(H // 2, generator=g, dtype=torch.float64) * 6.0 - 3.0).float()
    dev = {k: _to(v, layout).cuda() for k, v in x.items()}
    prob = rb.problem_for(dev["P1"], 1.0, 0.5, True, layout)
    th = theta.cuda()
    p0 = torch.tensor(pos0, dtype=torch.int32).cuda() if pos0 is not None else None
    P1, P2, It = (torch.empty_like(dev["P1"]) for _ in range(3))
    rb.relation_prologue_fwd(prob, dev["P1"], dev["P2"], dev["V"], th, pairing, base, p0, P1, P2, It)
    assert rb.relation_last_launch_count() == 2
    torch.cuda.synchronize()
    xs = {k: _np(v) for k, v in x.items()}
    ref_P1 = po.rope(xs["P1"], base, pos0)
    ref_P2 = po.rope(xs["P2"], base, pos0)
    ref_It = po.givens(xs["V"], theta.double().numpy(), pairing)
    scale = max(float(np.max(np.abs(xs[k]))) for k in ("P1", "P2", "V"))
    for got, ref in ((P1, ref_P1), (P2, ref_P2), (It, ref_It)):
        assert _err(_np(_back(got, layout)), ref) <= TOL[dtype] * scale

    # Backward with dY standing in for the three upstream gradients.
    G = dev["dY"]
    dX1, dX2, dI = (torch.empty_like(G) for _ in range(3))
    dth = torch.empty(H // 2, device="cuda")
    rb.relation_prologue_bwd(prob, G, G, G, It, th, pairing, base, p0, dX1, dX2, dI, dth)
    torch.cuda.synchronize()
    gs = xs["dY"]
    ref_dX = po.rope_bwd(gs, base, pos0)
    ref_dI, ref_dth = po.givens_bwd(gs, _np(_back(It, layout)), theta.double().numpy(), pairing)
    gscale = float(np.max(np.abs(gs)))
    assert _err(_np(_back(dX1, layout)), ref_dX) <= TOL[dtype] * gscale
    assert _err(_np(_back(dX2, layout)), ref_dX) <= TOL[dtype] * gscale
    assert _err(_np(_back(dI, layout)), ref_dI) <= TOL[dtype] * gscale
    assert _err(dth.cpu().numpy(), ref_dth) <= DTH_TOL[dtype] * max(1.0, float(np.max(np.abs(ref_dth))))


def test_rope_disabled_is_a_copy():
    w = rin.Workload("copy", 1, 2, 33, 64, torch.bfloat16, 1.0, 0.5, True, 1.0)
    x = {k: v.cuda() for k, v in rin.make(w).items()}
    prob = rb.problem_for(x["P1"], 1.0, 0.5, True)
    th = torch.zeros(1, device="cuda")
    P1, P2, It = (torch.empty_like(x["P1"]) for _ in range(3))
    rb.relation_prologue_fwd(prob, x["P1"], x["P2"], x["V"], th, 0, 0.0, None, P1, P2, It)
    torch.cuda.synchronize()
    assert torch.equal(P1, x["P1"]) and torch.equal(P2, x["P2"]) and torch.equal(It, x["V"])


def test_prologue_operator_chain_matches_composed_oracles():
    """RoPE + Givens -> Full Relation forward -> backward -> prologue backward equals the
    oracles composed in float64 (the gradients of X1, X2, I and theta)."""
    B, H, T, d, tau, lam, base, pairing = 1, 4, 160, 64, 2.0, 0.5, 1e4, 1
    w = rin.Workload("chain", B, H, T, d, torch.bfloat16, tau, lam, True, 1.0, backward=True)
    x = rin.make(w)
    theta = torch.tensor([0.4, -1.2], dtype=torch.float32)
    dev = {k: v.cuda() for k, v in x.items()}
    prob = rb.problem_for(dev["P1"], tau, lam, True)
    th = theta.cuda()
    P1, P2, It = (torch.empty_like(dev["P1"]) for _ in range(3))
    rb.relation_prologue_fwd(prob, dev["P1"], dev["P2"], dev["V"], th, pairing, base, None, P1, P2, It)
    Y, L = rb.fwd(P1, P2, It, tau, lam, True)
    dP1, dP2, dV, _ = rb.bwd(P1, P2, It, Y, L, dev["dY"], tau, lam, True)
    dX1, dX2, dI = (torch.empty_like(dP1) for _ in range(3))
    dth = torch.empty(H // 2, device="cuda")
    rb.relation_prologue_bwd(prob, dP1, dP2, dV, It, th, pairing, base, None, dX1, dX2, dI, dth)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0

    xs = {k: _np(v) for k, v in x.items()}
    rP1, rP2 = po.rope(xs["P1"], base), po.rope(xs["P2"], base)
    rIt = po.givens(xs["V"], theta.double().numpy(), pairing)
    rY, _ = oracle.fwd(rP1, rP2, rIt, tau, lam, True)
    gP1, gP2, gV, _ = oracle.bwd(rP1, rP2, rIt, xs["dY"], tau, lam, True)
    rdX1, rdX2 = po.rope_bwd(gP1, base), po.rope_bwd(gP2, base)
    rdI, rdth = po.givens_bwd(gV, rIt, theta.double().numpy(), pairing)
    assert _err(_np(Y), rY) <= 1e-2 * float(np.max(np.abs(rIt)))
    for got, ref in ((dX1, rdX1), (dX2, rdX2), (dI, rdI)):
        assert _err(_np(got), ref) <= 2e-2 * float(np.max(np.abs(ref)))
    assert _err(dth.cpu().numpy(), rdth) <= 2e-2 * max(1.0, float(np.max(np.abs(rdth))))


def test_prologue_benchmark_workload_in_full():
    """bench.py --prologue at full size (the headline workload's tensors, B4 H16 T4096 d64, pairing B,
    theta = linspace(-1, 1, H/2), base 1e4): every output against the oracle."""
    w = rin.WORKLOADS["mhr_fwd_bwd_T4096"]
    x = rin.make(w, with_dy=True)
    dev = {k: v.cuda() for k, v in x.items()}
    prob = rb.problem_for(dev["P1"], w.tau_S, w.lam, True)
    theta = torch.linspace(-1.0, 1.0, w.H // 2)
    th = theta.cuda()
    outs = [torch.empty_like(dev["P1"]) for _ in range(3)]
    rb.relation_prologue_fwd(prob, dev["P1"], dev["P2"], dev["V"], th, 1, 1e4, None, *outs)
    grads = [torch.empty_like(dev["P1"]) for _ in range(3)]
    dth = torch.empty(w.H // 2, device="cuda")
    rb.relation_prologue_bwd(prob, dev["dY"], dev["dY"], dev["dY"], outs[2], th, 1, 1e4, None, *grads, dth)
    torch.cuda.synchronize()
    xs = {k: _np(v) for k, v in x.items()}
    scale = max(float(np.max(np.abs(xs[k]))) for k in ("P1", "P2", "V"))
    assert _err(_np(outs[0]), po.rope(xs["P1"], 1e4)) <= TOL[torch.bfloat16] * scale
    assert _err(_np(outs[1]), po.rope(xs["P2"], 1e4)) <= TOL[torch.bfloat16] * scale
    Im = po.givens(xs["V"], theta.double().numpy(), 1)
    assert _err(_np(outs[2]), Im) <= TOL[torch.bfloat16] * scale
    gs = xs["dY"]
    gscale = float(np.max(np.abs(gs)))
    assert _err(_np(grads[0]), po.rope_bwd(gs, 1e4)) <= TOL[torch.bfloat16] * gscale
    dI, dthr = po.givens_bwd(gs, _np(outs[2]), theta.double().numpy(), 1)
    assert _err(_np(grads[2]), dI) <= TOL[torch.bfloat16] * gscale
    assert _err(dth.cpu().numpy(), dthr) <= DTH_TOL[torch.bfloat16] * max(1.0, float(np.max(np.abs(dthr))))
