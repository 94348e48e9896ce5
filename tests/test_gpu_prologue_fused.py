"""GPU parity of the operator with its input prologue fused into the tensor-core
kernels' operand loads ("Ask Self, Ask Others", Sec. 3.1 below eq.(1) and Appendix
B.3: RoPE on P1, P2; Sec. 3.2 eq.(4) and Appendix A.2.2-A.2.3: Givens head-pair
mixing of the information states), against the float64 oracles composed in the same
order: oracle.prologue (RoPE, Givens) then the Full Relation oracle.

Tolerances are the operator's bf16 ones: Y <= 1e-2 * max|I~| (the bf16 output bound),
L <= 1e-3 * max(1, |L|).  The fused kernel rounds the rotated and mixed values to bf16
once, as the standalone prologue does before the operator reads them, so it is also
compared with that two-call chain on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import prologue as po
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

BHTD, BTHD = rb.RELATION_LAYOUT_BHTD, rb.RELATION_LAYOUT_BTHD


def _to(t, layout):
    return t.permute(0, 2, 1, 3).contiguous() if layout == BTHD else t.contiguous()


def _back(t, layout):
    return t.permute(0, 2, 1, 3) if layout == BTHD else t


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _err(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def _l_err(a, b):
    return float(np.max(np.abs(a - b) / (1e-3 * np.maximum(1.0, np.abs(b)))))


CASES = [
    # name, B, H, T, pairing, layout, pos0, causal, tau
    ("A_bhtd", 2, 4, 300, 0, BHTD, None, True, 2.0),
    ("B_bhtd_pos0", 2, 4, 300, 1, BHTD, [3, 1000], True, 1.0),
    ("A_bthd_pos0", 1, 6, 259, 0, BTHD, [77], True, 0.5),
    ("B_bthd", 2, 2, 128, 1, BTHD, None, True, 2.0),
    ("B_noncausal", 1, 4, 200, 1, BHTD, [5], False, 1.0),
]


@pytest.mark.parametrize("name,B,H,T,pairing,layout,pos0,causal,tau", CASES, ids=[c[0] for c in CASES])
def test_fused_forward_matches_composed_oracles(name, B, H, T, pairing, layout, pos0, causal, tau):
    lam, base, d = 0.5, 1e4, 64
    w = rin.Workload("fused", B, H, T, d, torch.bfloat16, tau, lam, causal, 1.0)
    x = rin.make(w)  # P1, P2, V stand for X1, X2, I
    g = torch.Generator().manual_seed(11)
    theta = (torch.rand(H // 2, generator=g, dtype=torch.float64) * 6.0 - 3.0).float()
    dev = {k: _to(v, layout).cuda() for k, v in x.items()}
    prob = rb.problem_for(dev["P1"], tau, lam, causal, layout)
    th = theta.cuda()
    p0 = torch.tensor(pos0, dtype=torch.int32).cuda() if pos0 is not None else None
    Y = torch.empty_like(dev["V"])
    L = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    rb.relation_fwd_prologue(prob, dev["P1"], dev["P2"], dev["V"], th, pairing, base, p0, Y, L)
    assert rb.relation_last_launch_count() == 1
    # The standalone chain on the GPU: prologue pass, then the operator.
    P1, P2, It = (torch.empty_like(dev["P1"]) for _ in range(3))
    rb.relation_prologue_fwd(prob, dev["P1"], dev["P2"], dev["V"], th, pairing, base, p0, P1, P2, It)
    Yc, Lc = rb.fwd(P1, P2, It, tau, lam, causal, layout=layout)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0

    xs = {k: _np(v) for k, v in x.items()}
    # The prologue's outputs are bf16 tensors (the operator's bf16 inputs), so the composed
    # oracle rounds them to bf16 before the operator, as both GPU paths do.
    rP1, rP2 = _bf16(po.rope(xs["P1"], base, pos0)), _bf16(po.rope(xs["P2"], base, pos0))
    rIt = _bf16(po.givens(xs["V"], theta.double().numpy(), pairing))
    rY, rL = oracle.fwd(rP1, rP2, rIt, tau, lam, causal)
    vmax = float(np.max(np.abs(rIt)))
    assert _err(_np(_back(Y, layout)), rY) <= 1e-2 * vmax
    assert _l_err(_np(L), rL) <= 1.0
    # Same rounding points as the two-call chain: the two agree far inside the tolerance.
    assert _err(_np(Y), _np(Yc)) <= 2e-3 * vmax
    assert float(np.max(np.abs(_np(L) - _np(Lc)))) <= 2e-3


def test_fused_forward_without_rotation_equals_operator_on_mixed_states():
    """rope_base <= 0 disables RoPE: the fused forward then matches relation_fwd on X1, X2 and
    the mixed states, which isolates the Givens part of the fused loads."""
    B, H, T, tau, lam = 1, 4, 256, 1.0, 0.5
    w = rin.Workload("mix", B, H, T, 64, torch.bfloat16, tau, lam, True, 1.0)
    dev = {k: v.cuda() for k, v in rin.make(w).items()}
    prob = rb.problem_for(dev["P1"], tau, lam, True)
    th = torch.tensor([0.3, -2.0], device="cuda")
    Y = torch.empty_like(dev["V"])
    L = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    rb.relation_fwd_prologue(prob, dev["P1"], dev["P2"], dev["V"], th, 1, 0.0, None, Y, L)
    P1, P2, It = (torch.empty_like(dev["P1"]) for _ in range(3))
    rb.relation_prologue_fwd(prob, dev["P1"], dev["P2"], dev["V"], th, 1, 0.0, None, P1, P2, It)
    Yc, Lc = rb.fwd(dev["P1"], dev["P2"], It, tau, lam, True)
    torch.cuda.synchronize()
    assert torch.equal(P1, dev["P1"])
    # Both round each mixed value once to bf16 (the two kernels may contract the products
    # into a fused multiply-add differently, so single last-bit differences can occur).
    vmax = float(It.float().abs().max())
    assert float((Y.float() - Yc.float()).abs().max()) <= 2e-3 * vmax
    assert float((L - Lc).abs().max()) <= 1e-3


def test_fused_forward_rejects_unsupported_problems():
    dev = {k: v.cuda() for k, v in rin.make(rin.Workload("u", 1, 2, 64, 48, torch.bfloat16, 1.0, 0.5)).items()}
    prob = rb.problem_for(dev["P1"], 1.0, 0.5, True)
    th = torch.zeros(1, device="cuda")
    Y = torch.empty_like(dev["V"])
    with pytest.raises(rb.RelationError) as e:
        rb.relation_fwd_prologue(prob, dev["P1"], dev["P2"], dev["V"], th, 0, 1e4, None, Y)
    assert e.value.code == 2  # d_h 48: unsupported by the fused kernel


BWD_CASES = [
    # name, B, H, T, pairing, layout, pos0, causal, tau
    ("A_bhtd", 2, 4, 300, 0, BHTD, None, True, 2.0),
    ("B_bthd_pos0", 1, 6, 259, 1, BTHD, [1000], True, 1.0),
    ("B_bhtd_noncausal", 1, 4, 200, 1, BHTD, [5], False, 1.0),
]


@pytest.mark.parametrize("name,B,H,T,pairing,layout,pos0,causal,tau", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_fused_backward_matches_composed_oracles(name, B, H, T, pairing, layout, pos0, causal, tau):
    """relation_fwd_prologue + relation_bwd_prologue against the composed float64 oracles
    (prologue outputs rounded to bf16, operator backward, prologue backward): dX1, dX2, dI at
    the operator's bf16 gradient tolerance 2e-2 * max|g|, d theta and d lambda likewise."""
    lam, base, d = 0.5, 1e4, 64
    w = rin.Workload("fusedb", B, H, T, d, torch.bfloat16, tau, lam, causal, 1.0, backward=True)
    x = rin.make(w)
    g = torch.Generator().manual_seed(12)
    theta = (torch.rand(H // 2, generator=g, dtype=torch.float64) * 6.0 - 3.0).float()
    dev = {k: _to(v, layout).cuda() for k, v in x.items()}
    th = theta.cuda()
    p0 = torch.tensor(pos0, dtype=torch.int32).cuda() if pos0 is not None else None
    Y, L, dX1, dX2, dI, dth, dlam = rb.fused_prologue_step(dev["P1"], dev["P2"], dev["V"], th, pairing, base, tau, lam,
                                                           dev["dY"], causal, p0, layout)
    assert rb.relation_last_launch_count() == 4
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0

    xs = {k: _np(v) for k, v in x.items()}
    rP1, rP2 = _bf16(po.rope(xs["P1"], base, pos0)), _bf16(po.rope(xs["P2"], base, pos0))
    rIt = _bf16(po.givens(xs["V"], theta.double().numpy(), pairing))
    gP1, gP2, gV, rdlam = oracle.bwd(rP1, rP2, rIt, xs["dY"], tau, lam, causal)
    rdX1, rdX2 = po.rope_bwd(gP1, base, pos0), po.rope_bwd(gP2, base, pos0)
    rdI, rdth = po.givens_bwd(gV, rIt, theta.double().numpy(), pairing)
    for got, ref in ((dX1, rdX1), (dX2, rdX2), (dI, rdI)):
        assert _err(_np(_back(got, layout)), ref) <= 2e-2 * float(np.max(np.abs(ref)))
    assert _err(dth.cpu().numpy(), rdth) <= 2e-2 * max(1.0, float(np.max(np.abs(rdth))))
    assert abs(float(dlam.item()) - float(rdlam)) <= 2e-2 * max(1.0, abs(float(rdlam)))


def test_fused_backward_matches_the_two_call_chain():
    """Against the standalone chain on the GPU (prologue, operator forward and backward,
    prologue backward) at the headline head width and a ragged length."""
    B, H, T, tau, lam, base, pairing = 1, 4, 333, 0.5, 0.5, 1e4, 0
    w = rin.Workload("chainb", B, H, T, 64, torch.bfloat16, tau, lam, True, 1.0, backward=True)
    dev = {k: v.cuda() for k, v in rin.make(w).items()}
    prob = rb.problem_for(dev["P1"], tau, lam, True)
    th = torch.tensor([0.7, -0.4], device="cuda")
    Y, L, dX1, dX2, dI, dth, dlam = rb.fused_prologue_step(dev["P1"], dev["P2"], dev["V"], th, pairing, base, tau, lam,
                                                           dev["dY"])
    P1, P2, It = (torch.empty_like(dev["P1"]) for _ in range(3))
    rb.relation_prologue_fwd(prob, dev["P1"], dev["P2"], dev["V"], th, pairing, base, None, P1, P2, It)
    Yc, Lc = rb.fwd(P1, P2, It, tau, lam, True)
    gP1, gP2, gV, dlc = rb.bwd(P1, P2, It, Yc, Lc, dev["dY"], tau, lam, True)
    cX1, cX2, cI = (torch.empty_like(gP1) for _ in range(3))
    cth = torch.empty(H // 2, device="cuda")
    rb.relation_prologue_bwd(prob, gP1, gP2, gV, It, th, pairing, base, None, cX1, cX2, cI, cth)
    torch.cuda.synchronize()
    for a, b in ((dX1, cX1), (dX2, cX2), (dI, cI)):
        assert float((a.float() - b.float()).abs().max()) <= 1e-2 * float(b.float().abs().max())
    assert float((dth - cth).abs().max()) <= 1e-2 * max(1.0, float(cth.abs().max()))
