"""GPU parity for the paper's other head widths and for heads stored [B, T, H, d_h].

The paper's models use head widths 48, 64 and 80 ("Ask Self, Ask Others", Table 2)
and 60 (the Hybrid model, Appendix F.1).  Every case is compared element by element
with the float64 oracle, which always takes contiguous [B, H, T, d] tensors: inputs
for the [B, T, H, d] layout are transposed on the host before the GPU call and the
GPU outputs transposed back before the comparison.  Tolerances are those of
test_gpu_parity.py (derived there from the arithmetic of each path).
"""
import numpy as np
import pytest
import torch

import oracle
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

Y_TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}
L_TOL = {torch.float32: 1e-6, torch.bfloat16: 1e-3}  # relative above |L| = 1; fp32 adds T 2^-24
G_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
BHTD, BTHD = rb.RELATION_LAYOUT_BHTD, rb.RELATION_LAYOUT_BTHD


def _to_layout(t, layout):
    return t.permute(0, 2, 1, 3).contiguous() if layout == BTHD else t.contiguous()


def _from_layout(t, layout):
    return t.permute(0, 2, 1, 3) if layout == BTHD else t


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _maxerr(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def _case(name, B, H, T, d, dtype, tau=1.0, lam=0.5, causal=True, layout=BHTD):
    return (rin.Workload(name, B, H, T, d, dtype, tau, lam, causal, 1.0, backward=True), layout)


CASES = [
    _case("f32_d48", 1, 2, 150, 48, torch.float32),
    _case("f32_d60", 2, 1, 129, 60, torch.float32, lam=0.0),
    _case("f32_d80_noncausal", 1, 2, 97, 80, torch.float32, causal=False),
    _case("bf16_d48", 2, 3, 300, 48, torch.bfloat16),
    _case("bf16_d48_tau2", 1, 2, 256, 48, torch.bfloat16, tau=2.0, lam=0.0),
    _case("bf16_d60", 1, 3, 300, 60, torch.bfloat16),
    _case("bf16_d80", 2, 2, 300, 80, torch.bfloat16),
    _case("bf16_d80_noncausal", 1, 2, 200, 80, torch.bfloat16, causal=False),
    _case("bf16_d64_bthd", 2, 3, 300, 64, torch.bfloat16, layout=BTHD),
    _case("bf16_d48_bthd", 1, 4, 257, 48, torch.bfloat16, layout=BTHD),
    _case("bf16_d80_bthd", 2, 2, 200, 80, torch.bfloat16, layout=BTHD),
    _case("bf16_d128_bthd", 1, 3, 150, 128, torch.bfloat16, layout=BTHD),
    _case("bf16_d60_bthd", 1, 2, 130, 60, torch.bfloat16, layout=BTHD),
    _case("f32_d64_bthd", 2, 2, 100, 64, torch.float32, layout=BTHD),
    _case("f32_d60_bthd", 1, 3, 65, 60, torch.float32, causal=False, layout=BTHD),
]


@pytest.mark.parametrize("w,layout", CASES, ids=[c[0].name for c in CASES])
def test_widths_and_layouts_match_oracle(w, layout):
    x_cpu = rin.make(w)
    x = {k: _to_layout(v, layout).cuda() for k, v in x_cpu.items()}
    Y, L = rb.fwd(x["P1"], x["P2"], x["V"], w.tau_S, w.lam, w.causal, layout=layout)
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, w.causal, layout)
    # bf16 d_h = 60 pads its operands into the forward's workspace first (one more launch).
    assert rb.relation_last_launch_count() == (2 if rb.relation_fwd_workspace_bytes(prob) else 1)
    dP1, dP2, dV, dlam = rb.bwd(x["P1"], x["P2"], x["V"], Y, L, x["dY"], w.tau_S, w.lam, w.causal, layout=layout)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    assert tuple(L.shape) == (w.B, w.H, w.T)

    Yr, Lr = oracle.fwd(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], w.tau_S, w.lam, w.causal)
    vmax = float(np.max(np.abs(_np(x_cpu["V"]))))
    assert _maxerr(_np(_from_layout(Y, layout)), Yr) <= Y_TOL[w.dtype] * vmax
    l_bound = L_TOL[w.dtype] * np.maximum(1.0, np.abs(Lr)) + (w.T * 2.0 ** -24 if w.dtype == torch.float32 else 0.0)
    assert float(np.max(np.abs(_np(L) - Lr) / l_bound)) <= 1.0

    ref = oracle.bwd(x_cpu["P1"], x_cpu["P2"], x_cpu["V"], x_cpu["dY"], w.tau_S, w.lam, w.causal)
    for got, exp, name in zip((dP1, dP2, dV), ref[:3], ("dP1", "dP2", "dV")):
        gmax = float(np.max(np.abs(exp)))
        err = _maxerr(_np(_from_layout(got, layout)), exp)
        assert err <= G_TOL[w.dtype] * gmax, (name, err, gmax)
    assert abs(float(dlam.item()) - ref[3]) <= 5 * G_TOL[w.dtype] * max(1.0, abs(ref[3]))


@pytest.mark.parametrize("layout", [BHTD, BTHD])
@pytest.mark.parametrize("T,causal", [(1, True), (130, True), (300, True), (257, False)])
def test_forward_from_padded_copies_equals_direct_forward(T, causal, layout):
    """d_h = 60: relation_fwd_ws (tiles loaded by TMA from the zero-padded copies in its
    workspace) and relation_fwd (tiles copied from the caller's 120-byte rows by cp.async)
    place the same zero-padded tile in shared memory, so Y and L agree bit for bit."""
    w = rin.Workload("d60_ws", 2, 3, T, 60, torch.bfloat16, 2.0, 0.5, causal, 1.0)
    x = {k: _to_layout(v, layout).cuda() for k, v in rin.make(w).items()}
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, w.causal, layout)
    Y0, L0 = torch.empty_like(x["V"]), torch.empty(w.B, w.H, w.T, device="cuda")
    rb.relation_fwd(prob, x["P1"], x["P2"], x["V"], Y0, L0)
    assert rb.relation_last_launch_count() == 1
    ws = rb.fwd_workspace(prob, "cuda")
    assert ws is not None and ws.numel() * 4 >= rb.relation_fwd_workspace_bytes(prob)
    ws.fill_(float("nan"))  # contents on entry are ignored
    Y1, L1 = torch.full_like(x["V"], float("nan")), torch.full((w.B, w.H, w.T), float("nan"), device="cuda")
    rb.relation_fwd_ws(prob, x["P1"], x["P2"], x["V"], Y1, L1, ws)
    assert rb.relation_last_launch_count() == 2
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    assert torch.equal(Y0, Y1) and torch.equal(L0, L1)


@pytest.mark.parametrize("d", [48, 64, 80])
def test_forward_with_workspace_needs_none_elsewhere(d):
    """Every other width: relation_fwd_ws takes no workspace and is relation_fwd."""
    w = rin.Workload("nows", 1, 2, 200, d, torch.bfloat16, 1.0, 0.5, True, 1.0)
    x = {k: v.cuda() for k, v in rin.make(w).items()}
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, w.causal)
    assert rb.relation_fwd_workspace_bytes(prob) == 0 and rb.fwd_workspace(prob, "cuda") is None
    Y0, L0 = torch.empty_like(x["V"]), torch.empty(w.B, w.H, w.T, device="cuda")
    Y1, L1 = torch.empty_like(x["V"]), torch.empty(w.B, w.H, w.T, device="cuda")
    rb.relation_fwd(prob, x["P1"], x["P2"], x["V"], Y0, L0)
    rb.relation_fwd_ws(prob, x["P1"], x["P2"], x["V"], Y1, L1, None)
    assert rb.relation_last_launch_count() == 1
    torch.cuda.synchronize()
    assert torch.equal(Y0, Y1) and torch.equal(L0, L1)


@pytest.mark.parametrize("d,layout", [(48, BHTD), (60, BHTD), (80, BHTD), (48, BTHD), (60, BTHD), (80, BTHD)])
def test_narrow_heads_write_only_their_tensors(d, layout):
    """Outputs sit between guard bands of NaN; no kernel may write outside them (the
    narrow-width epilogues mask the zero-padding columns of their tiles)."""
    w = rin.Workload("guard", 1, 2, 200, d, torch.bfloat16, 1.0, 0.5, True, 1.0, backward=True)
    x = {k: _to_layout(v, layout).cuda() for k, v in rin.make(w).items()}
    n = x["P1"].numel()
    guard = 4096

    def banded():
        buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
        return buf, buf[guard:guard + n].view(x["P1"].shape)

    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, w.causal, layout)
    bY, Y = banded()
    L = torch.empty(w.B, w.H, w.T, device="cuda")
    rb.relation_fwd(prob, x["P1"], x["P2"], x["V"], Y, L)
    banded_out = [(bY, Y)]
    nws = rb.relation_fwd_workspace_bytes(prob)
    if nws:  # the padded-copy forward, its workspace also between NaN guard bands
        bY2, Y2 = banded()
        wbuf = torch.full((nws // 4 + 2 * guard,), float("nan"), device="cuda")
        rb.relation_fwd_ws(prob, x["P1"], x["P2"], x["V"], Y2, L, wbuf[guard:guard + nws // 4])
        torch.cuda.synchronize()
        assert torch.isnan(wbuf[:guard]).all() and torch.isnan(wbuf[guard + nws // 4:]).all()
        assert torch.equal(Y2, Y)
        banded_out.append((bY2, Y2))
    outs = [banded() for _ in range(3)]
    ws = torch.empty((rb.relation_bwd_workspace_bytes(prob) + 3) // 4, device="cuda")
    dlam = torch.empty(1, device="cuda")
    rb.relation_bwd(prob, x["P1"], x["P2"], x["V"], Y, L, x["dY"], outs[0][1], outs[1][1], outs[2][1], dlam, ws)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    for buf, inner in banded_out + outs:
        assert torch.isnan(buf[:guard].float()).all() and torch.isnan(buf[guard + n:].float()).all()
        assert torch.isfinite(inner.float()).all()
