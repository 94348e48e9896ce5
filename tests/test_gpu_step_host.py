"""GPU parity of relation_step_host (a training step from and to host memory, in batch slices
whose copies overlap the kernels): against the device-memory path (relation_fwd + relation_bwd
on the whole batch) and, on one small case, against the float64 oracle.

Heads are independent and every slice runs the same kernels on the same rows, so Y and L (and,
on the tensor-core path, dP2 and dV) are bit-identical to the device path's; fp32 dP2 and dV
within 1e-6 of their maximum.  dP1 sums the key tiles' partials in an order the GPU
picks, and dlambda adds the slices' sums in slice order: both within a few fp32 roundings
(dP1 <= 2^-7 * max|dP1| after its bf16 rounding, dlambda <= 1e-4 relative).  Oracle bounds
as in test_gpu_parity (bf16: Y 1e-2 max|V|, L 1e-3 max(1, |L|), gradients 2e-2 max|g|).
"""
import numpy as np
import pytest
import torch

import oracle
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

BHTD, BTHD = rb.RELATION_LAYOUT_BHTD, rb.RELATION_LAYOUT_BTHD


def _to(t, layout):
    return t.permute(0, 2, 1, 3).contiguous() if layout == BTHD else t.contiguous()


def _pinned(t):
    return t.contiguous().pin_memory()


CASES = [
    ("bf16_d64_B4_c4", 4, 2, 300, 64, torch.bfloat16, BHTD, 4),
    ("bf16_d64_B4_c2_bthd", 4, 3, 200, 64, torch.bfloat16, BTHD, 2),
    ("bf16_d64_B3_c1", 3, 2, 130, 64, torch.bfloat16, BHTD, 1),
    ("bf16_d60_B2_c2", 2, 4, 160, 60, torch.bfloat16, BHTD, 2),  # forward through its padded workspace
    ("bf16_d128_B2_c2", 2, 2, 260, 128, torch.bfloat16, BHTD, 2),
    ("f32_d64_B2_c2", 2, 2, 90, 64, torch.float32, BHTD, 2),
]


@pytest.mark.parametrize("name,B,H,T,d,dtype,layout,chunks", CASES, ids=[c[0] for c in CASES])
def test_step_host_matches_device_path(name, B, H, T, d, dtype, layout, chunks):
    w = rin.Workload(name, B, H, T, d, dtype, 1.0, 0.5, True, 1.0, backward=True)
    x = {k: _to(v, layout) for k, v in rin.make(w).items()}
    dev = {k: v.cuda() for k, v in x.items()}
    Yd, Ld = rb.fwd(dev["P1"], dev["P2"], dev["V"], w.tau_S, w.lam, True, layout=layout)
    g = rb.bwd(dev["P1"], dev["P2"], dev["V"], Yd, Ld, dev["dY"], w.tau_S, w.lam, True, layout=layout)
    h = {k: _pinned(v) for k, v in x.items()}
    Y, L, dP1, dP2, dV, dlam = rb.step_host(h["P1"], h["P2"], h["V"], h["dY"], w.tau_S, w.lam, True, chunks=chunks,
                                            want_L=True, layout=layout)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    assert torch.equal(Y, Yd.cpu())
    assert torch.equal(L, Ld.cpu())
    if dtype == torch.bfloat16:  # the tensor-core kernels accumulate dP2 and dV in a fixed order
        assert torch.equal(dP2, g[1].cpu())
        assert torch.equal(dV, g[2].cpu())
    else:
        for got, ref in ((dP2, g[1].cpu()), (dV, g[2].cpu())):
            assert float((got - ref).abs().max()) <= 1e-6 * float(ref.abs().max())
    ref1 = g[0].float().cpu()
    assert float((dP1.float() - ref1).abs().max()) <= 2.0 ** -7 * float(ref1.abs().max())
    lam_ref = float(g[3].cpu())
    assert abs(float(dlam) - lam_ref) <= 1e-4 * max(1.0, abs(lam_ref))


def test_step_host_against_the_oracle():
    w = rin.Workload("host_oracle", 4, 2, 150, 64, torch.bfloat16, 2.0, 0.5, True, 1.0, backward=True)
    x = rin.make(w)
    h = {k: _pinned(v) for k, v in x.items()}
    Y, L, dP1, dP2, dV, dlam = rb.step_host(h["P1"], h["P2"], h["V"], h["dY"], w.tau_S, w.lam, True, chunks=2,
                                            want_L=True)
    torch.cuda.synchronize()
    xs = {k: v.double().numpy() for k, v in x.items()}
    rY, rL = oracle.fwd(xs["P1"], xs["P2"], xs["V"], w.tau_S, w.lam, True)
    gP1, gP2, gV, glam = oracle.bwd(xs["P1"], xs["P2"], xs["V"], xs["dY"], w.tau_S, w.lam, True)
    assert np.max(np.abs(Y.double().numpy() - rY)) <= 1e-2 * np.max(np.abs(xs["V"]))
    assert np.max(np.abs(L.double().numpy() - rL) / np.maximum(1.0, np.abs(rL))) <= 1e-3
    for got, ref in ((dP1, gP1), (dP2, gP2), (dV, gV)):
        assert np.max(np.abs(got.double().numpy() - ref)) <= 2e-2 * np.max(np.abs(ref))
    assert abs(float(dlam) - float(glam)) <= 2e-2 * max(1.0, abs(float(glam)))


def test_step_host_reuses_its_buffer_and_queues_on_the_stream():
    """Two steps through one device buffer on a side stream: the second's results are the
    first's (same inputs), and the stream's completion covers every copy out."""
    w = rin.Workload("host_twice", 4, 2, 256, 64, torch.bfloat16, 1.0, 0.5, True, 1.0, backward=True)
    x = {k: _pinned(v) for k, v in rin.make(w).items()}
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, True)
    buf = torch.empty((rb.relation_step_host_device_bytes(prob, 4) + 3) // 4, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    first = rb.step_host(x["P1"], x["P2"], x["V"], x["dY"], w.tau_S, w.lam, True, chunks=4, device_buffer=buf,
                         stream=s)
    second = rb.step_host(x["P1"], x["P2"], x["V"], x["dY"], w.tau_S, w.lam, True, chunks=4, device_buffer=buf,
                          stream=s)
    s.synchronize()
    for a, b in ((first[0], second[0]), (first[3], second[3]), (first[4], second[4])):
        assert torch.equal(a, b)
    assert float((first[2].float() - second[2].float()).abs().max()) <= 2.0 ** -7 * float(first[2].float().abs().max())
