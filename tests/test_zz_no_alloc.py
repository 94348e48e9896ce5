"""relation_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (code whose device memory belongs to a host framework's allocator
they cannot reach, serving loops that must not allocate once running) get the
backward with the library's own fixed scratch array as workspace.  These tests
call it through the C ABI and compare it with relation_bwd given a caller
workspace, on two calls in a row with different problems, so that the second
call starts from the first call's leftovers in the shared array.

This file is named to be collected last; it also runs on its own in a fresh
process (the binding builds and loads the library itself).
"""
import ctypes

import numpy as np
import pytest
import torch

from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

# the tolerances of the parity tests: bf16 gradients within 2e-2 * max|g|, fp32 within 1e-4 * max|g|
G_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def _case(B, H, T, d, dtype, causal=True, seed=0):
    w = rin.Workload("noalloc", B, H, T, d, dtype, 1.0, 0.5, causal, backward=True,
                     seeds={k: v + seed for k, v in rin.SEEDS.items()})
    x = {k: v.cuda() for k, v in rin.make(w).items()}
    Y, L = rb.fwd(x["P1"], x["P2"], x["V"], w.tau_S, w.lam, causal)
    return w, x, Y, L


def _with_workspace(w, x, Y, L):
    return rb.bwd(x["P1"], x["P2"], x["V"], Y, L, x["dY"], w.tau_S, w.lam, w.causal)


def _noalloc(w, x, Y, L):
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, w.causal)
    dP1, dP2, dV = (torch.full_like(x["V"], float("nan")) for _ in range(3))
    dlam = torch.full((1,), float("nan"), device="cuda")
    rb.relation_bwd_noalloc(prob, x["P1"], x["P2"], x["V"], Y, L, x["dY"], dP1, dP2, dV, dlam)
    return dP1, dP2, dV, dlam


def _compare(w, got, ref):
    for g, r in zip(got[:3], ref[:3]):
        r64 = r.double()
        tol = G_TOL[w.dtype] * max(float(r64.abs().max()), 1e-30)
        assert torch.isfinite(g).all()
        assert float((g.double() - r64).abs().max()) <= tol
    assert abs(float(got[3].item()) - float(ref[3].item())) <= 5 * G_TOL[w.dtype] * max(1.0, abs(float(ref[3])))


def test_noalloc_matches_workspace_backward_on_two_calls_in_a_row():
    cases = [_case(2, 3, 300, 64, torch.bfloat16, seed=0), _case(1, 2, 200, 128, torch.bfloat16, seed=7)]
    for w, x, Y, L in cases:
        ref = _with_workspace(w, x, Y, L)
        got = _noalloc(w, x, Y, L)
        torch.cuda.synchronize()
        assert rb.relation_check_device_status() == 0
        _compare(w, got, ref)


def test_noalloc_reserves_nothing_after_the_first_call():
    """After a first call (which may be when the driver reserves the array on
    this device), further calls leave the device's free memory unchanged."""
    w, x, Y, L = _case(1, 2, 260, 64, torch.bfloat16, seed=3)
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, w.causal)
    outs = [torch.empty_like(x["V"]) for _ in range(3)]
    dlam = torch.empty((1,), device="cuda")
    rb.relation_bwd_noalloc(prob, x["P1"], x["P2"], x["V"], Y, L, x["dY"], *outs, dlam)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        rb.relation_bwd_noalloc(prob, x["P1"], x["P2"], x["V"], Y, L, x["dY"], *outs, dlam)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
    assert rb.relation_check_device_status() == 0


def test_noalloc_fp32_path_twice():
    for seed in (1, 2):
        w, x, Y, L = _case(1, 2, 150, 64, torch.float32, causal=seed == 1, seed=seed)
        ref = _with_workspace(w, x, Y, L)
        got = _noalloc(w, x, Y, L)
        torch.cuda.synchronize()
        _compare(w, got, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = rb.load()
    p = rb.Problem(4, 16, 4096, 64, rb.RELATION_BF16, 1.0, 0.5, 1)  # needs ~68 MB of workspace
    assert rb.relation_bwd_workspace_bytes(p) > (32 << 20)
    fake = [0x10000 * k for k in range(1, 11)]
    assert lib.relation_bwd_noalloc(ctypes.byref(p), *fake, None) == 4  # RELATION_ERR_WORKSPACE_TOO_SMALL
    bad = rb.Problem(1, 1, 128, 64, rb.RELATION_BF16, -1.0, 0.5, 1)
    assert lib.relation_bwd_noalloc(ctypes.byref(bad), *fake, None) == 1
