"""The persistent backward (d_h <= 64): a CTA that has issued its key tile's loads takes the key
tile of a CTA not yet launched, through launch control, so with more key tiles than SMs most are
computed by CTAs other than their own.  Checked in full against the same backward run one head at
a time (8 key tiles per call, fewer CTAs than SMs, so nothing is taken over): every key tile's dP2
and dV rows come from one CTA's fixed sequence of products, so they must be bit-identical; dP1
adds the key tiles' partials in an order the GPU picks (within 2^-7 max|dP1|, one bf16 rounding),
and dlambda is the sum over heads (within 1e-4 relative)."""
import pytest
import torch

from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,T,causal", [(2, 64, 1024, True), (1, 48, 640, False)], ids=["causal", "noncausal"])
def test_taken_over_key_tiles_equal_one_head_at_a_time(B, H, T, causal):
    w = rin.Workload("persist", B, H, T, 64, torch.bfloat16, 1.0, 0.5, causal, 1.0, backward=True)
    x = {k: v.cuda() for k, v in rin.make(w).items()}
    Y, L = rb.fwd(x["P1"], x["P2"], x["V"], w.tau_S, w.lam, causal)
    dP1, dP2, dV, dlam = rb.bwd(x["P1"], x["P2"], x["V"], Y, L, x["dY"], w.tau_S, w.lam, causal)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    lam_sum = 0.0
    for b in range(B):
        for h in range(H):
            sl = lambda t: t[b:b + 1, h:h + 1].contiguous()  # noqa: E731
            g = rb.bwd(sl(x["P1"]), sl(x["P2"]), sl(x["V"]), sl(Y), sl(L), sl(x["dY"]), w.tau_S, w.lam, causal)
            assert torch.equal(g[1][0, 0], dP2[b, h])
            assert torch.equal(g[2][0, 0], dV[b, h])
            ref = g[0][0, 0].float()
            assert float((dP1[b, h].float() - ref).abs().max()) <= 2.0 ** -7 * float(ref.abs().max())
            lam_sum += float(g[3])
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    assert abs(float(dlam) - lam_sum) <= 1e-4 * max(1.0, abs(lam_sum))
