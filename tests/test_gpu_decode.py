"""GPU parity of Relation Cache decoding ("Ask Self, Ask Others", Sec. 5.3 eq.(18),
Appendix A.5) through the C ABI.

The new row at position t+1 must equal row t+1 of the causal operator over the t+1
tokens, so the reference is the float64 oracle's selected-row forward at row t of the
full sequences (the cache holds rows 0..t-1 of P2 and V, the new token is row t).  Cache
rows past each batch's position are filled with NaN: reading one would poison Y.
Tolerances: fp32 <= 1e-5 * max|V|; bf16 <= 1e-2 * max|V| (fp32 arithmetic on bf16
inputs, bf16 output), as for the forward.
"""
import numpy as np
import pytest
import torch

import oracle
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

Y_TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}
L_TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-3}
BHTD, BTHD = rb.RELATION_LAYOUT_BHTD, rb.RELATION_LAYOUT_BTHD


def _to_layout(t, layout):
    return t.permute(0, 2, 1, 3).contiguous() if layout == BTHD else t.contiguous()


def _setup(B, H, T, d, dtype, positions, tau, lam, layout):
    w = rin.Workload("decode", B, H, T, d, dtype, tau, lam, True, 1.0)
    x = rin.make(w)  # [B, H, T, d]
    P2c = x["P2"].clone()
    Vc = x["V"].clone()
    for b, t in enumerate(positions):  # history only: rows >= t are never read
        P2c[b, :, t:] = float("nan")
        Vc[b, :, t:] = float("nan")
    idx = torch.tensor(positions)
    new = {k: torch.stack([x[k][b, :, positions[b]] for b in range(B)]) for k in ("P1", "P2", "V")}  # [B, H, d]
    dev = dict(P1n=new["P1"].cuda(), P2n=new["P2"].cuda(), Vn=new["V"].cuda(),
               P2c=_to_layout(P2c, layout).cuda(), Vc=_to_layout(Vc, layout).cuda(),
               pos=idx.to(torch.int32).cuda())
    return x, dev


def _reference(x, positions, H, tau, lam):
    heads = [b * H + h for b in range(len(positions)) for h in range(H)]
    rows = [positions[b] for b in range(len(positions)) for _ in range(H)]
    Y, L = oracle.fwd_rows(x["P1"], x["P2"], x["V"], tau, lam, True, heads, rows)
    return Y.reshape(len(positions), H, -1), L.reshape(len(positions), H)


CASES = [
    ("bf16_d64", 3, 2, 1100, 64, torch.bfloat16, [0, 37, 1099], BHTD),
    ("bf16_d64_bthd", 2, 3, 700, 64, torch.bfloat16, [512, 699], BTHD),
    ("bf16_d48", 2, 2, 600, 48, torch.bfloat16, [1, 513], BHTD),
    ("bf16_d60", 2, 2, 600, 60, torch.bfloat16, [255, 599], BHTD),
    ("bf16_d80_bthd", 2, 2, 300, 80, torch.bfloat16, [5, 299], BTHD),
    ("bf16_d128", 1, 4, 2100, 128, torch.bfloat16, [2047], BHTD),
    ("f32_d64", 2, 2, 600, 64, torch.float32, [0, 599], BHTD),
    ("f32_d60_bthd", 2, 2, 300, 60, torch.float32, [17, 290], BTHD),
    # the remaining bulk-copy instantiations ([B, H, T, d], 16-byte rows), with the new token
    # first in its chunk (that chunk copies no cached row) and last in its chunk
    ("bf16_d80", 2, 2, 700, 80, torch.bfloat16, [128, 699], BHTD),
    ("f32_d48", 2, 2, 600, 48, torch.float32, [127, 599], BHTD),
    ("f32_d60", 2, 2, 300, 60, torch.float32, [128, 299], BHTD),
    ("f32_d80", 2, 2, 400, 80, torch.float32, [64, 399], BHTD),
    ("f32_d128", 2, 2, 300, 128, torch.float32, [63, 299], BHTD),
    ("f32_d128_bthd", 2, 2, 300, 128, torch.float32, [100, 299], BTHD),
]


@pytest.mark.parametrize("name,B,H,T,d,dtype,positions,layout", CASES, ids=[c[0] for c in CASES])
def test_decode_row_matches_oracle(name, B, H, T, d, dtype, positions, layout):
    tau, lam = 1.0, 0.5
    x, g = _setup(B, H, T, d, dtype, positions, tau, lam, layout)
    Y, L = rb.decode(g["P1n"], g["P2n"], g["Vn"], g["P2c"], g["Vc"], g["pos"], tau, lam, append=False,
                     layout=layout)
    # One cluster launch for caches the streaming pass reads ([B, H, T, d], rows a
    # multiple of 16 bytes); a partial pass and a merge otherwise.
    streamed = layout == BHTD and (d * (2 if dtype == torch.bfloat16 else 4)) % 16 == 0
    assert rb.relation_last_launch_count() == (1 if streamed else 2)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    Yr, Lr = _reference(x, positions, H, tau, lam)
    vmax = float(x["V"].abs().max())
    assert np.max(np.abs(Y.float().cpu().numpy() - Yr)) <= Y_TOL[dtype] * vmax
    assert np.max(np.abs(L.cpu().numpy() - Lr)) <= L_TOL[dtype]


def test_first_token_is_its_own_state():
    """t = 0: the row holds only the Self entry, so Y = V_new exactly (Appendix A.1.7)."""
    x, g = _setup(2, 3, 64, 64, torch.bfloat16, [0, 0], 1.0, 0.5, BHTD)
    Y, _ = rb.decode(g["P1n"], g["P2n"], g["Vn"], g["P2c"], g["Vc"], g["pos"], 1.0, 0.5, append=False)
    torch.cuda.synchronize()
    assert torch.equal(Y, g["Vn"])


@pytest.mark.parametrize("layout", [BHTD, BTHD])
def test_append_writes_row_t_only(layout):
    positions = [3, 200]
    x, g = _setup(2, 2, 256, 64, torch.bfloat16, positions, 1.0, 0.5, layout)
    before_p2, before_v = g["P2c"].clone(), g["Vc"].clone()
    rb.decode(g["P1n"], g["P2n"], g["Vn"], g["P2c"], g["Vc"], g["pos"], 1.0, 0.5, append=True, layout=layout)
    torch.cuda.synchronize()
    for cache, before, new in ((g["P2c"], before_p2, g["P2n"]), (g["Vc"], before_v, g["Vn"])):
        c = cache if layout == BHTD else cache.permute(0, 2, 1, 3)
        bfr = before if layout == BHTD else before.permute(0, 2, 1, 3)
        for b, t in enumerate(positions):
            assert torch.equal(c[b, :, t], new[b])
            rest = torch.cat([c[b, :, :t], c[b, :, t + 1:]], dim=1)
            rest_b = torch.cat([bfr[b, :, :t], bfr[b, :, t + 1:]], dim=1)
            assert torch.equal(torch.nan_to_num(rest, nan=7.0), torch.nan_to_num(rest_b, nan=7.0))


def test_autoregressive_decoding_reproduces_the_full_forward():
    """Decoding token by token with cache appends gives every row of the full causal
    forward (the cache is exact, Appendix A.5)."""
    B, H, T, d, tau, lam = 2, 2, 96, 64, 0.7, 0.5
    w = rin.Workload("ar", B, H, T, d, torch.bfloat16, tau, lam, True, 1.0)
    x = rin.make(w)
    P2c = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    Vc = torch.zeros_like(P2c)
    dev = {k: v.cuda() for k, v in x.items()}
    Yr, _ = oracle.fwd(x["P1"], x["P2"], x["V"], tau, lam, True)
    vmax = float(x["V"].abs().max())
    worst = 0.0
    for t in range(T):
        pos = torch.full((B,), t, dtype=torch.int32, device="cuda")
        Y, _ = rb.decode(dev["P1"][:, :, t].contiguous(), dev["P2"][:, :, t].contiguous(),
                         dev["V"][:, :, t].contiguous(), P2c, Vc, pos, tau, lam, append=True)
        worst = max(worst, float(np.max(np.abs(Y.float().cpu().numpy() - Yr[:, :, t]))))
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    assert worst <= Y_TOL[torch.bfloat16] * vmax, worst


def test_position_outside_cache_is_reported():
    x, g = _setup(2, 2, 128, 64, torch.bfloat16, [5, 10], 1.0, 0.5, BHTD)
    g["pos"][1] = 128  # == capacity: invalid
    Y = torch.full_like(g["P1n"], 3.0)
    L = torch.empty(2, 2, device="cuda")
    prob = rb.Problem(2, 2, 128, 64, rb.RELATION_BF16, 1.0, 0.5, 1, BHTD)
    ws = torch.empty((rb.relation_decode_workspace_bytes(prob) + 3) // 4, device="cuda")
    rb.relation_decode(prob, g["P1n"], g["P2n"], g["Vn"], g["P2c"], g["Vc"], g["pos"], 0, Y, L, ws)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 1  # RELATION_ERR_INVALID_ARGUMENT
    assert rb.relation_check_device_status() == 0  # cleared
    assert torch.all(Y[1] == 3.0)  # the skipped batch is not written
    Yr, _ = _reference(x, [5, 10], 2, 1.0, 0.5)
    assert np.max(np.abs(Y[0].float().cpu().numpy() - Yr[0])) <= 1e-2 * float(x["V"].abs().max())


def test_decode_benchmark_workload_every_head():
    """bench.py --decode at full size: the headline workload's tensors (B4 H16 T4096 d64, large
    |U|, tau 0.5, lambda 0.5), 4095 cached tokens per sequence, decoding token 4096; every
    head's row against the oracle."""
    w = rin.WORKLOADS["mhr_fwd_bwd_T4096"]
    x = rin.make(w)
    t = w.T - 1
    dev = {k: v.cuda() for k, v in x.items()}
    P1n, P2n, Vn = (dev[k][:, :, t].contiguous() for k in ("P1", "P2", "V"))
    pos = torch.full((w.B,), t, dtype=torch.int32, device="cuda")
    Y, L = rb.decode(P1n, P2n, Vn, dev["P2"], dev["V"], pos, w.tau_S, w.lam, append=False)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    heads = list(range(w.B * w.H))
    Yr, Lr = oracle.fwd_rows(x["P1"], x["P2"], x["V"], w.tau_S, w.lam, True, heads, [t] * len(heads))
    vmax = float(x["V"].abs().max())
    assert np.max(np.abs(Y.float().cpu().numpy().reshape(len(heads), -1) - Yr)) <= Y_TOL[torch.bfloat16] * vmax
    assert np.max(np.abs(L.cpu().numpy().reshape(-1) - Lr.reshape(-1))) <= L_TOL[torch.bfloat16]
