#!/usr/bin/env python3
"""Benchmark of the fused Full Relation forward + backward on GB300.

One step = relation_fwd + relation_bwd (prepare, main, finish) over one batch
of seeded synthetic bf16 inputs already resident in HBM.  Default workload:
causal, B=4, H=16, T=4096, d_h=64, tau_S=0.5, lambda=0.5, P1/P2 ~ N(0,1)*3/d^(1/4),
V, dY ~ N(0,1).  Throughput counts algorithmic work: 4*d flops per visible
pair forward, 8*d backward (the U recompute of the backward is not counted).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
L2_CLEAN_BYTES = 256 << 20  # read after the flush, so that no dirty line of it is left to write back
L2_NOTE = ("flushed between timed steps: 512 MB written, then 256 MB of another buffer read, outside the "
           "events (the read leaves only clean lines, so no write-back of the flush lands in the timed region)")


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer larger than L2, then reads another one
    so that the lines left in L2 are clean (the written lines would otherwise be written
    back to HBM during the next timed kernel)."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        return self.r.sum()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="mhr_fwd_bwd_T4096")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="batch slices of relation_step_host in the e2e measurement (copies overlap the kernels)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", action="store_true",
                    help="time one Relation Cache decode step (full caches of the workload's T) instead")
    ap.add_argument("--prologue", action="store_true",
                    help="time the input prologue (RoPE + Givens) forward and backward of the workload instead")
    ap.add_argument("--prologue-fused", action="store_true",
                    help="time the operator step with the input prologue fused into its kernels' loads, beside "
                         "the plain operator step and the two-call chain (prologue passes + operator)")
    ap.add_argument("--linear", action="store_true",
                    help="time Linear Relation forward + backward (workload from the linear set, default "
                         "linear_d60_T2048) instead")
    return ap.parse_args()


def pairs(T: int, causal: bool) -> int:
    return T * (T + 1) // 2 if causal else T * T


def flops(w, per_pair: int) -> float:
    return float(per_pair) * w.d * pairs(w.T, w.causal) * w.B * w.H


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured"
    return 1900.0, 1700.0, "fallback"


def kernel_source_hash(names) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "relation_token_mixing_gb300", "csrc")
    for n in names:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, source_hash: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this workload and
    matches the current source.  A kernel captured on several workloads has one entry per extra
    workload, keyed "<kernel> @ <workload>"."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(f"{kernel} @ {workload}") or rec.get(kernel)
    if not e or e.get("source_hash") != source_hash or e.get("workload") != workload:
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for k, n in enumerate(names):
                if parts[5 + k].lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def decode_bytes_per_step(w, t: int) -> int:
    """Algorithmic HBM bytes of one decoding step (bf16): both caches' t rows, the new token's
    three rows, Y and L, for every head."""
    e = 2
    return w.B * w.H * (2 * t * w.d * e + 3 * w.d * e + w.d * e + 4)


def decode_kernels(w) -> str:
    """The decoding kernels the bench's [B, H, T, d] bf16 caches run on."""
    if (w.d * 2) % 16 == 0:
        return "decode_cluster_kernel"  # streaming pass and in-cluster merge, one launch
    return "decode_partial_kernel + decode_combine_kernel"


def decode_config(w, t: int) -> dict:
    return {"workload": f"decode_{w.name}", "B": w.B, "H": w.H, "cache_tokens": t, "d_h": w.d,
            "tau_S": w.tau_S, "lambda": w.lam, "l2": L2_NOTE}


PROLOGUE_PAIRING, PROLOGUE_BASE = 1, 1e4


def prologue_bytes_per_step(w) -> int:
    """Algorithmic HBM bytes of the prologue forward (P1, P2, V in; three out) and backward
    (three gradients and the mixed states in; three out), bf16."""
    tb = w.B * w.H * w.T * w.d * 2
    return (3 + 3) * tb + (4 + 3) * tb


def prologue_config(w) -> dict:
    return {"workload": f"prologue_{w.name}", "B": w.B, "H": w.H, "T": w.T, "d_h": w.d, "pairing": "B",
            "rope_base": PROLOGUE_BASE, "l2": L2_NOTE}


def relation_config(w, world: int) -> dict:
    """The `config` of every Relation fwd+bwd line (both arms): the workload, not the sample."""
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d_h": w.d, "causal": w.causal,
            "tau_S": w.tau_S, "lambda": w.lam, "p_scale": round(w.p_scale, 6),
            "parallelism": f"independent heads, {world} replica(s)", "l2": L2_NOTE}


def linear_config(w, world: int) -> dict:
    """The `config` of every Linear Relation line (both arms)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d_h": w.d, "tau_S": w.tau_S,
            "g_scale": w.g_scale, "parallelism": f"independent heads, {world} replica(s)", "l2": L2_NOTE}


def cpu_baseline(w, target_s: float = 12.0):
    """The float64 oracle (as it stands) on a bounded sample of the workload: whole heads at the
    workload's T and d.  A first pass runs one head per oracle thread; when it ends well inside
    target_s, the sample grows by whole multiples of the thread count toward target_s (at most
    the whole workload) and that second pass is the one reported."""
    import oracle
    from relation_token_mixing_gb300 import inputs as rin

    threads = oracle.threads()
    total = w.B * w.H

    def timed_pass(heads):
        b, h = (heads // w.H, w.H) if heads % w.H == 0 else (1, heads)
        ws = rin.Workload(w.name, b, h, w.T, w.d, w.dtype, w.tau_S, w.lam, w.causal, w.p_scale, backward=True)
        x = rin.make(ws)
        t0 = time.perf_counter()
        oracle.fwd(x["P1"], x["P2"], x["V"], ws.tau_S, ws.lam, ws.causal)
        oracle.bwd(x["P1"], x["P2"], x["V"], x["dY"], ws.tau_S, ws.lam, ws.causal)
        return ws, time.perf_counter() - t0

    heads = min(total, max(1, threads))
    ws, dt = timed_pass(heads)
    grow = min(total // heads, int(target_s / max(dt, 1e-9)))
    if dt < target_s / 2 and grow >= 2:
        heads *= grow
        ws, dt = timed_pass(heads)
    value = flops(ws, 12) / dt / 1e12
    part = "the whole workload" if heads == total else f"{heads} of {total} heads"
    return {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"fwd+bwd of B={ws.B} H={ws.H} ({part}) at T={w.T} d={w.d}, float64, {dt:.1f} s"}


def run_decode(args, w):
    """One Relation Cache step per timed iteration: every sequence has T-1 cached tokens
    (full caches of capacity T) and decodes token T; caches are not appended, so every
    step reads the same state.  HBM-bound: value = cache bytes read / time."""
    import torch

    from relation_token_mixing_gb300 import binding as rb
    from relation_token_mixing_gb300 import inputs as rin

    rb.load()
    dev = torch.device("cuda", 0)
    x = {k: v.to(dev) for k, v in rin.make(w).items()}
    t = w.T - 1
    P1n, P2n, Vn = (x[k][:, :, t].contiguous() for k in ("P1", "P2", "V"))
    P2c, Vc = x["P2"], x["V"]
    pos = torch.full((w.B,), t, dtype=torch.int32, device=dev)
    prob = rb.Problem(w.B, w.H, w.T, w.d, rb.RELATION_BF16, w.tau_S, w.lam, 1, rb.RELATION_LAYOUT_BHTD)
    ws = torch.empty((rb.relation_decode_workspace_bytes(prob) + 3) // 4, dtype=torch.float32, device=dev)
    Y = torch.empty_like(P1n)
    L = torch.empty(w.B, w.H, dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    bytes_step = decode_bytes_per_step(w, t)
    times = []
    with ClockSampler(0) as clk:
        for k in range(args.warmup + args.steps):
            flush()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev[0].record()
            rb.relation_decode(prob, P1n, P2n, Vn, P2c, Vc, pos, 0, Y, L, ws)
            ev[1].record()
            torch.cuda.synchronize()
            if k >= args.warmup:
                times.append(ev[0].elapsed_time(ev[1]))
    assert rb.relation_check_device_status() == 0
    ms = statistics.mean(times)
    hbm = load_peaks_hbm()
    line = {
        "metric": "Relation Cache decode: cache bytes read per second (bf16)",
        "value": bytes_step / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 arithmetic on bf16", "data": "synthetic (seeded Gaussian caches, resident in HBM)",
        "config": decode_config(w, t),
        "tokens_per_s": w.B / (ms * 1e-3),
        "roofline": {"kernel": decode_kernels(w), "bound": "hbm",
                     "achieved": bytes_step / (ms * 1e-3) / 1e9, "peak": hbm[0], "unit": "GB/s",
                     "frac": bytes_step / (ms * 1e-3) / 1e9 / hbm[0], "peak_source": hbm[1], "traffic": None},
        "gpu_launches": (1 if (w.d * 2) % 16 == 0 else 2) * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        heads = list(range(w.B * w.H))  # the whole decoding step (one row per head is cheap for the oracle)
        xc = {k: x[k].cpu() for k in ("P1", "P2", "V")}  # host copies made before the oracle's clock starts
        t0 = time.perf_counter()
        oracle.fwd_rows(xc["P1"], xc["P2"], xc["V"], w.tau_S, w.lam, True, heads, [t] * len(heads))
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": bytes_step * len(heads) / (w.B * w.H) / dt / 1e9, "unit": "GB/s",
                                "cores": oracle.threads(), "kind": "oracle",
                                "sample": f"row {t} of all {len(heads)} heads (the whole workload), float64, "
                                          f"{dt:.2f} s"}
    print(json.dumps(line), flush=True)
    return 0


def run_prologue(args, w):
    """Prologue forward (RoPE of P1, P2; Givens mixing of V) plus backward (transposed
    rotations and d theta) of the workload's tensors, inputs larger than L2.  HBM-bound:
    value = bytes read and written / time."""
    import torch

    from relation_token_mixing_gb300 import binding as rb
    from relation_token_mixing_gb300 import inputs as rin

    rb.load()
    dev = torch.device("cuda", 0)
    x = {k: v.to(dev) for k, v in rin.make(w, with_dy=True).items()}
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, True)
    theta = torch.linspace(-1.0, 1.0, w.H // 2, device=dev)
    outs = [torch.empty_like(x["P1"]) for _ in range(3)]
    grads = [torch.empty_like(x["P1"]) for _ in range(3)]
    dth = torch.empty(w.H // 2, device=dev)
    flush = L2Flush(dev)
    bytes_step = prologue_bytes_per_step(w)
    tf, tbw = [], []
    with ClockSampler(0) as clk:
        for k in range(args.warmup + args.steps):
            flush()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record()
            rb.relation_prologue_fwd(prob, x["P1"], x["P2"], x["V"], theta, PROLOGUE_PAIRING, PROLOGUE_BASE, None,
                                     *outs)
            ev[1].record()
            rb.relation_prologue_bwd(prob, x["dY"], x["dY"], x["dY"], outs[2], theta, PROLOGUE_PAIRING,
                                     PROLOGUE_BASE, None, *grads, dth)
            ev[2].record()
            torch.cuda.synchronize()
            if k >= args.warmup:
                tf.append(ev[0].elapsed_time(ev[1]))
                tbw.append(ev[1].elapsed_time(ev[2]))
    ms = statistics.mean(tf) + statistics.mean(tbw)
    hbm = load_peaks_hbm()
    gbs = bytes_step / (ms * 1e-3) / 1e9
    line = {
        "metric": "Relation input prologue (RoPE + Givens) fwd+bwd bytes per second (bf16)",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 arithmetic on bf16",
        "data": "synthetic (seeded Gaussian tensors, resident in HBM)",
        "config": prologue_config(w),
        "breakdown_ms": {"fwd": statistics.mean(tf), "bwd": statistics.mean(tbw)},
        "roofline": {"kernel": "rope_kernel + givens_kernel", "bound": "hbm", "achieved": gbs, "peak": hbm[0],
                     "unit": "GB/s", "frac": gbs / hbm[0], "peak_source": hbm[1], "traffic": None},
        "gpu_launches": 4 * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_prologue_fused(args, w):
    """One step = relation_fwd_prologue + relation_bwd_prologue (X1 = P1, X2 = P2, I = V of the
    workload; RoPE base 1e4, pairing B, theta = linspace(-1, 1, H/2)).  Timed beside the plain
    operator step (relation_fwd + relation_bwd on the same tensors) and the two-call chain
    (relation_prologue_fwd, the operator step, relation_prologue_bwd), each with the L2 flushed
    before every step.  value = the operator's algorithmic TFLOP/s over the fused step."""
    import torch

    from relation_token_mixing_gb300 import binding as rb
    from relation_token_mixing_gb300 import inputs as rin

    rb.load()
    dev = torch.device("cuda", 0)
    x = {k: v.to(dev) for k, v in rin.make(w, with_dy=True).items()}
    prob = rb.problem_for(x["P1"], w.tau_S, w.lam, w.causal)
    theta = torch.linspace(-1.0, 1.0, w.H // 2, device=dev)
    Y = torch.empty_like(x["V"])
    L = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
    g = [torch.empty_like(x["P1"]) for _ in range(3)]
    dth = torch.empty(w.H // 2, device=dev)
    dlam = torch.empty(1, device=dev)
    wsp = torch.empty((rb.relation_bwd_prologue_workspace_bytes(prob) + 3) // 4, dtype=torch.float32, device=dev)
    ws = torch.empty((rb.relation_bwd_workspace_bytes(prob) + 3) // 4, dtype=torch.float32, device=dev)
    pro = [torch.empty_like(x["P1"]) for _ in range(3)]
    flush = L2Flush(dev)

    def fused():
        rb.relation_fwd_prologue(prob, x["P1"], x["P2"], x["V"], theta, PROLOGUE_PAIRING, PROLOGUE_BASE, None, Y, L)
        rb.relation_bwd_prologue(prob, x["P1"], x["P2"], x["V"], theta, PROLOGUE_PAIRING, PROLOGUE_BASE, None, Y, L,
                                 x["dY"], *g, dth, dlam, wsp)

    def operator(P1, P2, V):
        rb.relation_fwd(prob, P1, P2, V, Y, L)
        rb.relation_bwd(prob, P1, P2, V, Y, L, x["dY"], *g, dlam, ws)

    def chain():
        rb.relation_prologue_fwd(prob, x["P1"], x["P2"], x["V"], theta, PROLOGUE_PAIRING, PROLOGUE_BASE, None, *pro)
        operator(*pro)
        rb.relation_prologue_bwd(prob, g[0], g[1], g[2], pro[2], theta, PROLOGUE_PAIRING, PROLOGUE_BASE, None,
                                 *g_chain, dth)

    g_chain = [torch.empty_like(x["P1"]) for _ in range(3)]
    arms = {"fused": fused, "operator": lambda: operator(x["P1"], x["P2"], x["V"]), "chain": chain}
    times = {k: [] for k in arms}
    with ClockSampler(0) as clk:
        for k in range(args.warmup + args.steps):
            for name, fn in arms.items():
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                if k >= args.warmup:
                    times[name].append(e0.elapsed_time(e1))
    if rb.relation_check_device_status() != 0:
        raise RuntimeError("device-side wait expired")
    ms = {k: statistics.mean(v) for k, v in times.items()}
    value = flops(w, 12) / (ms["fused"] * 1e-3) / 1e12
    peak_burst, _, peak_src = load_peaks()
    peak = (peak_burst, f"{peak_src} bf16 burst")
    line = {
        "metric": "Relation fwd+bwd with the input prologue fused into its loads, TFLOP/s (bf16, causal)",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms["fused"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded Gaussian inputs, resident in HBM)",
        "config": {"workload": f"prologue_fused_{w.name}", "B": w.B, "H": w.H, "T": w.T, "d_h": w.d,
                   "causal": w.causal, "tau_S": w.tau_S, "lambda": w.lam, "pairing": "B", "rope_base": PROLOGUE_BASE,
                   "l2": L2_NOTE},
        "breakdown_ms": {"fused_step": ms["fused"], "operator_step": ms["operator"], "two_call_chain": ms["chain"]},
        "fused_over_operator": ms["fused"] / ms["operator"],
        "fused_over_chain": ms["fused"] / ms["chain"],
        "roofline": {"kernel": "fused step (relation_fwd_tc_kernel + relation_bwd_tc64_kernel with the prologue)",
                     "bound": "tensor", "achieved": value, "peak": peak[0], "unit": "TFLOP/s",
                     "frac": value / peak[0], "peak_source": peak[1], "traffic": None},
        "gpu_launches": 5 * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def linear_bytes_per_head_token(d: int) -> int:
    """Algorithmic HBM bytes of one Linear Relation fwd+bwd per head and token: forward
    reads P1, P2, I~ (bf16) and G (fp32) and writes Y (bf16): 12 d; backward reads P1,
    P2, I~, dY (bf16) and G (fp32) and writes dP1, dP2, dI~ (bf16) and dG (fp32): 22 d."""
    return 34 * d


def linear_cpu_sample(w, target_s: float):
    """The float64 Linear Relation oracle (as it stands) on whole heads of the workload until
    about target_s seconds of CPU work; returns (head-tokens per second, heads, seconds)."""
    import numpy as np

    from oracle import linear as lo
    from relation_token_mixing_gb300 import inputs as rin

    x = rin.make_linear(rin.LinearWorkload(w.name, 1, 1, w.T, w.d, w.tau_S, w.g_scale, backward=True))
    xs = {k: v.float().numpy().astype(np.float64) for k, v in x.items()}
    heads, t0 = 0, time.perf_counter()
    while True:
        lo.fwd(xs["P1"], xs["P2"], xs["I"], xs["G"], w.tau_S)
        lo.bwd(xs["P1"], xs["P2"], xs["I"], xs["G"], w.tau_S, xs["dY"])
        heads += 1
        dt = time.perf_counter() - t0
        if dt >= target_s:
            return heads * w.T / dt, heads, dt


def run_linear(args, w):
    """Linear Relation forward + backward over B*H heads of length T, inputs larger than L2, the
    backward reusing the forward's segment states from the shared workspace (as a training step
    does).  value = tokens (B*T) per second; the roofline is HBM bytes of the whole step."""
    import torch

    from relation_token_mixing_gb300 import binding as rb
    from relation_token_mixing_gb300 import inputs as rin
    from relation_token_mixing_gb300 import replicas as rrep

    ranks = rrep.from_env()
    dev = torch.device("cuda", ranks.local)
    torch.cuda.set_device(dev)
    rrep.init(ranks, "nccl")
    rb.load()
    x_cpu = rin.make_linear(w)
    x = {k: v.to(dev) for k, v in x_cpu.items()}
    prob = rb.problem_for(x["P1"], w.tau_S, 0.0, True)
    ws = rb.linear_workspace(prob, dev)
    Y = torch.empty_like(x["I"])
    g = [torch.empty_like(x["P1"]), torch.empty_like(x["P2"]), torch.empty_like(x["I"]), torch.empty_like(x["G"])]
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    launches = [0]

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        rb.relation_linear_fwd(prob, x["P1"], x["P2"], x["I"], x["G"], Y, None, ws, stream)
        launches[0] += rb.relation_last_launch_count()
        if evs:
            evs[1].record(stream)
        rb.relation_linear_bwd(prob, x["P1"], x["P2"], x["I"], x["G"], x["dY"], *g, 1, ws, stream)
        launches[0] += rb.relation_last_launch_count()
        if evs:
            evs[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if rb.relation_check_device_status() != 0:
        raise RuntimeError("device-side wait expired during warm-up")
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    launches[0] = 0
    rrep.barrier(ranks)
    torch.cuda.synchronize()
    with ClockSampler(ranks.local) as clk:
        for k in range(args.steps):
            flush()
            step(evsets[k])
        torch.cuda.synchronize()
    rrep.barrier(ranks)
    if rb.relation_check_device_status() != 0:
        raise RuntimeError("device-side wait expired during the timed region")
    tf = [e[0].elapsed_time(e[1]) for e in evsets]
    tb = [e[1].elapsed_time(e[2]) for e in evsets]
    ms = rrep.max_over_ranks(ranks, statistics.mean(tf) + statistics.mean(tb), dev)
    tokens = w.B * w.T
    value = rrep.job_rate(ranks, tokens, ms * 1e-3)
    step_bytes = linear_bytes_per_head_token(w.d) * w.B * w.H * w.T
    gbs = step_bytes / (ms * 1e-3) / 1e9  # per GPU: the roofline is one device's
    hbm = load_peaks_hbm()

    e2e = None
    if not args.no_e2e:
        h_in = {k: v.pin_memory() for k, v in x_cpu.items()}
        h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in [Y] + g]

        def e2e_step():
            for k in ("P1", "P2", "I", "G", "dY"):
                x[k].copy_(h_in[k], non_blocking=True)
            step()
            for h, t in zip(h_out, [Y] + g):
                h.copy_(t, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = 0.0
        for _ in range(args.steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step()
            b.record(stream)
            b.synchronize()
            e_ms += a.elapsed_time(b)
        e_ms = rrep.max_over_ranks(ranks, e_ms, dev)
        e2e = {"value": rrep.job_rate(ranks, tokens * args.steps, e_ms * 1e-3), "unit": "tok/s",
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in h_in.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in h_out)}

    if ranks.rank != 0:
        rrep.finish(ranks)
        return 0
    line = {
        "metric": "Linear Relation fwd+bwd tokens per second (bf16 operands, fp32 state)",
        "value": value, "unit": "tok/s", "n_gpus": ranks.world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 operands, f32 state and accumulation",
        "data": "synthetic (seeded Gaussian P1, P2, I~, dY; log-retention G with the statistics of its "
                "initialisation), resident in HBM",
        "config": linear_config(w, ranks.world),
        "breakdown_ms": {"fwd": statistics.mean(tf), "bwd": statistics.mean(tb)},
        "roofline": {"kernel": "relation_linear_fwd + relation_linear_bwd (all launches)", "bound": "hbm",
                     "achieved": gbs, "peak": hbm[0], "unit": "GB/s", "frac": gbs / hbm[0],
                     "peak_source": hbm[1],
                     "traffic": recorded_traffic("linear fwd+bwd step",
                                                 kernel_source_hash(["linear.cu", "common.cuh", "ptx_sm100.cuh",
                                                                     "tile_copy.cuh"]), w.name),
                     "algorithmic_bytes_per_head_token": linear_bytes_per_head_token(w.d)},
        "gpu_launches": launches[0],
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and ranks.world == 1:
        try:
            rate, heads, dt = linear_cpu_sample(w, 10.0)
            line["cpu_baseline"] = {"value": rate / w.H, "unit": "tok/s", "cores": 1, "kind": "oracle",
                                    "sample": f"fwd+bwd of {heads} whole head(s) at T={w.T} d={w.d}, float64, "
                                              f"{dt:.1f} s; tok/s = head-tokens/s divided by H={w.H}"}
        except Exception as exc:
            line["cpu_baseline"] = {"value": None, "unit": "tok/s", "cores": None, "kind": "oracle",
                                    "sample": f"failed: {exc}"}
    print(json.dumps(line), flush=True)
    rrep.finish(ranks)
    return 0


def run_linear_reference(args, w):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    rate = []
    for _ in range(args.warmup):
        linear_cpu_sample(w, 0.0)
    for _ in range(args.steps):
        r, heads, dt = linear_cpu_sample(w, 0.0)
        rate.append(r / w.H)
    value = statistics.mean(rate)
    sample = f"each step: fwd+bwd of 1 whole head (of {w.B * w.H}) at T={w.T} d={w.d}, float64"
    print(json.dumps({
        "impl": "reference", "metric": "Linear Relation fwd+bwd tokens per second (bf16 operands, fp32 state)",
        "value": value, "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": w.T / w.H / value * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded, bf16-rounded then upcast)",
        "config": linear_config(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def load_peaks_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured copy"
    return 6800.0, "fallback"


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from relation_token_mixing_gb300 import inputs as rin

    threads = oracle.threads()
    heads = max(1, threads)
    ws = rin.Workload(w.name, 1, heads, w.T, w.d, w.dtype, w.tau_S, w.lam, w.causal, w.p_scale, backward=True)
    x = rin.make(ws)

    def step():
        oracle.fwd(x["P1"], x["P2"], x["V"], ws.tau_S, ws.lam, ws.causal)
        oracle.bwd(x["P1"], x["P2"], x["V"], x["dY"], ws.tau_S, ws.lam, ws.causal)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = flops(ws, 12) / dt / 1e12
    sample = f"each step: fwd+bwd of B=1 H={heads} (of {w.B * w.H} heads) at T={w.T} d={w.d}, float64"
    print(json.dumps({
        "impl": "reference", "metric": "Relation fwd+bwd TFLOP/s (bf16, causal) and % of GB300 dense bf16 peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Gaussian, bf16-rounded then upcast)",
        "config": relation_config(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def _reference_line(metric, unit, value, args, ms, config, sample, cores):
    return {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Gaussian, bf16-rounded then upcast)", "config": config,
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_decode_reference(args, w):
    """The float64 oracle's selected-row forward on row T-1 of every head: the whole decoding
    step of the workload, timed on the host cores."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import oracle
    from relation_token_mixing_gb300 import inputs as rin

    x = rin.make(w)
    t = w.T - 1
    heads = list(range(w.B * w.H))
    rows = [t] * len(heads)

    def step():
        oracle.fwd_rows(x["P1"], x["P2"], x["V"], w.tau_S, w.lam, True, heads, rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = decode_bytes_per_step(w, t) / dt / 1e9
    sample = f"each step: row {t} of all {len(heads)} heads (the whole workload), float64"
    print(json.dumps(_reference_line("Relation Cache decode: cache bytes read per second (bf16)", "GB/s", value,
                                     args, dt * 1e3, decode_config(w, t), sample, oracle.threads())))
    return 0


def run_prologue_reference(args, w):
    """The float64 prologue oracle (RoPE of P1 and P2, Givens mixing of V, and their backward
    with d theta) over the whole workload, timed on the host."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import numpy as np

    from oracle import prologue as po
    from relation_token_mixing_gb300 import inputs as rin

    # One whole batch (Givens mixing pairs heads inside a batch): a bounded sample.
    x = {k: v[:1].double().numpy() for k, v in rin.make(w, with_dy=True).items()}
    theta = np.linspace(-1.0, 1.0, w.H // 2)

    def step():
        po.rope(x["P1"], PROLOGUE_BASE)
        po.rope(x["P2"], PROLOGUE_BASE)
        mixed = po.givens(x["V"], theta, PROLOGUE_PAIRING)
        po.rope_bwd(x["dY"], PROLOGUE_BASE)
        po.rope_bwd(x["dY"], PROLOGUE_BASE)
        po.givens_bwd(x["dY"], mixed, theta, PROLOGUE_PAIRING)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = prologue_bytes_per_step(w) / w.B / dt / 1e9
    sample = f"each step: forward and backward of batch 1 of {w.B} ({w.H} heads, T={w.T}), float64 (numpy)"
    print(json.dumps(_reference_line("Relation input prologue (RoPE + Givens) fwd+bwd bytes per second (bf16)",
                                     "GB/s", value, args, dt * 1e3, prologue_config(w), sample, 1)))
    return 0


def main():
    args = parse()
    from relation_token_mixing_gb300 import inputs as rin

    if args.linear:
        name = args.workload if args.workload in rin.LINEAR_WORKLOADS else "linear_d60_T2048"
        lw = rin.LINEAR_WORKLOADS[name]
        return run_linear_reference(args, lw) if args.impl == "reference" else run_linear(args, lw)
    w = rin.WORKLOADS[args.workload]
    if args.decode:
        return run_decode_reference(args, w) if args.impl == "reference" else run_decode(args, w)
    if args.prologue:
        return run_prologue_reference(args, w) if args.impl == "reference" else run_prologue(args, w)
    if args.prologue_fused:
        if args.impl == "reference":
            return run_reference(args, w)
        return run_prologue_fused(args, w)
    if args.impl == "reference":
        return run_reference(args, w)

    import torch

    from relation_token_mixing_gb300 import binding as rb
    from relation_token_mixing_gb300 import replicas as rrep

    ranks = rrep.from_env()
    world, rank, local = ranks.world, ranks.rank, ranks.local
    if ranks.distributed:
        torch.cuda.set_device(local)
    rrep.init(ranks, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rb.load()

    # Inputs: every rank processes its own copy of the workload (independent heads; weak scaling).
    x_cpu = rin.make(w, with_dy=True)
    x = {k: v.to(dev) for k, v in x_cpu.items()}
    P1, P2, V, dY = x["P1"], x["P2"], x["V"], x["dY"]
    prob = rb.problem_for(P1, w.tau_S, w.lam, w.causal)
    Y = torch.empty_like(V)
    L = torch.empty(P1.shape[:3], dtype=torch.float32, device=dev)
    dP1, dP2, dV = torch.empty_like(P1), torch.empty_like(P2), torch.empty_like(V)
    dlam = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty((rb.relation_bwd_workspace_bytes(prob) + 3) // 4, dtype=torch.float32, device=dev)
    fws = rb.fwd_workspace(prob, dev)  # None unless the head width needs padded copies (d_h = 60)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    launches = [0]

    def step(events=None):
        if events:
            events[0].record(stream)
        rb.relation_fwd_ws(prob, P1, P2, V, Y, L, fws, stream)
        launches[0] += rb.relation_last_launch_count()
        if events:
            events[1].record(stream)
        args_b = (prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlam, ws, stream)
        rb.relation_bwd_prepare(*args_b)
        launches[0] += rb.relation_last_launch_count()
        if events:
            events[2].record(stream)
        rb.relation_bwd_main(*args_b)
        launches[0] += rb.relation_last_launch_count()
        if events:
            events[3].record(stream)
        rb.relation_bwd_finish(*args_b)
        launches[0] += rb.relation_last_launch_count()
        if events:
            events[4].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if rb.relation_check_device_status() != 0:
        raise RuntimeError("device-side wait expired during warm-up")

    ev_sets = [[ev() for _ in range(5)] for _ in range(args.steps)]
    launches[0] = 0
    rrep.barrier(ranks)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for k in range(args.steps):
            flush()  # evict L2 between timed steps (outside the events)
            step(ev_sets[k])
        torch.cuda.synchronize()
    rrep.barrier(ranks)
    if rb.relation_check_device_status() != 0:
        raise RuntimeError("device-side wait expired during the timed region")
    timed_launches = launches[0]

    t_step = [e[0].elapsed_time(e[4]) for e in ev_sets]
    t_fwd = [e[0].elapsed_time(e[1]) for e in ev_sets]
    t_prep = [e[1].elapsed_time(e[2]) for e in ev_sets]
    t_main = [e[2].elapsed_time(e[3]) for e in ev_sets]
    t_fin = [e[3].elapsed_time(e[4]) for e in ev_sets]
    total_ms = rrep.max_over_ranks(ranks, sum(t_step), dev)
    ms_per_step = total_ms / args.steps
    f_fwd, f_bwd = flops(w, 4), flops(w, 8)
    value = rrep.job_rate(ranks, (f_fwd + f_bwd) * args.steps, total_ms * 1e-3) / 1e12
    executed = rrep.job_rate(ranks, flops(w, 14) * args.steps, total_ms * 1e-3) / 1e12

    # e2e: the same step through the C ABI's host-memory entry point (relation_step_host) with
    # pinned host buffers: every step copies P1, P2, V, dY in and Y, dP1, dP2, dV, dlambda out,
    # in batch slices whose copies overlap the kernels, all inside the timed region.
    e2e = None
    if not args.no_e2e:
        h_in = {k: v.pin_memory() for k, v in x_cpu.items()}
        h_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in (("Y", Y), ("dP1", dP1),
                                                                                     ("dP2", dP2), ("dV", dV))}
        h_lam = torch.empty(1, dtype=torch.float32).pin_memory()
        chunks = args.e2e_chunks if args.e2e_chunks >= 1 and w.B % args.e2e_chunks == 0 else 1
        hbuf = torch.empty((rb.relation_step_host_device_bytes(prob, chunks) + 3) // 4, dtype=torch.float32,
                           device=dev)

        def e2e_step():
            rb.relation_step_host(prob, h_in["P1"], h_in["P2"], h_in["V"], h_in["dY"], h_out["Y"], None, h_out["dP1"],
                                  h_out["dP2"], h_out["dV"], h_lam, chunks, hbuf, stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = 0.0
        for _ in range(args.steps):
            flush()
            a, b = ev(), ev()
            a.record(stream)
            e2e_step()
            b.record(stream)
            b.synchronize()
            e_ms += a.elapsed_time(b)
        e_ms = rrep.max_over_ranks(ranks, e_ms, dev)
        h2d = sum(v.numel() * v.element_size() for v in h_in.values())
        d2h = sum(v.numel() * v.element_size() for v in h_out.values()) + 4
        e2e = {"value": rrep.job_rate(ranks, (f_fwd + f_bwd) * args.steps, e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.steps,
               "path": f"relation_step_host, {chunks} batch slice(s), pinned host buffers"}

    if rank != 0:
        rrep.finish(ranks)
        return 0

    peak_burst, peak_sust, peak_src = load_peaks()
    mean_fwd, mean_main = statistics.mean(t_fwd), statistics.mean(t_main)
    # Kernels by head width: 48, 60 and 64 run the 64-wide tensor-core kernels, 80 and
    # 128 the 128-wide ones (zero-padded tiles); 60 reads zero-padded copies of its
    # operands (made by one extra launch in the forward and one in the backward).
    tile = 64 if w.d <= 64 else 128
    srcs_common = ["ptx_sm100.cuh", "common.cuh", "tile_copy.cuh", "prologue_tiles.cuh", "kernels.h"]
    fwd_k = f"relation_fwd_tc_kernel<{tile}, false>"
    fwd_src = ["fwd_tc.cu"] + srcs_common
    if tile == 64:
        bwd_k, bwd_src = "relation_bwd_tc64_kernel<0>", ["bwd_tc64.cu", "bwd_elementwise.cuh"] + srcs_common
    else:
        bwd_k, bwd_src = "relation_bwd_tc_kernel<128>", ["bwd_tc.cu", "bwd_elementwise.cuh"] + srcs_common
    if mean_main >= mean_fwd:
        dom, srcs, dom_ms, dom_flops = bwd_k, bwd_src, mean_main, f_bwd
    else:
        dom, srcs, dom_ms, dom_flops = fwd_k, fwd_src, mean_fwd, f_fwd
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    line = {
        "metric": "Relation fwd+bwd TFLOP/s (bf16, causal) and % of GB300 dense bf16 peak",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded Gaussian inputs, resident in HBM)",
        "config": relation_config(w, world),
        "frac_of_peak": {"value": value / peak_burst, "peak_tflops": peak_burst, "source": peak_src,
                         "sustained_frac": value / peak_sust},
        "executed_tflops": executed,
        "breakdown_ms": {"fwd": mean_fwd, "bwd_prepare": statistics.mean(t_prep), "bwd_main": mean_main,
                         "bwd_finish": statistics.mean(t_fin)},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": achieved / peak_burst, "peak_source": f"{peak_src} bf16 burst",
                     "traffic": recorded_traffic(dom, kernel_source_hash(srcs), w.name)},
        "gpu_launches": timed_launches,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and world == 1:
        try:
            line["cpu_baseline"] = cpu_baseline(w)
        except Exception as exc:  # the baseline is context only; keep the GPU line
            line["cpu_baseline"] = {"value": None, "unit": "TFLOP/s", "cores": None, "kind": "oracle",
                                    "sample": f"failed: {exc}"}
    print(json.dumps(line))
    rrep.finish(ranks)
    return 0


if __name__ == "__main__":
    sys.exit(main())
