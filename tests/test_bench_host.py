"""Host-side arithmetic of bench.py (no GPU): the visible-pair count and flop model the throughput is
computed from, the Linear Relation byte model, and the DRAM-traffic record that the roofline reports only
for the workload and kernel sources it was captured on."""
import json
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from relation_token_mixing_gb300 import inputs as rin  # noqa: E402


@pytest.mark.parametrize("T,causal", [(1, True), (7, True), (128, True), (7, False), (129, False)])
def test_visible_pairs_by_brute_force(T, causal):
    expect = sum(1 for i in range(T) for j in range(T) if (j <= i or not causal))
    assert bench.pairs(T, causal) == expect


def test_flops_count_every_head_and_pair():
    w = rin.Workload("x", 2, 3, 10, 64, torch.bfloat16, 1.0, 0.5, True, 1.0)
    assert bench.flops(w, 12) == 2 * 3 * (10 * 11 // 2) * 12 * 64


def test_linear_bytes_per_head_token():
    # forward: P1, P2, I~, Y in bf16 (2 bytes) and G in fp32: 4*2d + 4d = 12d
    # backward: P1, P2, I~, dY, dP1, dP2, dI~ in bf16 and G, dG in fp32: 7*2d + 2*4d = 22d
    for d in (48, 60, 64):
        assert bench.linear_bytes_per_head_token(d) == 12 * d + 22 * d


def test_recorded_traffic_is_keyed_by_workload_and_source():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    for key, e in rec.items():
        if key.startswith("_"):
            continue
        kernel = key.split(" @ ")[0]
        if " @ " in key:
            assert key.split(" @ ")[1] == e["workload"]
        assert bench.recorded_traffic(kernel, e["source_hash"], e["workload"]) == e["bytes_per_launch"]
        assert bench.recorded_traffic(kernel, e["source_hash"], e["workload"] + "_other") is None
        assert bench.recorded_traffic(kernel, "0" * 16, e["workload"]) is None
    assert bench.recorded_traffic("no_such_kernel", "0" * 16, "mhr_fwd_bwd_T4096") is None


@pytest.mark.parametrize("B,H,per_head_s,expect_heads,expect_shape", [
    (4, 16, 0.125, 64, (4, 16)),     # first pass 0.5 s: grows to the whole workload (8 s)
    (64, 16, 0.125, 96, (6, 16)),    # grows by 24 (12 s / 0.5 s), six whole batches
    (4, 16, 10.0, 4, (1, 4)),        # first pass 40 s: no second pass
    (1, 3, 0.1, 3, (1, 3)),          # fewer heads than threads: one pass over all of them
])
def test_cpu_baseline_sample_grows_toward_its_target(monkeypatch, B, H, per_head_s, expect_heads, expect_shape):
    """The oracle pass is sized in whole multiples of the oracle's thread count toward the target
    time, at most the whole workload; the reported value is from the last pass.  The oracle and
    the clock are stand-ins here, so only the sizing rule runs."""
    import oracle

    now = [0.0]
    passes = []

    def fake_fwd(P1, *a, **k):
        heads = P1.shape[0] * P1.shape[1]
        passes.append((P1.shape[0], P1.shape[1]))
        now[0] += per_head_s * heads

    monkeypatch.setattr(oracle, "threads", lambda: 4)
    monkeypatch.setattr(oracle, "fwd", fake_fwd)
    monkeypatch.setattr(oracle, "bwd", lambda *a, **k: None)
    monkeypatch.setattr(bench.time, "perf_counter", lambda: now[0])
    w = rin.Workload("x", B, H, 8, 64, torch.bfloat16, 1.0, 0.5, True, 1.0, backward=True)
    out = bench.cpu_baseline(w, target_s=12.0)
    assert passes[-1] == expect_shape and passes[-1][0] * passes[-1][1] == expect_heads
    assert len(passes) == (2 if expect_heads > min(4, B * H) else 1)
    dt = per_head_s * expect_heads
    sample = rin.Workload("x", *expect_shape, 8, 64, torch.bfloat16, 1.0, 0.5, True, 1.0)
    assert out["value"] == pytest.approx(bench.flops(sample, 12) / dt / 1e12)
    assert out["cores"] == 4 and out["kind"] == "oracle"
    assert ("the whole workload" in out["sample"]) == (expect_heads == B * H)


@pytest.mark.parametrize("arm", ["relation", "decode", "prologue", "linear"])
def test_reference_lines_carry_the_workload_config(capsys, arm):
    """`--impl reference` times the float64 oracle on a bounded sample, but its line names the
    same workload `config` as the GPU arm's (the sample is described in cpu_baseline.sample);
    value, cpu_baseline and e2e agree.  Small shapes and the real oracle."""
    import argparse

    args = argparse.Namespace(gpus=1, steps=1, warmup=0)
    if arm == "linear":
        w = rin.LinearWorkload("small_linear", 1, 2, 64, 60, backward=True)
        bench.run_linear_reference(args, w)
        expect = bench.linear_config(w, 1)
    else:
        w = rin.Workload("small", 2, 4, 64, 64, torch.bfloat16, 1.0, 0.5, True, 1.0, backward=True)
        fn, expect = {"relation": (bench.run_reference, bench.relation_config(w, 1)),
                      "decode": (bench.run_decode_reference, bench.decode_config(w, w.T - 1)),
                      "prologue": (bench.run_prologue_reference, bench.prologue_config(w))}[arm]
        fn(args, w)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"] == expect
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
