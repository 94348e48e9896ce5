"""The key-stationary backward's CTA order (grouped_tile_order in csrc/common.cuh), checked on the
host: a small program compiled with nvcc from the same header walks every linear block index and
asserts that each (head, key tile) pair is visited exactly once, group by group, tiles in
non-decreasing order inside a group (heaviest causal tiles first), including a ragged last group."""
import os
import subprocess

import pytest

from relation_token_mixing_gb300 import build as rbuild

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "_build", "tile_order_check")


@pytest.fixture(scope="module")
def checker():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    src = os.path.join(HERE, "tile_order_check.cu")
    cmd = [rbuild._nvcc(), *rbuild.ARCH, "-std=c++17", "-O2", "-I", rbuild.CSRC, src, "-o", OUT]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return OUT


def test_small_sizes_every_group(checker):
    r = subprocess.run([checker], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout
    assert r.stdout.strip() == "ok " + str(sum(bh * 12 for bh in range(1, 41)))


@pytest.mark.parametrize("BH,n_tiles,groups", [
    (64, 32, [1, 7, 30, 63, 64]),      # B4 H16, T 4096 (128-key tiles)
    (32, 128, [1, 3, 5, 32]),          # B1 H32, T 16384, d 128
    (128, 16, [1, 11, 17, 128]),       # B16 H8, T 2048
    (37, 33, [4, 5, 36]),              # ragged in both
])
def test_measured_shapes(checker, BH, n_tiles, groups):
    args = [str(v) for g in groups for v in (BH, n_tiles, g)]
    r = subprocess.run([checker, *args], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout
    assert r.stdout.strip() == f"ok {len(groups)}"
