"""The benchmark's byte accounting and JSON contract, on the CPU.

The roofline's `achieved` divides algorithmic bytes by the measured time, so
the byte counts are checked here against totals worked out by hand from the
shapes: dsv3 (R=8, N=4096, H=7168 bf16, top-8 of 256) moves every token row
once (470 MB) plus every receive row once in dispatch, and the reverse in
combine; with the expected 173,495 receive rows (uniform routing:
c = R(1 - C(E - E/R, K)/C(E, K)) = 5.2947 destinations per token) that is
2.957 GB each way, 5.914 GB per step, plus about 16 MB of index metadata."""
import json
import math
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_expected_receive_rows_closed_form():
    R, N, E, K = 8, 4096, 256, 8
    El = E // R
    c = R * (1.0 - math.comb(E - El, K) / math.comb(E, K))
    assert abs(c - 5.2947) < 1e-4
    assert round(R * N * c) == 173495


def test_algorithmic_bytes_dsv3():
    R, N, K, E, H, T = 8, 4096, 8, 256, 7168, 173495
    ab = bench.algorithmic_bytes(R, N, K, E, H, T)
    x = R * N * H * 2                  # 469,762,048 B of token rows
    rows = T * H * 2                   # 2,487,224,320 B of receive rows
    assert abs((x + rows) / 1e9 - 2.957) < 1e-3
    send_row = R * N * R * 4
    assert ab["rows"] == x + rows + send_row
    assert ab["combine"] == rows + x + send_row
    meta = ab["layout"] + ab["offsets"]
    assert 15e6 < meta < 18e6          # "+~16 MB metadata"
    assert abs((ab["rows"] + ab["combine"]) / 1e9 - 5.914) < 0.003


def test_algorithmic_bytes_fp8_scales():
    """e4m3 rows move H bytes plus H/128 fp32 scales per row, read once and written
    once per destination."""
    R, N, K, E, H, T = 8, 8192, 8, 256, 7168, 347210
    ab = bench.algorithmic_bytes(R, N, K, E, H, T, elt=1, scales_per_row=H // 128)
    assert ab["rows"] == R * N * H + T * H + (R * N + T) * 56 * 4 + R * N * R * 4


def test_reference_arm_prints_the_contract_line():
    """--impl reference (the CPU oracle) prints one JSON line with the contract's keys;
    run on a tiny workload so it takes seconds."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and "workload" in d["config"]
