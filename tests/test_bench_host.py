"""Host-side arithmetic of bench.py, on CPU: algorithmic KV bytes (bits per value of each
block type, the headline's bytes per decode launch), the DRAM-traffic record that is used
only for the decode kernel it was measured on, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

import bench
import oracle
import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bits_per_value_match_block_sizes():
    # bytes per value = block bytes / 32: the oracle's block sizes where it carries them (the
    # tier ladder's types), else the block layouts written out (codes + fifth bits + scales)
    layout = {"f16": 32 * 2, "q8_0": 32 + 2, "q4_0": 16 + 2, "q4_1": 16 + 2 + 2, "q5_0": 16 + 4 + 2,
              "q5_1": 16 + 4 + 2 + 2}
    for t, bpv in bench.BPV.items():
        assert bpv == pytest.approx(oracle.BLOCK_BYTES.get(t, layout[t]) / 32), t
        assert oracle.BLOCK_BYTES.get(t, layout[t]) == layout[t], t


def test_headline_bytes_per_launch():
    wl = bench.headline_workload()
    assert (wl.layers, wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim) == (10, 1, 16, 2, 256)
    # 2 KV heads x 256 values x (34 + 34) bytes per 32 values = 1088 B per position and layer
    assert bench.row_bytes(wl) == pytest.approx(1088.0)
    assert bench.step_kv_bytes(wl, [65537]) / wl.layers == pytest.approx(65537 * 1088)


def test_traffic_record_only_for_its_kernel_and_workload():
    wl = bench.headline_workload()
    v = bench.traffic_from_profiles(wl)
    assert v is not None and 1.0 <= v / (65537 * 1088) <= 1.05  # ncu bytes ~ algorithmic bytes
    assert bench.traffic_from_profiles(syn.dense14b(131072, "q8_0", "q4_0")) is None


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
