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


def test_traffic_record_only_for_its_kernel_and_workload(tmp_path):
    wl = bench.headline_workload()
    rec = tmp_path / "traffic.txt"
    rec.write_text(f"# header\nworkload: {wl.name}\ndecode kernel sha256: {bench.decode_kernel_sha()}\n"
                   f"dram bytes per launch (read+write): 71596672\n")
    assert bench.traffic_from_profiles(wl, str(rec)) == 71596672.0
    assert bench.traffic_from_profiles(syn.dense14b(131072, "q8_0", "q4_0"), str(rec)) is None
    # a record taken on other kernel sources is not used
    rec.write_text(f"workload: {wl.name}\ndecode kernel sha256: {'0' * 64}\n"
                   f"dram bytes per launch (read+write): 71596672\n")
    assert bench.traffic_from_profiles(wl, str(rec)) is None
    # the committed record, when it matches the current kernel, is close to the algorithmic bytes
    v = bench.traffic_from_profiles(wl)
    assert v is None or 1.0 <= v / (65537 * 1088) <= 1.05


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_compact_cell_table():
    sweep = [
        {"workload": "hybrid-10L-q8_0-q8_0-ctx65536", "kv": "q8_0/q8_0", "ctx": 65536, "steps_per_s": 4675.0,
         "kv_gbs": 3334.2, "pct_hbm_peak": 49.97},
        {"workload": "hybrid-10L-q8_0-q8_0-ctx4096", "kv": "q8_0/q8_0", "ctx": 4096, "steps_per_s": 99999.0,
         "kv_gbs": 4000.0, "pct_hbm_peak": 60.0, "rotating": {"pct_hbm_peak": 30.0}},
        {"workload": "multi-session-48L", "kv": "q8_0/q4_0", "ctx": [8192, 9000], "steps_per_s": 95.5,
         "kv_gbs": 4358.0, "pct_hbm_peak": 65.3},
        {"workload": "hybrid-10L-window4096-f16+q8_0-q8_0-ctx65536", "kv": "f16 window + q8_0/q8_0 tail",
         "ctx": 65536, "steps_per_s": 3111.0, "kv_gbs": 2341.0, "pct_hbm_peak": 35.1},
        {"workload": "verify-nq4-dense-48L-q8_0-q4_0-ctx131072", "kv": "q8_0/q4_0", "ctx": 131072, "n_q": 4,
         "steps_per_s": 172.7, "kv_gbs": 1808.0, "pct_hbm_peak": 27.1},
        {"workload": "dense-48L-q5_1-q4_0-ctx131072", "kv": "q5_1/q4_0", "ctx": 131072, "steps_per_s": 400.0,
         "kv_gbs": 3000.0, "pct_hbm_peak": 44.0},
    ]
    cells = bench.compact_cells(sweep, {"us_per_chunk": 32.5, "gbs": 1239.3})
    assert cells[0] == ["hyb q8/q8 64K", 4675.0, 3334, 50.0]
    assert cells[1] == ["hyb q8/q8 4K", 99999.0, 4000, 60.0, 30.0]
    assert cells[2][0] == "ms16 q8/q4 mix"
    assert cells[3][0] == "hyb w+q8/q8 64K"
    assert cells[4][0] == "vfy4-d48 q8/q4 128K"
    assert cells[5][0] == "d48 q51/q4 128K"
    assert cells[-1] == ["chunk4096 q8/q4", 32.5, 1239, None]
    assert len(json.dumps(cells)) < 600


def test_stamp_spans():
    import torch
    # 2 graphs x 3 layers, 2 CTAs per launch: (start, exit) in ns
    se = [[[0, 10_000], [1_000, 12_000]], [[9_000, 20_000], [9_500, 21_000]],
          [[19_000, 30_000], [20_000, 29_000]],
          [[100_000, 110_000], [100_000, 111_000]], [[108_000, 120_000], [109_000, 119_000]],
          [[118_000, 131_000], [118_000, 130_000]]]
    st = torch.zeros((6, 2, 2), dtype=torch.int64)
    for i, launch in enumerate(se):
        for c, (a, e) in enumerate(launch):
            st[i, c, 0], st[i, c, 1] = a, e
    spans, gaps = bench.stamp_spans(st.flatten(), 6, 3, 2)
    assert spans == [12.0, 12.0, 11.0, 11.0, 12.0, 13.0]
    assert gaps == [9.0, 9.0, 9.0, 11.0]
