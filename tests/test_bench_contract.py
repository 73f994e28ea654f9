"""bench.py's JSON line (the reference arm runs the oracle, so it needs no GPU): one line
with the contract's keys, and the ours-arm helpers that build the line."""
import json
import os
import subprocess
import sys

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert BASE_KEYS <= set(d)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["steps"] == 1
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith(bench.HEADLINE)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_every_workload_has_a_config_description():
    for name, wl in W.WORKLOADS.items():
        c = bench.workload_config(wl)
        assert c["workload"].startswith(name) and c["l2"] and c["parallelism"] == "replicas"


def test_algorithmic_work_of_the_prefills():
    """4 D Hq B flops per visible pair; Q + K + V read once, out + lse written once."""
    wl = W.WORKLOADS["qwen3_0.6b_prefill"]
    flops, bytes_, pairs = bench.prefill_work(wl)
    assert pairs == 512 * 513 // 2
    assert flops == 4 * 64 * 16 * 8 * pairs
    assert bytes_ == 8 * 512 * (16 + 8 + 8) * 64 * 2 + 8 * 512 * 16 * 64 * 2 + 8 * 512 * 16 * 4
    # the headline: the Gemma-4 global layer, B1 S8192 Hq16 Hkv2 D512 causal
    wl = W.WORKLOADS[bench.HEADLINE]
    assert (wl.B, wl.S, wl.L, wl.Hq, wl.Hkv, wl.D, wl.causal) == (1, 8192, 8192, 16, 2, 512, True)
    flops, bytes_, pairs = bench.prefill_work(wl)
    assert pairs == 8192 * 8193 // 2
    assert flops == 4 * 512 * 16 * pairs  # 1.0996 TFLOP
    assert bytes_ == 8192 * 16 * 512 * 2 * 2 + 2 * 8192 * 2 * 512 * 2 + 8192 * 16 * 4
    # sliding window: 1024 keys per row once the window is full
    wl = W.WORKLOADS["gemma4_sliding_prefill"]
    assert bench.visible_pairs(8192, 8192, True, 1024) == 1024 * 1025 // 2 + (8192 - 1024) * 1024


def test_decode_work_counts_each_kv_element_once_per_kv_head():
    wl = W.WORKLOADS[bench.COMPANION]
    flops, bytes_, keys = bench.decode_work(wl, [32768] * 8)
    assert keys == 8 * 32768
    assert bytes_ == keys * 2 * 512 * 2 * 2 + 8 * 16 * 512 * 2 * 2 + 8 * 16 * 4
    assert flops == 4.0 * 512 * 16 * keys


def test_oracle_sample_shares_are_exact():
    """The CPU baseline's row sample carries exactly the visible pairs of its rows."""
    wl = W.WORKLOADS["gemma4_sliding_prefill"]
    rows = W.sample_rows(wl.B * wl.S, wl.S, extra=(1023, 1024, 1025), n_random=16)
    per_row = bench.row_pairs(wl, rows)
    for r, n in zip(rows, per_row):
        i = r % wl.S
        assert n == min(i + 1, 1024)


import pytest  # noqa: E402


@pytest.mark.gpu
def test_ours_arm_prints_one_contract_line(cuda_device):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3",
                        "--warmup", "3", "--no-extra", "--no-cpu"], capture_output=True,
                       text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert BASE_KEYS <= set(d) and d["n_gpus"] == 1 and d["steps"] == 3
    assert d["value"] > 0 and d["gpu_launches"] == 3
    assert d["config"]["workload"].startswith(bench.HEADLINE)
    dec = d["decode"]
    assert dec["workload"].startswith(bench.COMPANION) and dec["unit"] == "GB/s"
    assert dec["value"] > 0 and dec["roofline"]["bound"] == "hbm"
    assert dec["e2e"]["h2d_bytes_per_step"] > 0 and dec["e2e"]["d2h_bytes_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor") and 0 < rf["frac"] < 2 and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
