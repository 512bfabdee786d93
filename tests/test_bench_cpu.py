"""The bench's output contract on CPU: the reference arm (the oracle, timed on the host
cores) prints one JSON line with the keys the GPU arm prints, and the helpers the GPU
arm reports through (algorithmic work, the source hash of a profiled kernel) behave.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "1", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "samples/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 1
    assert d["vs_baseline"] is None and d["scaling"] == "weak"
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_algorithmic_gram_flops_count_only_the_block_lower_part():
    # F = n * S^2 * (1 - 1/s): the s(s-1)/2 strictly lower b x b blocks, 2n flops each entry
    n, b, s = 2000, 256, 32
    S = b * s
    work = bench.alg_work(n, S, s, b, 400000)
    blocks = s * (s - 1) // 2
    assert work["gram"]["flops"] == pytest.approx(blocks * b * b * 2 * n, rel=1e-12)


def test_source_hash_tracks_the_kernel_sources():
    h = bench.source_hash("gram_recur_far")
    assert len(h) == 16 and int(h, 16) >= 0
    assert h == bench.source_hash("gram_recur_far")  # deterministic


def test_tensor_peak_is_burst_unless_the_clock_record_says_otherwise():
    pk = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.tensor_peak(pk, full)[0] == 1900.0
    capped = dict(full, reasons=["sw_power_cap"])
    peak, which = bench.tensor_peak(pk, capped)
    assert peak == 1700.0 and "sw_power_cap" in which
    slow = {"sm_mhz": 1460.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.tensor_peak(pk, slow)[0] == 1700.0
    unsampled = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
    assert bench.tensor_peak(pk, unsampled)[0] == 1900.0
