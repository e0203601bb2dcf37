"""Host-side logic of the benchmark on CPU: the peak figures the roofline divides by,
the rule that reports the measured DRAM traffic only for the kernel sources it was
measured on, the percentile helper, the fixed oracle sample, and the reference arm's
JSON line (it times the CPU oracle, so it runs here)."""
import hashlib
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import bench
from structured_sparse_dnn_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_tensor_peak_effective():
    pk = {"bf16_tflops": 1000.0, "bf16_tflops_sustained": 900.0}
    assert bench.tensor_peak_effective("bf16", pk) == 1000.0
    assert bench.tensor_peak_effective("f16", pk) == 1000.0
    assert bench.tensor_peak_effective("e4m3", pk) == 2000.0
    assert bench.tensor_peak_effective("e4m3", pk, sustained=True) == 1800.0


def test_peaks_fall_back_without_the_measured_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.peaks()
    assert pk["source"] == "fallback"
    assert pk["bf16_tflops"] > 0 and pk["hbm_gbs"] > 0


def _key(root):
    h = hashlib.sha256()
    for name in ("gemm.cu", "ptx.cuh", "common.cuh"):
        with open(os.path.join(root, "structured_sparse_dnn_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def test_measured_traffic_only_for_the_measured_sources(monkeypatch, tmp_path):
    """The committed figure is reported while the three kernel sources hash to the
    recorded key, and withheld (None) as soon as one of them changes."""
    csrc = tmp_path / "structured_sparse_dnn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("gemm.cu", "ptx.cuh", "common.cuh"):
        shutil.copy(os.path.join(ROOT, "structured_sparse_dnn_gb300", "csrc", name), csrc / name)
    (tmp_path / "profiles").mkdir()
    tab = {"llm_ffn_e4m3": {"kernel_src_sha256_16": _key(str(tmp_path)), "dram_bytes_per_launch": 12345}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(tab))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("llm_ffn_e4m3") == 12345
    assert bench.measured_traffic("llm_ffn_bf16") is None
    with open(csrc / "ptx.cuh", "a") as f:
        f.write("\n// changed\n")
    assert bench.measured_traffic("llm_ffn_e4m3") is None


def test_committed_traffic_record_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        tab = json.load(f)
    ent = tab["llm_ffn_e4m3"]
    assert ent["dram_bytes_per_launch"] == ent["dram_read_bytes"] + ent["dram_write_bytes"]
    assert len(ent["kernel_src_sha256_16"]) == 16


def test_pct_interpolates():
    xs = [4.0, 1.0, 3.0, 2.0]
    assert bench.pct(xs, 0) == 1.0
    assert bench.pct(xs, 100) == 4.0
    assert bench.pct(xs, 50) == pytest.approx(2.5)


def test_cpu_sample_is_fixed_and_in_range():
    wl = I.WORKLOADS["llm_ffn_e4m3"]
    a, b = bench.cpu_sample(wl), bench.cpu_sample(wl)
    assert np.array_equal(a, b)
    assert len(np.unique(a)) == len(a) == bench.CPU_SAMPLE_ROWS
    assert a.min() >= 0 and a.max() < wl.M


def test_reference_arm_line():
    """`bench.py --impl reference` prints one JSON line with the contract's keys, timing
    the oracle on the fixed sample (no GPU needed)."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["steps"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"]["sample_rows"] == bench.CPU_SAMPLE_ROWS
