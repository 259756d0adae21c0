"""bench.py's algorithmic counts and whole-step roofline fractions, on the
CPU (no GPU run): closed forms for a tiny shape and the binding choice."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from transformer_encoder_layer_gb300.inputs import SHAPES, tiny_shape  # noqa: E402


def test_visible_keys_closed_form():
    # L = 4, valid_len 2: rows see 1, 2, 2, 2 keys; valid_len 4: 1, 2, 3, 4
    assert bench.sum_visible_keys(np.array([2, 4]), 4) == 7 + 10


def test_counts_of_a_tiny_shape():
    s = tiny_shape(dtype="f16", batch=2, seq_len=4, d_model=8, n_heads=2, d_ff=16, n_layers=3)
    c = bench.algorithmic_counts(s, np.array([2, 4]))
    T, d, dff = 8, 8, 16
    per_layer = 2 * T * 3 * d * d + 4 * d * 17 + 2 * T * d * d + 2 * 2 * T * d * dff
    assert c["flops"] == pytest.approx(3 * per_layer)
    assert c["sfu_ops"] == 3 * (17 * 2 + T * dff)


def test_step_fractions_pick_the_path_roofline():
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 5000.0, "sm_max_mhz": 2000.0}
    counts = {"flops": 1e12, "hbm_bytes": 1e9, "sfu_ops": 1e9}
    f = bench.step_fractions(counts, 10.0, peaks, 100, "f16")   # 10 ms
    assert f["tensor"] == pytest.approx(1e14 / 1e15)
    assert f["hbm"] == pytest.approx(1e11 / 5e12)
    assert f["sfu"] == pytest.approx(1e11 / (100 * bench.SFU_PER_SM_CLK * 2e9))
    assert "fp32_alu" not in f        # a 16-bit path runs on the tensor cores
    assert f["binding"] == "tensor"
    g = bench.step_fractions(counts, 10.0, peaks, 100, "f32")
    assert "tensor" not in g          # fp32 I/O runs on the CUDA cores
    assert g["fp32_alu"] == pytest.approx(1e14 / (100 * 256 * 2e9))
    assert g["binding"] == "fp32_alu"


def test_step_fractions_of_the_bench_workload_are_plausible():
    s = SHAPES["short_d128_L64_B4096"]
    vl = np.full(s.batch, 48)
    c = bench.algorithmic_counts(s, vl)
    f = bench.step_fractions(c, 1.93, bench.load_peaks(), 152, s.dtype)
    assert 0.05 < f["tensor"] < 0.5 and f["hbm"] < f["tensor"]


def test_kernel_roofline_uses_the_bounding_unit():
    s = SHAPES["short_d128_L64_B4096"]
    c = bench.algorithmic_counts(s, np.full(s.batch, 48))
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0, "sm_max_mhz": 2000.0, "source": "measured"}
    r = bench.kernel_roofline({"megakernel": (20.0, 10)}, s, c, peaks, 152, 20.0)
    assert r["kernel"] == "megakernel" and r["bound"] == "tensor" and r["peak"] == 2000.0
    assert r["achieved"] == pytest.approx(c["flops"] / 2e-3 / 1e12)
    assert r["share_of_step"] == pytest.approx(1.0)
    t = SHAPES["batch1_d256_L512"]
    ct = bench.algorithmic_counts(t, np.full(1, 400))
    r = bench.kernel_roofline({"dag": (1.0, 4)}, t, ct, peaks, 152, 1.0)
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(152 * 256 * 2e9 / 1e12)


def test_percentiles():
    assert bench.percentile([1, 2, 3, 4, 5], 50) == 3
    assert bench.percentile([1.0] * 7, 90) == 1.0
