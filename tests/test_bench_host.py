"""Host-side logic of bench.py that needs no GPU: the peak denominators
(measured file or the stated fallback) and the algorithmic byte counts of the
HBM-bound kernels on the 16K-token Qwen3-30B-A3B-shaped prefill."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_peaks_measured_file_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback"
    assert (p["hbm_gbs"], p["bf16_tflops"]) == (6800.0, 1900.0)
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 7100.5, "bf16_tflops": 2010.0, "bf16_tflops_sustained": 1750.0}))
    p = bench.load_peaks()
    assert p["source"] == "measured"
    assert (p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"]) == (7100.5, 2010.0, 1750.0)
    # a file without the two denominators falls back
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"clocks": 2070}))
    assert bench.load_peaks()["source"] == "fallback"


def test_algorithmic_bytes_of_the_prefill_workload():
    T, H, E, k, I = 16384, 2048, 128, 8, 768
    M = T * k
    b = bench.algorithmic_bytes(T, H, E, k, I)
    # route + quant: read x (bf16) and the fp32 logits; write the e4m3 rows,
    # their e8m0 scales and four int32/fp32 words per expanded row
    x, logits = T * H * 2, T * E * 4
    xq, xs, idx = M * H * 1, M * (H // 32), M * 16
    assert b["route"] == x + logits + xq + xs + idx
    assert round(b["route"] / 1e6, 1) == 354.4
    # finalize: read the bf16 y rows, write the bf16 output, read weight + index
    assert b["finalize"] == M * H * 2 + T * H * 2 + M * 8
    assert round(b["finalize"] / 1e6) == 605
    # load-time weight quant: bf16 in, e4m3 + e8m0 out, w13 [E, 2I, H] and w2 [E, H, I]
    n_w = E * 2 * I * H + E * H * I
    assert b["weight_quant"] == pytest.approx(n_w * (2 + 1 + 1 / 32))
    assert round(b["weight_quant"] / 1e6) == 1831
