"""Pins the byte accounting used for every achieved-GB/s figure against the
table of the analytic decode gap model printed on page "PDL and megakernel"
(fixture tests/golden/decode_gaps.json, with its citation)."""
import json
import os

import pytest

from pdl_persistent_megakernel_gb300 import bytes_model
from pdl_persistent_megakernel_gb300.synth import CONFIGS

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "decode_gaps.json")))
BW = GOLD["assumptions"]["bandwidth_bytes_per_s"]
GAPS = (0.5, 1.0, 2.0, 3.0)


@pytest.mark.parametrize("row", GOLD["rows"], ids=lambda r: f"{r['model']}-b{r['batch']}")
def test_gap_model_table(row):
    ks = bytes_model.gap_model_kernels(**GOLD["models"][row["model"]],
                                       batch=row["batch"], context=row["context"])
    g = bytes_model.gap_model(ks, BW, GAPS)
    assert g["kernels"] == row["kernels"]
    assert round(g["data_us"]) == row["data_us"]
    eager = max(g["kernels"] * 5.0, g["data_us"] + g["kernels"] * GAPS[0])
    assert round(eager) == row["eager_us"]
    assert [round(t) for t in g["with_gap_us"]] == row["gap_us"]
    assert [round(100 * s) for s in g["gap_share"]] == row["gap_pct"]


def test_gap_model_small_kernels_and_exercise():
    s = GOLD["small_kernels"]
    ks = bytes_model.gap_model_kernels(**GOLD["models"][s["model"]],
                                       batch=s["batch"], context=s["context"])
    g = bytes_model.gap_model(ks, BW, GAPS)
    assert g["under_1us"] == s["under_1us"] and g["kernels"] == s["kernels"]
    assert round(g["mean_us"], 2) == s["mean_us"]
    ex = GOLD["exercise_fusion"]
    n_after = 28 * 6 + 3
    assert n_after == ex["kernels_after"]
    assert round(g["data_us"] + n_after * ex["gap_g_us"]) == ex["step_after_us"]
    assert round(g["data_us"] + n_after * 1.0) == ex["step_after_g1_us"]


def test_algorithmic_bytes_of_the_headline_configs():
    # per-config totals quoted in the measurement plan (rounded to 0.1 MB)
    q8 = bytes_model.algorithmic_bytes(CONFIGS["q8_layer_m16_ctx8192_fp8"])
    assert abs(q8["weights"] - 192.99e6) < 0.05e6
    assert abs(q8["kv_read"] - 67.11e6) < 0.01e6
    assert abs(q8["total"] - 260.6e6) < 0.2e6
    q06 = bytes_model.algorithmic_bytes(CONFIGS["q06_layer_b1_ctx1024"])
    assert abs(q06["weights"] - 31.46e6) < 0.01e6
    assert abs(q06["total"] - 35.66e6) < 0.01e6
    full = bytes_model.algorithmic_bytes(CONFIGS["q8_step_b1_ctx8192"])
    assert abs(full["total"] - 16.34e9) < 0.01e9
