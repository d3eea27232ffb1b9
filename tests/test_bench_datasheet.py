"""bench.py's optional datasheet fractions (host logic, no GPU)."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_no_file_gives_no_datasheet_entry():
    assert bench.datasheet_fracs(None, 1500.0, {"rope": 5000.0}) is None


def test_fractions_of_the_supplied_peaks(tmp_path):
    p = tmp_path / "sheet.json"
    p.write_text(json.dumps({"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}))
    d = bench.datasheet_fracs(str(p), 1500.0, {"rope": 6000.0, "normalize_patchify": 4000.0})
    assert d["file"] == "sheet.json"
    assert d["frac"] == pytest.approx(0.75)
    assert d["hbm_fracs"] == {"rope": pytest.approx(0.75), "normalize_patchify": pytest.approx(0.5)}


def test_either_key_may_be_absent(tmp_path):
    p = tmp_path / "tensor_only.json"
    p.write_text(json.dumps({"bf16_tflops": 2250.0}))
    d = bench.datasheet_fracs(str(p), 1125.0, {"rope": 1.0})
    assert d["frac"] == pytest.approx(0.5) and "hbm_fracs" not in d
