"""The planner-calibration tool's host side: rank correlation and regret bookkeeping."""
import json

import pytest

from transformer_mlp_gemms_gb300 import build as kbuild
from transformer_mlp_gemms_gb300 import calibrate
from transformer_mlp_gemms_gb300 import kt_mlp


def test_spearman_matches_scipy_with_ties():
    stats = pytest.importorskip("scipy.stats")
    a = [3.0, 1.0, 4.0, 1.0, 5.0, 9.0, 2.0, 6.0]
    b = [2.7, 1.8, 2.8, 1.8, 4.5, 9.0, 0.5, 7.1]
    assert calibrate._spearman(a, b) == pytest.approx(stats.spearmanr(a, b).correlation, abs=1e-12)
    assert calibrate._spearman([1, 2, 3], [3, 2, 1]) == pytest.approx(-1.0)


def test_evaluate_reports_zero_regret_when_the_pick_is_the_fastest(tmp_path, capsys):
    kbuild.build()
    kt_mlp.load()
    # measurements that agree with the model's order exactly: the pick must be the fastest
    rows = []
    for gemm, val in calibrate._configs():
        calibrate._clear_env()
        import os
        os.environ["KT_FORCE_UP" if gemm == "up" else "KT_FORCE_DOWN"] = val
        try:
            g = kt_mlp.kt_mlp_plan_info(729, 1152, 4304, 1, 0, False, 152)[gemm]
        except kt_mlp.KtError:
            continue
        rows.append({"gemm": gemm, "force": val, "BM": g["BM"], "BN": g["BN"], "BK": g["BK"], "SK": g["split_k"],
                     "CL": g["cluster_sk"], "us_mean": g["est_us"]})
    calibrate._clear_env()
    (tmp_path / "calib_siglip.json").write_text(json.dumps(rows))
    total = calibrate.evaluate(["siglip"], str(tmp_path))
    out = capsys.readouterr().out
    assert "| siglip | up |" in out and "| siglip | down |" in out
    assert total == pytest.approx(0.0, abs=1e-9)
