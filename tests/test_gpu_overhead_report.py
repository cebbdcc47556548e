"""GPU test of the N3 model report (overhead_report.report) on one short
sequence: the measured legs, the Burst-Gap and counterfactual predictions,
the refit on tensor-core-gap probe points, and the traced per-tile spans
come out complete and consistent (the completion-coupled counterfactual
never predicts less than the Burst-Gap equation; spans and busy shares are
positive)."""
import math

import pytest

from attention_all_layout_gb300 import overhead_report as orep

pytestmark = pytest.mark.gpu


def test_report_at_one_sequence_length():
    res = orep.report(H=8, s_list=(1024,))
    assert res["R_GBps"] > 0
    for fit in ("mma_gap_fit_bulk", "mma_gap_fit_rows"):
        assert res[fit]["R_GBps"] > 0 and res[fit]["heldout"]["n"] > 0
    (row,) = res["rows"]
    for key in ("fused_ms", "fused_row_stores_ms", "contig_ms", "contig_row_stores_ms", "permute_ms"):
        assert row[key] > 0 and math.isfinite(row[key])
    assert row["pred_completion_coupled"] >= row["pred_burst_gap"] >= 0
    assert row["pred_unbounded_async"] == 0
    for name in ("fused_bulk", "fused_rows", "contig_bulk"):
        tr = row["traced"][name]
        assert tr["store_span_ns"]["n"] > 0 and tr["store_span_ns"]["p50"] > 0
        assert sum(tr["store_span_hist_ns"]["counts"]) == tr["store_span_ns"]["n"]
        busy = tr["cta_qloop_busy_fraction"]
        assert 0 < busy["min"] <= busy["max"] <= 1
        assert len(tr["cta0_timeline_ns"]) > 0
