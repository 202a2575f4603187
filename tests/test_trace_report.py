"""The task-trace summary on a hand-built trace (no GPU)."""
import numpy as np
import pytest

from persistent_megakernel_sm_gb300.trace_report import EXIT_TASK, format_summary, summarize


def _rec(cta, ttype, payload, claim, start, end):
    return cta, (ttype << 28) | payload, claim, start, end


def _trace(records):
    a = np.array(records, dtype=np.int64)
    return {"cta": a[:, 0], "task": a[:, 1], "t_claim": a[:, 2], "t_start": a[:, 3],
            "t_end": a[:, 4]}


def test_summary_of_a_two_cta_trace():
    us = 1000  # trace times are ns
    recs = [
        # CTA 0: a router tile 0-10 us, a gate/up tile 12-30 us
        _rec(0, 1, 0, 0, 0, 10 * us), _rec(0, 3, 5, 11 * us, 12 * us, 30 * us),
        # CTA 1: a gather 10-14 us, a down tile 20-40 us
        _rec(1, 2, 1, 9 * us, 10 * us, 14 * us), _rec(1, 4, 7, 19 * us, 20 * us, 40 * us),
        # one plan phase record and the two exit records
        _rec(0, 6, 1, 10 * us, 10 * us, 10 * us),
        (0, EXIT_TASK, 0, 0, 41 * us), (1, EXIT_TASK, 0, 0, 41 * us),
    ]
    s = summarize(_trace(recs), n_bins=4)
    assert s["grid"] == 2
    assert s["span_us"] == pytest.approx(40.0)
    assert s["types"]["route"] == {"n": 1, "start_us": 0.0, "end_us": 10.0,
                                   "median_us": 10.0, "max_us": 10.0}
    assert s["types"]["down"]["median_us"] == pytest.approx(20.0)
    # (10 + 18 + 4 + 20) us of tasks over 2 CTAs
    assert s["busy_us"] == pytest.approx(26.0)
    # window [0, 10): CTA 0 routes all of it -> half the grid's time
    assert s["bins"][0]["route"] == pytest.approx(0.5)
    assert s["bins"][0]["total"] == pytest.approx(0.5)
    # window [10, 20): gate/up 8 us + gather 4 us of 20 CTA-us
    assert s["bins"][1]["gateup"] == pytest.approx(0.4)
    assert s["bins"][1]["gather"] == pytest.approx(0.2)
    # gaps: CTA 0 10 -> 12 us, CTA 1 14 -> 20 us
    assert s["gaps"]["n"] == 2
    assert s["gaps"]["median_us"] == pytest.approx(4.0)
    assert s["gaps"]["sum_over_grid_us"] == pytest.approx(4.0)
    assert s["plan_phases_us"] == [pytest.approx(10.0)]
    text = format_summary(s)
    assert "gateup" in text and "span 40.0 us" in text


def test_summary_of_an_empty_trace():
    s = summarize(_trace([(0, EXIT_TASK, 0, 0, 5)]))
    assert s["types"] == {} and s["grid"] == 1 and s["bins"] == []
