"""CPU tests of the trace reader (attention_all_layout_gb300.tile_trace) on
hand-made records: spans, cycles, Q-loop durations, row masks, per-CTA
timelines and the busy fraction."""
import numpy as np
import pytest

from attention_all_layout_gb300 import tile_trace as tt


def make(items=4, grid=2, S=4 * 256 - 100):
    rec = np.zeros((items, 2, 4, tt.RECORD), dtype=np.int64)
    for i in range(items):
        c, k = i % grid, i // grid
        for t in range(2):
            q0 = 1000 + k * 1000 + t * 10
            rec[i, t, :, 0] = q0
            rec[i, t, :, 1] = q0 + 800
            for w in range(4):
                rec[i, t, w, 2] = q0 + 810 + w  # warps start issuing one ns apart
                rec[i, t, w, 3] = q0 + 850 + 2 * w
                rec[i, t, w, 4] = 40 + w
            rec[i, t, :, 6] = c
            rec[i, t, :, 7] = (2 * i + t) * 128
    return rec, S, grid


def test_spans_cycles_qloop():
    rec, S, grid = make()
    assert np.all(tt.store_span_ns(rec) == (850 + 6) - 810)
    assert np.all(tt.issue_cycles(rec) == 43)
    assert np.all(tt.qloop_ns(rec) == 800)


def test_row_mask_and_records_shape():
    rec, S, grid = make(items=4, S=7 * 128 + 5)
    m = tt.tile_rows(rec, S)
    assert m.sum() == 8  # rows 0..901: every tile up to the one starting at 896
    flat = rec.reshape(-1)
    assert tt.records(flat, 1, 1, 8 * 128).shape == (4, 2, 4, tt.RECORD)


def test_timeline_and_busy_fraction():
    rec, S, grid = make(items=4, grid=2)
    tl = tt.cta_timeline(rec, 0, grid)
    assert [r[:2] for r in tl] == [(0, 0), (0, 1), (2, 0), (2, 1)]
    assert tl[0][2] == 0
    s = tt.summary(rec, S=8 * 128, grid=grid)
    # per CTA: Q loops cover [0, 810) and [1000, 1810) of a life ending at 1866
    assert s["cta_qloop_busy_fraction"]["p50"] == pytest.approx(1620 / 1866)
    assert s["store_span_ns"]["n"] == 8


def test_histogram_counts_everything():
    x = np.array([1, 2, 3, 10, 100, 1000], dtype=float)
    h = tt.histogram(x, bins=5)
    assert sum(h["counts"]) == len(x)
