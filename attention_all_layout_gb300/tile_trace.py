"""Host-side reading of the per-tile trace of a traced attention call.

The X-Stage pages validate their model with two views of the fused kernel
("Results": tensor-core timelines, and the distribution of store spans that
runs from broad and drain-limited to a narrow backpressure-free floor). A
call given `trace=` (the C ABI's attn_a2a_opts.trace) records, for every work
item (a pair of 128-row query tiles of one (b, h)), query tile t and warp w of
the tile owner's warpgroup, eight int64:

  0 %globaltimer ns, the tile's first scores ready (its Q loop starts)
  1 %globaltimer ns, its O accumulator final (the Q loop ends)
  2 %globaltimer ns, the warp starts issuing the tile's output stores
  3 %globaltimer ns, the warp has issued them and resumes
  4 SM cycles from 2 to 3
  5 SM id, 6 CTA index, 7 first sequence row of the tile

Everything here is arithmetic on those records: the store span of a tile
(first warp starting to issue to last warp resuming), its issue cycles, and
per-CTA timelines of the Q loops (when the tensor core works on which tile).
"""
from __future__ import annotations

import numpy as np

RECORD = 8


def records(trace, B: int, H: int, S: int) -> np.ndarray:
    """The trace as an int64 array [items, 2 tiles, 4 warps, RECORD]."""
    pairs = ((S + 127) // 128 + 1) // 2
    items = B * H * pairs
    a = trace.detach().cpu().numpy() if hasattr(trace, "detach") else np.asarray(trace)
    return a[: items * 2 * 4 * RECORD].reshape(items, 2, 4, RECORD)


def tile_rows(rec: np.ndarray, S: int) -> np.ndarray:
    """Mask [items, 2]: the tile holds at least one row < S (an odd block count
    leaves the second tile of a head's last item without rows)."""
    return rec[:, :, 0, 7] < S


def store_span_ns(rec: np.ndarray) -> np.ndarray:
    """[items, 2]: from the first warp starting to issue the tile's stores to
    the last warp resuming."""
    return rec[:, :, :, 3].max(axis=2) - rec[:, :, :, 2].min(axis=2)


def issue_cycles(rec: np.ndarray) -> np.ndarray:
    """[items, 2]: the longest issue time of the tile's four warps, SM cycles."""
    return rec[:, :, :, 4].max(axis=2)


def qloop_ns(rec: np.ndarray) -> np.ndarray:
    """[items, 2]: duration of the tile's Q loop (first scores to final O)."""
    return rec[:, :, 0, 1] - rec[:, :, 0, 0]


def quantiles(x: np.ndarray, qs=(0.1, 0.5, 0.9, 0.99)) -> dict:
    x = np.asarray(x, dtype=np.float64).ravel()
    out = {f"p{int(q * 100)}": float(np.quantile(x, q)) for q in qs}
    out["min"] = float(x.min())
    out["max"] = float(x.max())
    out["n"] = int(x.size)
    return out


def histogram(x: np.ndarray, bins: int = 12) -> dict:
    """Log-spaced histogram of positive values (counts and bin edges)."""
    x = np.asarray(x, dtype=np.float64).ravel()
    x = x[x > 0]
    lo, hi = x.min(), x.max()
    if hi <= lo:
        hi = lo * 1.01
    edges = np.geomspace(lo, hi, bins + 1)
    counts, _ = np.histogram(x, bins=edges)
    return {"edges": [float(e) for e in edges], "counts": [int(c) for c in counts]}


def cta_timeline(rec: np.ndarray, cta: int, grid: int) -> list:
    """The Q loops and store spans of one CTA's tiles, in item order, relative
    to the CTA's first stamp (ns): (item, tile, q_start, q_end, st_begin, st_end)."""
    items = range(cta, rec.shape[0], grid)
    rows = []
    for i in items:
        for t in range(2):
            r = rec[i, t]
            rows.append((i, t, int(r[0, 0]), int(r[0, 1]), int(r[:, 2].min()), int(r[:, 3].max())))
    if not rows:
        return []
    base = min(r[2] for r in rows)
    return [(i, t, a - base, b - base, c - base, d - base) for (i, t, a, b, c, d) in rows]


def summary(rec: np.ndarray, S: int, grid: int) -> dict:
    """Span distribution and per-CTA busy fraction of a traced call."""
    m = tile_rows(rec, S)
    span = store_span_ns(rec)[m]
    cyc = issue_cycles(rec)[m]
    ql = qloop_ns(rec)[m]
    # per CTA: the share of its lifetime in which at least one of its tiles is
    # in its Q loop (the tensor core has work)
    busy = []
    for c in range(min(grid, rec.shape[0])):
        tl = cta_timeline(rec, c, grid)
        if not tl:
            continue
        iv = sorted((a, b) for (_, _, a, b, _, _) in tl)
        end = max(d for (*_, d) in tl)
        covered, cur_a, cur_b = 0, iv[0][0], iv[0][1]
        for a, b in iv[1:]:
            if a > cur_b:
                covered += cur_b - cur_a
                cur_a, cur_b = a, b
            else:
                cur_b = max(cur_b, b)
        covered += cur_b - cur_a
        busy.append(covered / end if end > 0 else 1.0)
    return {"store_span_ns": quantiles(span), "store_span_hist_ns": histogram(span),
            "issue_cycles": quantiles(cyc), "qloop_ns": quantiles(ql),
            "cta_qloop_busy_fraction": quantiles(np.array(busy)) if busy else None}
