"""Issuer-visible overhead of the piggybacked all-to-all across sequence
length, next to the Burst-Gap prediction and the two counterfactual models
the X-Stage pages test against ("Results", FlashAttention-A2A optimisation:
the fused kernel's overhead over attention alone stays flat and near zero as
S grows, contradicting a completion-coupled model whose overhead grows with
S; "Key Contributions": neither fully blocking nor unbounded-asynchronous
models capture issuer-visible behaviour).

For each S the same kernel runs with the all-to-all epilogue (fused) and with
the contiguous epilogue (attention alone), each with bulk tensor stores and
with row stores from registers; the serial baseline (attention alone with
bulk stores, then the separate permute) is compared with the fused call under
the automatic store kind. The models, per work item of a CTA (two 128-row tiles, so
V_item = 2 * 128 * 2d bytes of stores, and a compute gap G_item = the item's
share of attention-alone time):

  * Burst-Gap (pages' equation, fitted T0 and R from a probe sweep on this
    GPU): the burst of all CTAs finishing an item together, V = n_SM * V_item,
    costs the issuer T_iss = max(T0(V), V/R - G_item) per item;
  * completion-coupled counterfactual: the issuer also waits until its stores
    are drained, i.e. T0(V) + V/R per item;
  * unbounded-asynchronous counterfactual: the issuer never waits: 0.
Predicted overhead = items per SM * per-item cost, relative to attention
alone. The measured overhead is t_fused / t_contig - 1.

Two fits of T0 and R enter: row stores use the fit on bursts followed by an
idle gap; bulk tensor stores use a fit on bursts followed by tensor-core work
(the probe's gap_kind 2), since the copies read shared memory, which the
tensor core also reads, and so drain at a different rate while it is busy.
Each fit reports its held-out residual.

Traced runs of the same calls give the per-tile view: the distribution of
store spans (first warp starting to issue a tile's stores to the last warp
resuming), which the Burst-Gap equation predicts as T_iss per tile, and the
share of each CTA's time in which one of its tiles is in its Q loop.

Usage: python -m attention_all_layout_gb300.overhead_report [--out FILE]
"""
from __future__ import annotations

import argparse
import json
import random
import statistics
import sys

import torch

from . import binding as bd
from . import burst_gap as bg
from . import probe_sweep as ps
from . import tile_trace as tt
from . import workloads

S_LIST = (1024, 2048, 4096, 8192, 16384, 32768)
ROUNDS = 3


def time_ms(fn, n):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def fit_store_model():
    """T0(V) table and R from a short probe sweep (st.global.v4, the epilogue's store kind)."""
    K = bd.num_sms()
    dst_bytes = (max(4 * ps.l2_bytes(), 256 * 2**20) // (4096 * K) + 1) * 4096 * K
    pr = ps.Prober(dst_bytes, K * 64 * 3)
    pts = []
    for vmb in (1, 2, 4, 8, 16, 32, 64):
        V = ps.round_volume(vmb * 2**20, K)
        for g in (0, 1, 2, 4, 10, 40):
            pts.append(pr.run(K, V, g * 1000, 48, store_kind=0))
    f = bg.fit(pts)
    table = sorted((V, t0) for (k, V, kind), t0 in f.T0.items())
    return f.R, table


def fit_store_model_mma(kind: int, seed: int = 0):
    """T0(V) table and R of one store kind with tensor-core work as the gap
    (probe gap_kind 2), fitted on a calibration split of a sweep; the held-out
    residual is returned with it. G is the measured gap."""
    K = bd.num_sms()
    dst_bytes = (max(4 * ps.l2_bytes(), 256 * 2**20) // (4096 * K) + 1) * 4096 * K
    pr = ps.Prober(dst_bytes, K * 64 * 3)
    cal = pr.run(K, ps.ps_round(K), 0, 16, gap_kind=2, fma_iters=4000)
    ns_per_mma = max(ps.measured_gap(cal) * 1e9, 1.0) / 4000
    gaps = (0, 1, 2, 4, 8, 12, 20, 40)
    rnd = random.Random(seed)
    cal, held_pts = [], []
    for vmb in (1, 2, 4, 8, 16, 32, 64):
        V = ps.round_volume(vmb * 2**20, K)
        for g in gaps:
            p = pr.run(K, V, 0, 32, store_kind=kind, gap_kind=2, fma_iters=int(round(g * 1000 / ns_per_mma)))
            p.G = ps.measured_gap(p)
            # the shortest and longest gap of every volume calibrate (R and the
            # long-gap floor T0); about a third of the others are held out
            interior = g not in (gaps[0], gaps[-1])
            (held_pts if interior and rnd.random() < 0.33 else cal).append(p)
    f = bg.fit(cal)
    res = bg.residuals(f, held_pts)
    held = {"n": len(res), "median_abs_rel": statistics.median(abs(r) for r in res) if res else None,
            "max_abs_rel": max((abs(r) for r in res), default=None),
            "frac_within_15pct": (sum(abs(r) <= 0.15 for r in res) / len(res)) if res else None}
    table = sorted((V, t0) for (k, V, kd), t0 in f.T0.items())
    return f.R, table, held


def t0_of(table, V):
    """Linear interpolation of the long-gap floor T0 at volume V."""
    if V <= table[0][0]:
        return table[0][1] * V / table[0][0]
    for (v0, t0), (v1, t1) in zip(table, table[1:]):
        if V <= v1:
            return t0 + (t1 - t0) * (V - v0) / (v1 - v0)
    return table[-1][1] * V / table[-1][0]


def traced_summary(fn, B, H, S):
    """Per-tile trace of one call (after the timed legs): span quantiles and busy fraction."""
    trace = torch.zeros(bd.trace_numel(B, H, S), dtype=torch.int64, device="cuda")
    fn(trace)
    fn(trace)  # the second call's stamps (warm caches and clocks)
    torch.cuda.synchronize()
    pairs = ((S + 127) // 128 + 1) // 2
    grid = min(bd.num_sms(), B * H * pairs)
    rec = tt.records(trace, B, H, S)
    out = tt.summary(rec, S, grid)
    # CTA 0's tensor-core timeline: its first work items' Q loops and store spans (ns)
    out["cta0_timeline_ns"] = tt.cta_timeline(rec, 0, grid)[:8]
    return out


def report(H=40, d=128, P=8, s_list=S_LIST):
    R, table = fit_store_model()
    R_b, table_b, held_b = fit_store_model_mma(kind=1)
    R_r, table_r, held_r = fit_store_model_mma(kind=0)
    n_sm = bd.num_sms()
    rows = []
    for S in s_list:
        cfg = workloads.AttnConfig(f"S{S}", B=1, H=H, S=S, d=d, P=P)
        q, k, v = workloads.make_qkv(cfg, seed=0, device="cuda")
        parts = bd.alloc_partitions(1, S, H, d, P)
        o = torch.empty((1, H, S, d), dtype=torch.bfloat16, device="cuda")
        n = max(5, int(2e11 / cfg.flops * 50)) if cfg.flops < 2e11 else 10
        legs = {
            "f": lambda: bd.attn_a2a_fwd(q, k, v, P, cfg.scale, parts, store_kind=1),  # bulk tensor stores
            "r": lambda: bd.attn_a2a_fwd(q, k, v, P, cfg.scale, parts, store_kind=2),  # row stores
            "c": lambda: bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o, store_kind=1),  # bulk tensor stores
            "cr": lambda: bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o, store_kind=2),  # row stores
            "p": lambda: bd.attn_a2a_permute(o, P, parts),
        }
        # the legs take turns over several rounds (median per leg), so that a
        # clock change under the power cap does not land on one leg only
        samples = {name: [] for name in legs}
        for _ in range(ROUNDS):
            for name, fn in legs.items():
                samples[name].append(time_ms(fn, n))
        med = {name: sorted(v)[len(v) // 2] for name, v in samples.items()}
        t_f, t_r, t_c, t_cr, t_p = med["f"], med["r"], med["c"], med["cr"], med["p"]
        t_auto = t_f if bd.attn_a2a_store_kind(S, P, 1) == 1 else t_r  # the automatic store kind
        items = H * ((S + 127) // 128 + 1) // 2
        items_per_sm = -(-items // n_sm)
        g_item = t_c * 1e-3 / items_per_sm
        v_item = 2 * 128 * 2 * d
        V = n_sm * v_item
        t0 = t0_of(table, V)
        burst_gap = bg.predict_t_iss(g_item, t0, V, R) * items_per_sm
        coupled = (t0 + V / R) * items_per_sm
        # bulk stores, constants from tensor-core gaps
        t0_b = t0_of(table_b, V)
        burst_gap_b = bg.predict_t_iss(g_item, t0_b, V, R_b) * items_per_sm
        # the per-tile view: one tile's stores from every SM at once
        v_tile = n_sm * 128 * 2 * d
        tile_pred = {"rows_idle_fit_us": bg.predict_t_iss(g_item, t0_of(table, v_tile), v_tile, R) * 1e6,
                     "rows_mma_fit_us": bg.predict_t_iss(g_item, t0_of(table_r, v_tile), v_tile, R_r) * 1e6,
                     "bulk_mma_fit_us": bg.predict_t_iss(g_item, t0_of(table_b, v_tile), v_tile, R_b) * 1e6}
        spans = {
            "fused_bulk": traced_summary(lambda tr: bd.attn_a2a_fwd(q, k, v, P, cfg.scale, parts, store_kind=1,
                                                                    trace=tr), 1, H, S),
            "fused_rows": traced_summary(lambda tr: bd.attn_a2a_fwd(q, k, v, P, cfg.scale, parts, store_kind=2,
                                                                    trace=tr), 1, H, S),
            "contig_bulk": traced_summary(lambda tr: bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o, store_kind=1,
                                                                           trace=tr), 1, H, S),
        }
        rows.append({"S": S, "fused_ms": t_f, "fused_row_stores_ms": t_r, "contig_ms": t_c,
                     "contig_row_stores_ms": t_cr, "permute_ms": t_p,
                     "measured_overhead": t_f / t_c - 1, "measured_overhead_row_stores": t_r / t_c - 1,
                     "measured_overhead_rows_vs_rows": t_r / t_cr - 1,
                     "fused_auto_ms": t_auto, "serial_over_fused": (t_c + t_p) / t_auto,
                     "pred_burst_gap": burst_gap / (t_c * 1e-3),
                     "pred_burst_gap_bulk_mma_fit": burst_gap_b / (t_c * 1e-3),
                     "pred_completion_coupled": coupled / (t_c * 1e-3),
                     "pred_unbounded_async": 0.0, "items_per_sm": items_per_sm,
                     "gap_item_us": g_item * 1e6, "burst_MB": V / 2**20,
                     "tile_t_iss_pred": tile_pred, "traced": spans})
        del q, k, v, parts, o
        torch.cuda.empty_cache()
    return {"R_GBps": R / 1e9, "T0_table_us": [(V / 2**20, t * 1e6) for V, t in table], "H": H, "d": d,
            "P": P,
            "mma_gap_fit_bulk": {"R_GBps": R_b / 1e9, "T0_table_us": [(V / 2**20, t * 1e6) for V, t in table_b],
                                 "heldout": held_b},
            "mma_gap_fit_rows": {"R_GBps": R_r / 1e9, "T0_table_us": [(V / 2**20, t * 1e6) for V, t in table_r],
                                 "heldout": held_r},
            "rows": rows}


def order_comparison(names=("image", "joint", "video")):
    """Sequence-order vs chunk-interleaved work items (burst shaping): same
    results, different store pattern. With the epilogue's bursts far past the
    Burst-Gap knee the model predicts no difference."""
    out = []
    for name in names:
        cfg = workloads.CONFIGS[name]
        q, k, v = workloads.make_qkv(cfg, seed=0, device="cuda")
        parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
        n = 10 if cfg.flops > 1e13 else 100
        t = [time_ms(lambda o=o: bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, parts, tile_order=o), n) for o in (0, 1)]
        out.append({"config": name, "sequence_order_ms": t[0], "chunk_interleaved_ms": t[1],
                    "interleaved_over_sequence": t[1] / t[0]})
        del q, k, v, parts
        torch.cuda.empty_cache()
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    ap.add_argument("--orders-only", action="store_true", help="only the burst-shaping order comparison")
    a = ap.parse_args(argv)
    if a.orders_only:
        res = {"orders": order_comparison()}
        print(json.dumps(res, indent=1))
        if a.out:
            with open(a.out, "w") as fh:
                fh.write(json.dumps(res, indent=1))
        return 0
    res = report()
    res["orders"] = order_comparison()
    text = json.dumps(res, indent=1)
    if a.out:
        with open(a.out, "w") as fh:
            fh.write(text)
    print(text)
    return 0


if __name__ == "__main__":
    sys.exit(main())
