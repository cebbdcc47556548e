"""Burst-Gap sweep on the current GPU: runs the probe over a (V, G, K, store
kind) grid, fits T0_iss, R and Q, and reports the equation's predictions on
held-out points (X-Stage pages, Technical Summary, "Methodology"; "Key
Contributions", characterisation and prediction).

Usage: python -m attention_all_layout_gb300.probe_sweep [--quick] [--out FILE]
       python -m attention_all_layout_gb300.probe_sweep --single V_MB [--rounds N]
           [--kind 0|1] [--G-us G] (one probe launch, e.g. for a profiler)
The destination of the bursts rotates through a buffer of at least four
times the L2 size and four times the largest burst. The grid holds bursts
smaller than L2 (1-64 MB), which L2 can absorb whole, and bursts of two to
four times L2 (128-512 MB), which it cannot; both are fitted and reported
apart, next to the write-only HBM rate of a plain fill (CUDA events).
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

G_US = (0, 0.5, 1, 2, 4, 6, 8, 10, 12, 16, 20)
V_MB = (1, 2, 4, 8, 16, 32, 64)
V_MB_BEYOND_L2 = (128, 256, 512)  # 1x-4x the 126.5 MB L2 of a GB300
G_US_BEYOND_L2 = (0, 5, 10, 20, 40, 60, 80, 120)


def round_volume(v_bytes: float, K: int) -> int:
    unit = 4096 * K
    return max(unit, int(round(v_bytes / unit)) * unit)


class Prober:
    """Probe launches into one destination buffer: device memory, or with
    host=True pinned host memory that the GPU stores to over the host link."""

    def __init__(self, dst_bytes: int, max_stamps: int, host: bool = False):
        if host:
            self.dst = torch.empty(dst_bytes, dtype=torch.uint8, pin_memory=True)
        else:
            self.dst = torch.empty(dst_bytes, dtype=torch.uint8, device="cuda")
        self.stamps = torch.zeros(max_stamps, dtype=torch.int64, device="cuda")

    def run(self, K, V, G_ns, rounds, store_kind=0, gap_kind=0, fma_iters=0, discard=None) -> bg.Point:
        st = self.stamps[: K * rounds * 3]
        bd.xstage_probe_run(K, rounds, V, int(G_ns), self.dst, st, store_kind=store_kind, gap_kind=gap_kind,
                            fma_iters=fma_iters)
        torch.cuda.synchronize()
        s = st.view(K, rounds, 3).cpu().tolist()
        # keep the second half: the queue needs rounds to reach its steady state
        t_iss, period, first = bg.reduce_stamps(s, discard=rounds // 2 if discard is None else discard)
        return bg.Point(K=K, V=float(V), G=G_ns * 1e-9, store_kind=store_kind, t_iss=t_iss, period=period,
                        first=first)


def measured_gap(p: bg.Point) -> float:
    """Median gap actually spent per round (period - issue time), seconds."""
    return statistics.median([per - iss for per, iss in zip(p.period, p.t_iss)])


def sweep_mma_gap(pr: "Prober", K: int, idle_fit: bg.Fit, vmbs=(8, 32, 64), gaps_us=(0, 1, 2, 4, 6, 8, 12, 20),
                  kinds=(0, 1), rounds: int = 48):
    """Burst-Gap check with tensor-core work as the gap (gap_kind 2): each
    round issues its stores, then tcgen05 MMAs that the producer waits for, so
    the issue time is the MMA pipe's stall. G is the measured gap. The points
    are predicted with T0 and R fitted on the idle-gap sweep, without refitting
    (the pages' claim: the measured quantities predict issuer-visible overhead
    without application-specific refitting); residuals are reported per store
    kind."""
    V0 = ps_round(K)
    cal = pr.run(K, V0, 0, 16, gap_kind=2, fma_iters=4000)
    ns_per_mma = max(measured_gap(cal) * 1e9, 1.0) / 4000
    pts = []
    for kind in kinds:
        for vmb in vmbs:
            V = round_volume(vmb * 2**20, K)
            for g in gaps_us:
                n = int(round(g * 1000 / ns_per_mma))
                p = pr.run(K, V, 0, rounds, store_kind=kind, gap_kind=2, fma_iters=n)
                p.G = measured_gap(p)
                pts.append(p)
    out = {"ns_per_mma_128x128x16": ns_per_mma, "per_kind": {}, "points": []}
    for kind in kinds:
        ks = [p for p in pts if p.store_kind == kind and (p.K, p.V, kind) in idle_fit.T0]
        res = [(idle_fit.predict(p) - p.t_iss_med) / p.t_iss_med for p in ks]
        if res:
            out["per_kind"][str(kind)] = {"n": len(res), "median_abs_rel": statistics.median(abs(r) for r in res),
                                          "max_abs_rel": max(abs(r) for r in res),
                                          "frac_within_15pct": sum(abs(r) <= 0.15 for r in res) / len(res)}
    for p in pts:
        key = (p.K, p.V, p.store_kind)
        out["points"].append({"V_MB": p.V / 2**20, "kind": p.store_kind, "G_us": p.G * 1e6,
                              "stall_us": p.t_iss_med * 1e6,
                              "pred_idle_fit_us": idle_fit.predict(p) * 1e6 if key in idle_fit.T0 else None})
    return out


def ps_round(K: int) -> int:
    return 4096 * K


def l2_bytes() -> int:
    return int(torch.cuda.get_device_properties(0).L2_cache_size)


def hbm_write_rates(gib: int = 4, reps: int = 5) -> dict:
    """Write-only HBM rate over `reps` back-to-back launches timed by CUDA
    events (a launch leaves up to one L2 of dirty lines, which the next
    launch's stores push out, so the average is the drain rate), three ways:
      * fill: torch's fill of a `gib` GiB float32 buffer (a plain vector-store kernel);
      * probe_K: the probe kernel as a fill, one round of one burst of `gib` GiB
        (st.global.v4, the epilogue's store kind) from K producer CTAs: K = the
        SM count (equal static shares: the slowest SM sets the time), and
        K = 1024 (many CTAs, handed out to SMs as they free up).
    Also the spread of the per-producer issue times of the K = SM-count burst."""
    n = gib * 2**30
    buf = torch.empty(n // 4, dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / reps

    out = {"bytes": n, "reps": reps, "fill_GBps": n / timed(lambda: buf.fill_(7.0)) / 1e9}
    nsm = bd.num_sms()
    stamps = torch.zeros(1024 * 3, dtype=torch.int64, device="cuda")
    for K in (nsm, 1024):
        V = (n // (4096 * K)) * 4096 * K
        st = stamps[: K * 3]
        out[f"probe_K{K}_GBps"] = V / timed(lambda: bd.xstage_probe_run(K, 1, V, 0, buf, st, store_kind=0)) / 1e9
        if K == nsm:
            s_ = st.view(K, 3).cpu().double()
            iss = (s_[:, 1] - s_[:, 0]) * 1e-3
            end = (s_[:, 1] - s_[:, 0].min()) * 1e-3
            out["probe_per_producer_issue_us"] = {"min": float(iss.min()), "median": float(iss.median()),
                                                  "max": float(iss.max())}
            out["probe_last_issue_end_us"] = float(end.max())
            out["probe_rate_by_last_end_GBps"] = V / (float(end.max()) * 1e-6) / 1e9
    del buf
    torch.cuda.empty_cache()
    return out


def single(V_mb: float, rounds: int, kind: int, G_us: float, K: int = 0) -> dict:
    """One probe launch of `rounds` bursts of V_mb MB from K producers (0 =
    one per SM), destination four bursts long; returns the stamps' summary,
    with the spread over producers. Sized for a profiler capture: one launch,
    a few hundred MB to ~4 GB on the device."""
    K = K or bd.num_sms()
    V = round_volume(V_mb * 2**20, K)
    pr = Prober(4 * V, K * rounds * 3)
    st = pr.stamps[: K * rounds * 3]
    bd.xstage_probe_run(K, rounds, V, int(G_us * 1000), pr.dst, st, store_kind=kind)
    torch.cuda.synchronize()
    s_ = st.view(K, rounds, 3).cpu().double()
    iss = (s_[:, :, 1] - s_[:, :, 0]) * 1e-3  # us, [K, rounds]
    span = (s_[:, -1, 1].max() - s_[:, 0, 0].min()) * 1e-3
    return {"K": K, "V_bytes": V, "rounds": rounds, "kind": kind, "G_us": G_us,
            "t_iss_mean_us": iss.mean(dim=0).tolist(), "t_iss_max_us": iss.max(dim=0).values.tolist(),
            "t_iss_min_us": iss.min(dim=0).values.tolist(),
            "first_start_to_last_issue_us": float(span),
            "rate_by_span_GBps": V * rounds / (float(span) * 1e-6) / 1e9}


def split_fit(points, seed: int, g_max: float):
    """Calibration / held-out split (about a third of the points with
    0 < G < g_max held out), the fit on the calibration points, and the
    held-out residuals."""
    rnd = random.Random(seed)
    held, cal = [], []
    for p in points:
        edge = p.G < 1e-12 or abs(p.G - g_max) < 1e-12
        (held if rnd.random() < 0.33 and not edge else cal).append(p)
    f = bg.fit(cal)
    res = bg.residuals(f, held)
    summary = {"n": len(held), "median_abs_rel": statistics.median([abs(r) for r in res]) if res else None,
               "max_abs_rel": max((abs(r) for r in res), default=None),
               "frac_within_15pct": (sum(abs(r) <= 0.15 for r in res) / len(res)) if res else None}
    return f, summary


def fit_summary(f: bg.Fit) -> dict:
    return {"R_GBps": f.R / 1e9, "Q_MB": None if f.Q is None else f.Q / 2**20,
            "T0_us": {f"K={k[0]} V={k[1] / 2**20:.2f}MB kind={k[2]}": v * 1e6 for k, v in f.T0.items()}}


def sweep(quick: bool = False, kinds=(0, 1), rounds: int = 64, seed: int = 0) -> dict:
    K = bd.num_sms()
    gs = G_US if not quick else (0, 1, 4, 10, 20)
    vs = V_MB if not quick else (2, 16, 64)
    gs_big = G_US_BEYOND_L2 if not quick else (0, 20, 60, 120)
    vs_big = V_MB_BEYOND_L2 if not quick else (256,)
    dst_bytes = max(4 * l2_bytes(), 4 * max(vs_big) * 2**20)
    dst_bytes = (dst_bytes // (4096 * K) + 1) * 4096 * K
    pr = Prober(dst_bytes, 1024 * rounds * 3)
    pr.run(K, round_volume(2**20, K), 0, 5)  # warm-up launch
    points, big = [], []
    for kind in kinds:
        for vmb in vs:
            V = round_volume(vmb * 2**20, K)
            for g in gs:
                points.append(pr.run(K, V, g * 1000, rounds, store_kind=kind))
        for vmb in vs_big:
            V = round_volume(vmb * 2**20, K)
            for g in gs_big:
                big.append(pr.run(K, V, g * 1000, max(16, rounds // 2), store_kind=kind))
    # T0 as a function of the producer count, backpressure-free (long gap)
    t0_k = []
    for k in (1, 8, 32, K):
        V = round_volume(8 * 2**20, k)
        p = pr.run(k, V, 20000, rounds, store_kind=0)
        t0_k.append({"K": k, "V": V, "t0_us": p.t_iss_med * 1e6})
    f, held = split_fit(points, seed, max(gs) * 1e-6)
    f_big, held_big = split_fit(big, seed, max(gs_big) * 1e-6)
    f_all, held_all = split_fit(points + big, seed, max(gs_big) * 1e-6)
    # bursts beyond L2, predicted by the fit on bursts within L2 (T0 of the
    # large bursts from their own long-gap floor, R from the small bursts)
    cross = None
    if f_big.T0:
        f_x = bg.Fit(T0=dict(f_big.T0), R=f.R, Q=f.Q)
        res = bg.residuals(f_x, big)
        cross = {"R_small_GBps": f.R / 1e9, "R_big_GBps": f_big.R / 1e9,
                 "median_abs_rel": statistics.median(abs(r) for r in res), "max_abs_rel": max(abs(r) for r in res)}
    mma = sweep_mma_gap(pr, K, f, rounds=max(16, rounds // 2)) if not quick else sweep_mma_gap(
        pr, K, f, vmbs=(16, 64), gaps_us=(0, 2, 6, 20), rounds=32)
    del pr
    torch.cuda.empty_cache()
    rates = hbm_write_rates(gib=2 if quick else 4)

    def rows(pts, fit_):
        return [{"V_MB": p.V / 2**20, "G_us": p.G * 1e6, "kind": p.store_kind, "t_iss_us": p.t_iss_med * 1e6,
                 "period_us": p.period_med * 1e6, "first_us": p.first * 1e6,
                 "pred_us": fit_.predict(p) * 1e6 if (p.K, p.V, p.store_kind) in fit_.T0 else None}
                for p in pts]

    out = {
        "K": K,
        "l2_bytes": l2_bytes(),
        "dst_bytes": dst_bytes,
        "rounds": rounds,
        "hbm_write": rates,
        "fit": fit_summary(f),
        "heldout": held,
        "fit_beyond_l2": fit_summary(f_big),
        "heldout_beyond_l2": held_big,
        "fit_all": fit_summary(f_all),
        "heldout_all": held_all,
        "beyond_l2_with_small_burst_R": cross,
        "t0_vs_K": t0_k,
        "mma_gap": mma,
        "points": rows(points, f),
        "points_beyond_l2": rows(big, f_big),
    }
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--out", default=None)
    ap.add_argument("--single", type=float, default=None, metavar="V_MB",
                    help="one probe launch of bursts of V_MB MB (all SMs) instead of the sweep")
    ap.add_argument("--rounds", type=int, default=4)
    ap.add_argument("--kind", type=int, default=0)
    ap.add_argument("--G-us", type=float, default=0.0)
    ap.add_argument("--K", type=int, default=0, help="producers of --single (0 = one per SM)")
    a = ap.parse_args(argv)
    if a.single is not None:
        res = single(a.single, a.rounds, a.kind, a.G_us, a.K)
        print(json.dumps(res), flush=True)
        return 0
    res = sweep(quick=a.quick)
    text = json.dumps(res, indent=1)
    if a.out:
        with open(a.out, "w") as fh:
            fh.write(text)
    keys = ("K", "hbm_write", "fit", "heldout", "fit_beyond_l2", "heldout_beyond_l2", "fit_all", "heldout_all",
            "beyond_l2_with_small_burst_R", "t0_vs_K")
    print(json.dumps({k: res[k] for k in keys}, indent=1))
    print(json.dumps({k: v for k, v in res["mma_gap"].items() if k != "points"}, indent=1))
    return 0


if __name__ == "__main__":
    sys.exit(main())
