"""Host side of the Burst-Gap probe: sweeps, fits of T0_iss, R and Q, and
predictions of the issuer-visible burst issue time.

X-Stage pages, Technical Summary, "Methodology": a burst of V bytes of
remote stores from K producers, followed by a useful producer gap G, takes
the issuer T_iss(G; K, V) = max(T0_iss(K, V), V/R - G) to issue, where T0_iss
is the backpressure-free issue time and R the effective drain rate; Q is the
effective pending capacity. "Key Contributions": the three quantities are
measured by parameterised microbenchmarks and then predict steady-state
periods, issuer-visible overhead and the onset of backpressure without
refitting.

The probe kernel (``xstage_probe_run``) records three %globaltimer stamps per
producer and round; everything here is arithmetic on those stamps.
Here stores go to local HBM, so R is the local store-drain rate.

Fitting (the pages give no procedure; this one is our own):
  * T0(K, V): median issue time of rounds whose gap is long enough that the
    previous burst has drained (the largest G measured for that K, V);
  * R: from the drain-dominated points, where the steady-state period
    T_iss + G equals V / R;
  * Q: from the knee of the long-gap floor against V. With an empty queue
    at each burst, the floor is the issue-limited time, which grows linearly
    in V, until one burst overflows the capacity; past the knee the floor is
    (V - Q) / R. The line through the two smallest volumes extrapolates the
    issue-limited time; for volumes whose floor exceeds it by 25 % or more,
    Q = V - R * floor. (This reading of Q is our own; the pages' equation
    does not contain Q.)
"""
from __future__ import annotations

import statistics
from dataclasses import dataclass, field


def predict_t_iss(G: float, T0: float, V: float, R: float) -> float:
    """Issuer-visible issue time of a burst (seconds): max(T0, V/R - G)."""
    drain = V / R - G
    return T0 if T0 >= drain else drain


@dataclass
class Point:
    """One probe launch: K producers, burst V bytes, gap G seconds, per-round stamps."""

    K: int
    V: float
    G: float
    store_kind: int
    t_iss: list  # seconds, per round (mean over producers), warm-up rounds dropped
    period: list  # seconds, per round
    first: float  # issue time of round 0 (empty queue), mean over producers

    @property
    def t_iss_med(self) -> float:
        return statistics.median(self.t_iss)

    @property
    def period_med(self) -> float:
        return statistics.median(self.period)


def reduce_stamps(stamps, discard: int = 3):
    """stamps: nested [K][rounds][3] ints (ns). Returns (t_iss, period, first) in seconds."""
    K = len(stamps)
    rounds = len(stamps[0])
    t_iss, period = [], []
    for r in range(rounds):
        iss = [stamps[p][r][1] - stamps[p][r][0] for p in range(K)]
        per = [stamps[p][r][2] - stamps[p][r][0] for p in range(K)]
        if r >= discard:
            t_iss.append(sum(iss) / K * 1e-9)
            period.append(sum(per) / K * 1e-9)
    first = sum(stamps[p][0][1] - stamps[p][0][0] for p in range(K)) / K * 1e-9
    return t_iss, period, first


@dataclass
class Fit:
    T0: dict = field(default_factory=dict)  # (K, V, store_kind) -> seconds
    R: float = 0.0  # bytes / second
    Q: float | None = None  # bytes

    def t0(self, K, V, store_kind):
        return self.T0[(K, V, store_kind)]

    def predict(self, p: Point) -> float:
        return predict_t_iss(p.G, self.t0(p.K, p.V, p.store_kind), p.V, self.R)


def fit(points: list[Point], drain_factor: float = 1.5) -> Fit:
    """Fit T0 per (K, V, kind), then R and Q (see module docstring)."""
    f = Fit()
    groups: dict = {}
    for p in points:
        groups.setdefault((p.K, p.V, p.store_kind), []).append(p)
    for key, ps in groups.items():
        gmax = max(p.G for p in ps)
        f.T0[key] = statistics.median([p.t_iss_med for p in ps if p.G == gmax])
    rates = []
    for p in points:
        if p.t_iss_med > drain_factor * f.T0[(p.K, p.V, p.store_kind)]:
            rates.append(p.V / (p.t_iss_med + p.G))
    if rates:
        f.R = statistics.median(rates)
    else:  # nothing drain-dominated: R is at least V / (T0 + G) for every point
        f.R = max(p.V / (p.t_iss_med + p.G) for p in points)
    qs = []
    kinds: dict = {}
    for (K, V, kind), t0 in f.T0.items():
        kinds.setdefault((K, kind), []).append((V, t0))
    for (_K, _kind), vt in kinds.items():
        vt.sort()
        if len(vt) < 3 or vt[1][0] == vt[0][0]:
            continue
        slope = (vt[1][1] - vt[0][1]) / (vt[1][0] - vt[0][0])
        for V, floor in vt[2:]:
            issue_limited = vt[0][1] + slope * (V - vt[0][0])
            if floor > 1.25 * issue_limited:
                qs.append(V - f.R * floor)
    f.Q = statistics.median(qs) if qs else None
    return f


def residuals(f: Fit, points: list[Point]) -> list[float]:
    """Relative error (predicted - measured) / measured of T_iss at each point."""
    return [(f.predict(p) - p.t_iss_med) / p.t_iss_med for p in points]


def calibrate_fma(run_gap_only, target_ns: float, iters0: int = 1000) -> int:
    """Dependent-FMA iterations per gap that last about target_ns.

    run_gap_only(iters) must return the measured mean gap in ns for that
    iteration count (a probe launch with a minimal burst)."""
    ns = run_gap_only(iters0)
    per_iter = max(ns, 1.0) / iters0
    return max(0, int(round(target_ns / per_iter)))
