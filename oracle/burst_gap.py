"""CPU oracle for the Burst-Gap model of remote-store issue time.

TEST INFRASTRUCTURE ONLY: used by ``tests/`` and by nothing on the product
path. It shares no code with the probe's own fitting routine.

Source (X-Stage: An Overlooked Pipeline Stage for Communication-Computation
Overlap in DiT Inference, gist.science explanation, Technical Summary,
"Methodology: the X-Stage abstraction and the Burst-Gap model"):

* three measured quantities: T0_iss, the issue time of a burst when nothing
  pushes back; R, the effective drain rate of the downstream path; Q, the
  effective pending capacity (bytes that may be outstanding before issue
  stalls);
* the issuer-visible burst issue time, for aggregate burst volume V, K
  producers and useful producer gap G between bursts, is
      T_iss(G; K, V) = max(T0_iss(K, V), V / R - G)
  (the Burst-Gap equation);
* two regimes: drain-dominated when G is short (T_iss = V/R - G) and
  backpressure-free when G drains the previous burst (T_iss = T0_iss).

Units: seconds, bytes and bytes/second (any consistent set works).

The equation does not contain Q. ``t_iss_with_capacity`` and
``fluid_queue_rounds`` are a reading of where Q enters, stated as a
derivation of our own and checked against the equation where the two must
agree: the X-stage is a fluid queue of capacity Q drained at R; the producer
issues at rate V/T0 while the queue has room and at R once it is full; during
the gap nothing is issued and the queue drains. In steady state that gives
      T_iss = max(T0, V/R - min(G, Q/R)),
which is the pages' equation whenever G <= Q/R, and which says that a gap
longer than Q/R cannot hide more than Q bytes of drain. Parity of the local
HBM drain rate against the pages' ~717 GB/s is unpinned: that figure is for
remote stores on an unnamed system.
"""
from __future__ import annotations


def t_iss(G: float, T0: float, V: float, R: float) -> float:
    """The Burst-Gap equation: max(T0, V/R - G)."""
    return max(T0, V / R - G)


def regime(G: float, T0: float, V: float, R: float) -> str:
    """'drain' when V/R - G exceeds T0 (drain-dominated), else 'free'."""
    return "drain" if V / R - G > T0 else "free"


def knee_gap(T0: float, V: float, R: float) -> float:
    """Smallest gap at which the burst issues backpressure-free: V/R - T0 (>= 0)."""
    return max(0.0, V / R - T0)


def t_iss_with_capacity(G: float, T0: float, V: float, R: float, Q: float) -> float:
    """Steady-state issue time of the fluid-queue reading: max(T0, V/R - min(G, Q/R))."""
    return max(T0, V / R - min(G, Q / R))


def single_burst_from_empty(T0: float, V: float, R: float, Q: float) -> float:
    """Issue time of one burst into an empty queue: T0, or (V-Q)/R once V - R*T0 > Q."""
    return max(T0, (V - Q) / R)


def fluid_queue_rounds(V: float, G: float, T0: float, R: float, Q: float, rounds: int):
    """Per-round issue time of a periodic burst/gap producer on a fluid queue.

    Each round: issue V bytes at rate rho = V/T0 while the queue level is
    below Q (it drains at R meanwhile), at rate R once the level reaches Q;
    then compute for G with no issue while the queue drains at R. Returns the
    list of per-round issue times, starting from an empty queue.
    """
    rho = V / T0
    level = 0.0
    out = []
    for _ in range(rounds):
        if rho <= R:
            t = T0  # the drain keeps up with issue: the queue never grows
            level = max(0.0, level + (rho - R) * T0)
        else:
            t_fill = (Q - level) / (rho - R) if level < Q else 0.0
            if rho * t_fill >= V:
                t = T0
                level = level + (rho - R) * T0
            else:
                t = t_fill + (V - rho * t_fill) / R
                level = Q
        out.append(t)
        level = max(0.0, level - R * G)
    return out
