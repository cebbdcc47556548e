"""Pins for the Burst-Gap oracle.

The equation is checked against an independent mechanism (a fluid-queue
simulation of the X-stage, whose steady state must reproduce it when the gap
fits in the capacity), at the pages' own drain rate, and against its two
regimes and the knee where they meet. The simulation itself is pinned by
cases solved by hand.
"""
import json
import os

import pytest

from oracle import burst_gap as bg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def pages_R():
    figs = json.load(open(GOLDEN))["figures"]
    return next(f["value"] for f in figs if f["name"] == "drain_rate_R")


def test_pages_drain_rate_units():
    R = pages_R()
    assert R == 717e9
    # 7.17 MB drains in exactly 10 us at 717 GB/s
    assert bg.t_iss(0.0, 1e-6, 7.17e6, R) == pytest.approx(10e-6, rel=1e-12)


@pytest.mark.parametrize("V", [1e6, 4e6, 16e6, 64e6])
@pytest.mark.parametrize("G_us", [0, 0.5, 2, 4, 8, 12, 20])
def test_fluid_queue_steady_state_equals_equation(V, G_us):
    R = pages_R()
    T0 = 2e-6 + V / 4e12  # an issue rate above R, so bursts can back up
    G = G_us * 1e-6
    Q = max(V, R * G) * 1.5  # capacity large enough that the gap fits: G <= Q/R
    rounds = bg.fluid_queue_rounds(V, G, T0, R, Q, 400)
    assert rounds[-1] == pytest.approx(bg.t_iss(G, T0, V, R), rel=1e-9)
    assert rounds[-1] == pytest.approx(rounds[-2], rel=1e-12)


@pytest.mark.parametrize("G_us", [0, 1, 5, 50])
def test_fluid_queue_capacity_reading(G_us):
    R, V, T0, Q = 717e9, 32e6, 5e-6, 4e6
    G = G_us * 1e-6
    rounds = bg.fluid_queue_rounds(V, G, T0, R, Q, 400)
    assert rounds[-1] == pytest.approx(bg.t_iss_with_capacity(G, T0, V, R, Q), rel=1e-9)


def test_single_burst_by_hand():
    # rho = V/T0 = 4e12 B/s, R = 1e12 B/s, Q = 3e6 B, V = 8e6 B, T0 = 2 us.
    # fill: Q/(rho-R) = 1 us, issuing 4e6 B; the remaining 4e6 B go at R: 4 us.
    t = bg.fluid_queue_rounds(8e6, 1.0, 2e-6, 1e12, 3e6, 1)[0]
    assert t == pytest.approx(5e-6, rel=1e-12)
    assert bg.single_burst_from_empty(2e-6, 8e6, 1e12, 3e6) == pytest.approx(5e-6, rel=1e-12)
    # the same burst with room for it: never stalls
    assert bg.fluid_queue_rounds(8e6, 1.0, 2e-6, 1e12, 7e6, 1)[0] == pytest.approx(2e-6)


def test_issue_slower_than_drain_never_stalls():
    assert bg.fluid_queue_rounds(1e6, 0.0, 10e-6, 1e12, 1.0, 50)[-1] == pytest.approx(10e-6)


def test_regimes_and_knee():
    R, V, T0 = 717e9, 16e6, 3e-6
    knee = bg.knee_gap(T0, V, R)
    assert knee == pytest.approx(V / R - T0)
    assert bg.regime(0.0, T0, V, R) == "drain"
    assert bg.regime(knee * 0.99, T0, V, R) == "drain"
    assert bg.regime(knee * 1.01, T0, V, R) == "free"
    assert bg.t_iss(knee, T0, V, R) == pytest.approx(T0)
    assert bg.t_iss(0.0, T0, V, R) == pytest.approx(V / R)
    assert bg.t_iss(1.0, T0, V, R) == T0
    prev = float("inf")
    for i in range(200):  # non-increasing in G
        cur = bg.t_iss(i * 0.2e-6, T0, V, R)
        assert cur <= prev + 1e-18
        prev = cur
    assert bg.knee_gap(T0, 1e3, R) == 0.0
