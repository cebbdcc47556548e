"""CPU tests of the probe's host-side analysis: stamp reduction, and the fit
of T0, R and Q recovering known parameters from bursts simulated by the
oracle's fluid queue (independent code)."""
import pytest

from attention_all_layout_gb300 import burst_gap as bg
from oracle import burst_gap as obg


def simulated_point(K, V, G, T0, R, Q, rounds=80, discard=40):
    ts = obg.fluid_queue_rounds(V, G, T0, R, Q, rounds)
    # per-producer stamps (ns): all producers identical
    stamps, t = [], 0.0
    rows = []
    for x in ts:
        rows.append([int(t * 1e9), int((t + x) * 1e9), int((t + x + G) * 1e9)])
        t += x + G
    stamps = [rows for _ in range(K)]
    t_iss, period, first = bg.reduce_stamps(stamps, discard=discard)
    return bg.Point(K=K, V=V, G=G, store_kind=0, t_iss=t_iss, period=period, first=first)


def test_reduce_stamps():
    stamps = [[[0, 10, 30], [30, 45, 65]], [[0, 20, 40], [40, 55, 75]]]
    t_iss, period, first = bg.reduce_stamps(stamps, discard=1)
    assert t_iss == pytest.approx([15e-9])
    assert period == pytest.approx([35e-9])
    assert first == pytest.approx(15e-9)


def test_fit_recovers_parameters():
    R, Q = 5e12, 24e6
    pts = []
    for V in (2e6, 8e6, 32e6, 64e6):
        T0 = 1e-6 + V / 40e12
        for G_us in (0, 1, 2, 4, 8, 12, 20, 40):
            pts.append(simulated_point(148, V, G_us * 1e-6, T0, R, Q))
    f = bg.fit(pts)
    assert f.R == pytest.approx(R, rel=2e-3)
    for V in (2e6, 8e6, 32e6, 64e6):
        # the long-gap floor: T0, or (V - Q)/R once one burst overflows the capacity
        floor = obg.single_burst_from_empty(1e-6 + V / 40e12, V, R, Q)
        assert f.t0(148, V, 0) == pytest.approx(floor, rel=1e-3)
    assert f.Q == pytest.approx(Q, rel=0.02)
    res = bg.residuals(f, pts)
    assert max(abs(r) for r in res) < 0.02


def test_predict_matches_equation():
    for G in (0.0, 1e-6, 5e-6, 50e-6):
        assert bg.predict_t_iss(G, 2e-6, 16e6, 717e9) == pytest.approx(obg.t_iss(G, 2e-6, 16e6, 717e9))


def test_calibrate_fma():
    iters = bg.calibrate_fma(lambda n: n * 2.5, target_ns=10000)
    assert iters == 4000
