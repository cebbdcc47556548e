"""GPU tests of the Burst-Gap probe: the kernel's stamps are consistent
(ordered, gaps honoured, both store kinds), a long gap brings the issue
time down to its floor while no gap leaves a large burst drain-dominated,
and the equation fitted on part of a small sweep predicts the rest."""
import statistics

import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import burst_gap as bg
from attention_all_layout_gb300 import probe_sweep as ps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prober():
    K = bd.num_sms()
    dst_bytes = (max(4 * ps.l2_bytes(), 4 * 256 * 2**20) // (4096 * K) + 1) * 4096 * K
    return ps.Prober(dst_bytes, K * 64 * 3), K


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_stamps_are_ordered_and_gaps_honoured(prober, kind):
    pr, K = prober
    V = ps.round_volume(8 * 2**20, K)
    G_ns = 5000
    rounds = 16
    st = pr.stamps[: K * rounds * 3]
    st.zero_()
    bd.xstage_probe_run(K, rounds, V, G_ns, pr.dst, st, store_kind=kind)
    torch.cuda.synchronize()
    s = st.view(K, rounds, 3).cpu()
    assert torch.all(s[:, :, 1] >= s[:, :, 0])
    assert torch.all(s[:, :, 2] - s[:, :, 1] >= G_ns)
    assert torch.all(s[:, 1:, 0] >= s[:, :-1, 2])


def test_fma_gap_kind_runs(prober):
    pr, K = prober
    p_short = pr.run(K, ps.round_volume(2**20, K), 0, 8, gap_kind=1, fma_iters=100)
    p_long = pr.run(K, ps.round_volume(2**20, K), 0, 8, gap_kind=1, fma_iters=20000)
    assert statistics.median(p_long.period) > statistics.median(p_short.period)


@pytest.mark.parametrize("kind", [0, 1])
def test_regimes_and_heldout_fit(prober, kind):
    """The equation, fitted on part of a small sweep, predicts the held-out
    points within 15 % (median |relative error| of the issue time), for
    bursts L2 can absorb (4-64 MB) and a burst twice the L2 size (256 MB)."""
    pr, K = prober
    pts = []
    grid = [(vmb, g, 48) for vmb in (4, 32, 64) for g in (0, 2, 5, 10, 20, 40)]
    grid += [(256, g, 16) for g in (0, 10, 20, 40, 80, 120)]
    for vmb, g, rounds in grid:
        pts.append(pr.run(K, ps.round_volume(vmb * 2**20, K), g * 1000, rounds, store_kind=kind))
    V64 = ps.round_volume(64 * 2**20, K)
    big0 = next(p for p in pts if p.V == V64 and p.G == 0)
    big40 = next(p for p in pts if p.V == V64 and p.G == 40e-6)
    assert big0.t_iss_med >= big40.t_iss_med
    f, held = ps.split_fit(pts, seed=1, g_max=120e-6)
    assert f.R > 0
    print(f"probe fit kind {kind}: R = {f.R / 1e9:.0f} GB/s, Q = {f.Q}, held-out {held}")
    assert held["n"] >= 5
    assert held["median_abs_rel"] <= 0.15


@pytest.mark.parametrize("kind", [0, 1])
def test_mma_gap_kind(prober, kind):
    """Tensor-core work as the gap: stamps stay ordered, more MMAs make a longer
    gap, and a drain-dominated burst stalls the MMA pipe longer with no work
    behind it than with a long MMA gap."""
    pr, K = prober
    V = ps.round_volume(64 * 2**20, K)
    short = pr.run(K, V, 0, 24, store_kind=kind, gap_kind=2, fma_iters=0)
    long = pr.run(K, V, 0, 24, store_kind=kind, gap_kind=2, fma_iters=2000)
    assert ps.measured_gap(long) > ps.measured_gap(short)
    assert short.t_iss_med >= long.t_iss_med
    st = pr.stamps[: K * 8 * 3]
    bd.xstage_probe_run(K, 8, V, 0, pr.dst, st, store_kind=kind, gap_kind=2, fma_iters=500)
    torch.cuda.synchronize()
    s = st.view(K, 8, 3).cpu()
    assert torch.all(s[:, :, 1] >= s[:, :, 0]) and torch.all(s[:, :, 2] >= s[:, :, 1])


@pytest.fixture(scope="module")
def host_prober():
    K = bd.num_sms()
    dst_bytes = (4 * 64 * 2**20 // (4096 * K) + 1) * 4096 * K
    return ps.Prober(dst_bytes, K * 16 * 3, host=True), K


@pytest.mark.parametrize("kind", [0, 2])
def test_host_destination_fit(host_prober, kind):
    """Bursts into pinned host memory, drained over the host link: a large
    burst with no gap is drain-dominated, a long gap brings the issue time to
    its floor, and the equation fitted on part of the sweep predicts the
    held-out points within 15 %."""
    pr, K = host_prober
    pts = []
    for vmb in (4, 16, 64):
        for g in (0, 10, 40, 100, 400):
            pts.append(pr.run(K, ps.round_volume(vmb * 2**20, K), g * 1000, 16, store_kind=kind, discard=8))
    V64 = ps.round_volume(64 * 2**20, K)
    p0 = next(p for p in pts if p.V == V64 and p.G == 0)
    p400 = next(p for p in pts if p.V == V64 and p.G == 400e-6)
    assert p0.t_iss_med > 5 * p400.t_iss_med
    f, held = ps.split_fit(pts, seed=2, g_max=400e-6)
    print(f"host destination, kind {kind}: R = {f.R / 1e9:.0f} GB/s, Q = {f.Q}, held-out {held}")
    assert held["n"] >= 3
    assert held["median_abs_rel"] <= 0.15
