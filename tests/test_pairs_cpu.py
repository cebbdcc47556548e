"""CPU test of the CTA-pair kernel's work decomposition (attn_a2a_opts.cta_pairs
= 1), restated here in Python from the kernel's piece_at / decode_item and the
launcher's grid rule, and checked for what the kernel relies on, over many
(B, H, S, grid) geometries:

* every (b, h, query-tile pair) of the problem is run exactly once, by one CTA
  of one cluster; the two CTAs of a cluster always run the same unit (b, h,
  quad) at the same step, so the leader's MMAs combine rows of one head and
  each CTA's half of the same key blocks;
* a CTA whose pair index lies past the head's last pair (an odd number of
  pairs per head) only ever gets rows at or beyond S, which the loads read as
  zeros and the epilogue never stores;
* the grid: an even number of CTAs, at most twice the resident clusters and
  twice the units, at least one cluster.

And the shared-memory budget of the pair configuration, restated from Cfg:
eight half-tile K/V stages take the bytes of four whole ones, so the barrier
block, the staging buffer and the alignment slack fit in 227 KB as before.
"""
import itertools

import pytest


def units(B, H, S):
    nblk = (S + 127) // 128
    npair = (nblk + 1) // 2
    nquad = (npair + 1) // 2
    return nblk, npair, nquad, B * H * nquad


def pair_grid(want, resident, total):
    """The launcher: clusters = min(want // 2, resident, total); grid = 2 * clusters."""
    clusters = min(want // 2, resident, total)
    return 2 * clusters if clusters >= 1 else 0


def decode(item, rank, nquad, H):
    quad = item % nquad
    bh = item // nquad
    return bh // H, bh % H, 2 * quad + rank


def schedule(B, H, S, grid):
    """{(b, h, pair): (cta, step)} and the per-step unit of every cluster."""
    _, npair, nquad, total = units(B, H, S)
    n = grid // 2
    ran, cluster_units = {}, {}
    for cta in range(grid):
        rank, c = cta % 2, cta // 2
        it = 0
        while True:
            item = c + it * n
            if item >= total:
                break
            b, h, pair = decode(item, rank, nquad, H)
            cluster_units.setdefault((c, it), set()).add((b, h, item % nquad))
            key = (b, h, pair)
            assert key not in ran, f"pair {key} run twice"
            ran[key] = (cta, it)
            it += 1
    return ran, cluster_units, npair


GEOMS = list(itertools.product([1, 2, 3], [1, 2, 5, 24], [128, 640, 1000, 2304, 4096, 4608], [2, 8, 14, 152]))


@pytest.mark.parametrize("B,H,S,grid", GEOMS)
def test_every_pair_run_once_and_clusters_stay_together(B, H, S, grid):
    nblk, npair, nquad, total = units(B, H, S)
    g = pair_grid(grid, 76, total)
    assert g % 2 == 0 and 2 <= g <= min(grid, 152, 2 * total)
    ran, cluster_units, _ = schedule(B, H, S, g)
    # every real pair exactly once
    for b in range(B):
        for h in range(H):
            for pair in range(npair):
                assert (b, h, pair) in ran
    # anything else run lies wholly past S
    for (b, h, pair) in ran:
        if pair >= npair:
            assert 2 * pair * 128 >= S and pair == npair and npair % 2 == 1
    # both CTAs of a cluster run one and the same unit at every step
    for units_at_step in cluster_units.values():
        assert len(units_at_step) == 1


def test_odd_pairs_leave_the_last_units_second_half_past_s():
    # S = 640: 5 query tiles, 3 pairs per head, 2 units; unit 1's rank 1 gets pair 3
    nblk, npair, nquad, total = units(1, 1, 640)
    assert (nblk, npair, nquad, total) == (5, 3, 2, 2)
    assert decode(1, 1, nquad, 1) == (0, 0, 3)
    assert 2 * 3 * 128 >= 640


def test_grid_rule():
    assert pair_grid(152, 76, 1000) == 152
    assert pair_grid(153, 76, 1000) == 152   # odd: cut to even
    assert pair_grid(152, 72, 1000) == 144   # fewer clusters resident
    assert pair_grid(152, 76, 3) == 6        # fewer units than clusters
    assert pair_grid(1, 76, 10) == 0         # no whole cluster: refused


def test_shared_memory_budget_of_the_pair_configuration():
    tile = 128 * 128 * 2
    for pair in (False, True):
        kv = tile // 2 if pair else tile
        nstage = 8 if pair else 4
        kv_off = 2 * tile
        bar_off = kv_off + nstage * kv
        nbar = 10 + 2 * nstage + 1 + 1 + 2 + 3  # QF..OE, KVF, KVE, DONE, STG, STGW, EVA..EVC
        used = bar_off + nbar * 8 + 16
        stg_off = (used + 1023) // 1024 * 1024
        assert nstage * kv == 4 * tile
        assert stg_off + tile + 1024 <= 227 * 1024
