"""CPU test of the split-tail work decomposition of the attention kernel
(plan_split_tail on the host, tail_piece / piece_at / merge_partials' CTA
range on the device), restated here in Python and checked for the properties
the kernel relies on, over many (items, grid, key blocks) geometries:

* every (item, key block) of the problem is computed exactly once;
* each CTA gets at most two tail pieces, and at most one of them is partial,
  processed first;
* every split item has exactly one final piece (it holds the item's last key
  block), and the CTAs the merge reads from are exactly the ones holding its
  partial pieces - so a final piece only waits on pieces that wait on nothing;
* the CTA ranges balance the tail: no CTA holds more than tail_len blocks;
* the launcher splits only when that saves at least 32 key blocks per CTA
  (the image and joint presets keep the unsplit schedule, video and long split).
"""
import pytest


def plan(total, grid, nblk, min_saved=32):
    waves = (total + grid - 1) // grid
    r = total - (waves - 1) * grid
    if r >= grid or nblk < 2:
        return total, 0
    length = (r * nblk + grid - 1) // grid
    if nblk - length < min_saved:
        return total, 0
    return (waves - 1) * grid, length


def tail_piece(total, tail_first, tail_len, nblk, cta, k):
    R = (total - tail_first) * nblk
    u0 = cta * tail_len
    u1 = min(u0 + tail_len, R)
    if u0 >= u1:
        return None
    i0, i1 = u0 // nblk, (u1 - 1) // nblk
    k0_first = u0 - i0 * nblk
    k1_last = u1 - i1 * nblk
    if k1_last < nblk:
        if k == 0:
            return (tail_first + i1, k0_first if i1 == i0 else 0, k1_last, 1)
        if i1 == i0 or k != 1:
            return None
        return (tail_first + i0, k0_first, nblk, 2 if k0_first > 0 else 0)
    i = i0 + k
    if i > i1:
        return None
    kb = k0_first if i == i0 else 0
    return (tail_first + i, kb, nblk, 2 if kb > 0 else 0)


def pieces(total, grid, nblk, cta, min_saved=0):
    tail_first, tail_len = plan(total, grid, nblk, min_saved)
    main_end = min(tail_first, total)
    out = [(item, 0, nblk, 0) for item in range(cta, main_end, grid)]
    if tail_first < total:
        for k in range(3):
            pc = tail_piece(total, tail_first, tail_len, nblk, cta, k)
            if pc is None:
                break
            out.append(pc)
    return out, tail_first, tail_len


GEOMS = [(total, grid, nblk) for total in (1, 2, 5, 20, 23, 152, 153, 384, 432, 5120)
         for grid in (1, 3, 7, 16, 152) for nblk in (1, 2, 3, 8, 32, 36, 256) if grid <= max(total, 1)]


@pytest.mark.parametrize("total,grid,nblk", GEOMS)
def test_split_tail_plan(total, grid, nblk):
    grid = min(grid, total)
    covered = {}
    per_cta = []
    tail_first = tail_len = None
    for cta in range(grid):
        pcs, tail_first, tail_len = pieces(total, grid, nblk, cta)
        per_cta.append(pcs)
        tail = [pc for pc in pcs if pc[0] >= tail_first]
        assert len(tail) <= 2
        partial = [i for i, pc in enumerate(tail) if pc[3] == 1]
        assert partial in ([], [0])  # a partial piece comes first
        assert sum(pc[2] - pc[1] for pc in tail) <= max(tail_len, nblk if tail_first >= total else tail_len)
        for item, k0, k1, kind in pcs:
            assert 0 <= k0 < k1 <= nblk
            assert (kind == 1) == (k1 < nblk) and (kind == 2) == (k1 == nblk and k0 > 0)
            for j in range(k0, k1):
                assert (item, j) not in covered
                covered[(item, j)] = cta
    assert len(covered) == total * nblk
    if tail_first < total:
        assert 1 <= tail_len <= nblk
        for item in range(tail_first, total):
            finals = [(c, pc) for c, pcs in enumerate(per_cta) for pc in pcs if pc[0] == item and pc[2] == nblk]
            assert len(finals) == 1
            c, (_, kb, _, kind) = finals[0]
            holders = sorted({covered[(item, j)] for j in range(kb)})
            if kind == 2:
                U = (item - tail_first) * nblk
                assert holders == list(range(U // tail_len, c))  # merge_partials' CTA range
                for h in holders:  # each holds exactly one partial piece: of this item
                    assert [pc for pc in per_cta[h] if pc[3] == 1] == [pc for pc in per_cta[h] if pc[0] == item]
            else:
                assert holders in ([], [c])


def test_tail_shapes_of_the_presets():
    # image: 384 items of 32 key blocks on 152 CTAs -> a last wave of 80 items; 17-block
    # ranges would save only 15 blocks per CTA, so the tail is not split
    assert plan(384, 152, 32, min_saved=0) == (304, 17)
    assert plan(384, 152, 32) == (384, 0)
    # joint: 432 items of 36 blocks -> 128 in the last wave, 31-block ranges: not split
    assert plan(432, 152, 36) == (432, 0)
    # video: 5120 items of 256 blocks -> 104 in the last wave, 176-block ranges (80 saved)
    assert plan(5120, 152, 256) == (5016, 176)
    # long: 11840 items of 591 blocks -> 136 in the last wave, 529-block ranges (62 saved)
    assert plan(11840, 152, 591) == (11704, 529)
    # a full last wave is not split
    assert plan(304, 152, 32) == (304, 0)
