"""CPU test of the split work decomposition of the attention kernel
(plan_split_tail on the host, tail_piece / piece_at / merge_partials' range of
ranges on the device), restated here in Python and checked for the properties
the kernel relies on, over many (items, grid, key blocks) geometries and both
split kinds (the last wave in a tail kernel; every item in one kernel):

* every (item, key block) of the problem is computed exactly once;
* a range holds at most tail_len blocks, at most one partial piece (its first)
  and at most one final piece (its last);
* every split item has exactly one final piece, the one holding its first key
  block; the ranges its merge reads are exactly those holding the item's other
  blocks, each of which holds exactly one partial piece, of this item, and
  runs on a CTA of lower index than the final piece's - so a final piece waits
  only on pieces that wait on nothing, on CTAs dispatched no later;
* the automatic choice takes the whole-schedule split where the K and V of
  every head fit in half of L2 and it saves at least 8 key blocks per CTA (the
  image preset), else the last wave's split where that saves at least 32 key
  blocks per CTA (video and long); joint stays unsplit.
"""
import pytest

AUTO, TAIL, ALL, NONE = 0, 1, 2, 3


L2 = 126 * 2**20  # an L2 of GB300 size, for the automatic choice


def plan(total, grid, nblk, split=AUTO, min_saved=32, kv_bytes=1 << 40, l2=L2):
    """(tail_first, tail_len, whole) as the host launcher computes them; kv_bytes =
    the K and V bytes of every head (4 * B * H * S * d)."""
    if split == NONE or nblk < 2:
        return total, 0, False
    waves = (total + grid - 1) // grid
    all_len = (total * nblk + grid - 1) // grid
    if split == ALL or (split == AUTO and 2 * kv_bytes <= l2 and waves * nblk - all_len >= 8):
        return 0, all_len, True
    r = total - (waves - 1) * grid
    if r >= grid:
        return total, 0, False
    length = (r * nblk + grid - 1) // grid
    if split == AUTO and nblk - length < min_saved:
        return total, 0, False
    return (waves - 1) * grid, length, False


def tail_piece(total, tail_first, tail_len, nblk, grid, cta, k):
    """Piece k of CTA cta's range (range g = grid - 1 - cta), or None."""
    g = grid - 1 - cta
    R = (total - tail_first) * nblk
    u0 = g * tail_len
    u1 = min(u0 + tail_len, R)
    if u0 >= u1:
        return None
    i0 = u0 // nblk
    i = i0 + k
    if i > (u1 - 1) // nblk:
        return None
    k0 = u0 - i0 * nblk if k == 0 else 0
    k1 = min(u1 - i * nblk, nblk)
    kind = 1 if k0 > 0 else (2 if k1 < nblk else 0)
    return (tail_first + i, k0, k1, kind)


def merge_ranges(item, tail_first, tail_len, nblk, grid, cta):
    """The ranges merge_partials reads for the final piece of `item` on CTA cta."""
    g = grid - 1 - cta
    g_last = ((item - tail_first) * nblk + nblk - 1) // tail_len
    return list(range(g + 1, g_last + 1))


def schedule(total, grid, nblk, split):
    tail_first, tail_len, whole = plan(total, grid, nblk, split)
    per_cta = []
    for cta in range(grid):
        out = [] if whole else [(item, 0, nblk, 0) for item in range(cta, min(tail_first, total), grid)]
        split_pcs = []
        if tail_first < total:
            k = 0
            while (pc := tail_piece(total, tail_first, tail_len, nblk, grid, cta, k)) is not None:
                split_pcs.append(pc)
                k += 1
        per_cta.append((out, split_pcs))
    return tail_first, tail_len, whole, per_cta


GEOMS = [(total, grid, nblk) for total in (1, 2, 5, 20, 23, 152, 153, 384, 432, 5120)
         for grid in (1, 3, 7, 16, 152) for nblk in (1, 2, 3, 8, 32, 36, 256) if grid <= max(total, 1)]


@pytest.mark.parametrize("split", [TAIL, ALL])
@pytest.mark.parametrize("total,grid,nblk", GEOMS)
def test_split_plan(total, grid, nblk, split):
    grid = min(grid, total)
    tail_first, tail_len, whole, per_cta = schedule(total, grid, nblk, split)
    covered = {}
    for cta, (plain, pcs) in enumerate(per_cta):
        if pcs:
            assert sum(k1 - k0 for _, k0, k1, _ in pcs) <= tail_len
        kinds = [pc[3] for pc in pcs]
        assert kinds.count(1) <= 1 and (1 not in kinds or kinds[0] == 1)  # a partial piece comes first
        assert kinds.count(2) <= 1 and (2 not in kinds or kinds[-1] == 2)  # a final piece comes last
        for item, k0, k1, kind in plain + pcs:
            assert 0 <= k0 < k1 <= nblk
            assert (kind == 1) == (k0 > 0) and (kind == 2) == (k0 == 0 and k1 < nblk)
            for j in range(k0, k1):
                assert (item, j) not in covered
                covered[(item, j)] = cta
    assert len(covered) == total * nblk
    if tail_first >= total:
        return
    assert tail_len >= 1 and (whole or tail_len <= nblk)
    for item in range(tail_first, total):
        holders = {covered[(item, j)] for j in range(nblk)}
        finals = [(c, pc) for c, (_, pcs) in enumerate(per_cta) for pc in pcs if pc[0] == item and pc[3] == 2]
        if len(holders) == 1:
            assert finals == []  # a whole item
            continue
        assert len(finals) == 1
        c, (_, k0, k1, _) = finals[0]
        assert k0 == 0
        others = sorted({covered[(item, j)] for j in range(k1, nblk)})
        read = [grid - 1 - g for g in merge_ranges(item, tail_first, tail_len, nblk, grid, c)]
        assert sorted(read) == others
        for h in others:
            assert h < c  # dispatched no later than the waiting CTA
            assert [pc for pc in per_cta[h][1] if pc[3] == 1] == [pc for pc in per_cta[h][1] if pc[0] == item]


def kv(B, H, S, d):
    return 4 * B * H * S * d


def test_split_shapes_of_the_presets():
    # image: 384 items of 32 key blocks on 152 CTAs -> a last wave of 80 items; 17-block
    # tail ranges would save only 15 blocks per CTA, the whole schedule in 81-block
    # ranges saves 15 of 96, and K and V (50 MB) fit in half of L2: the whole schedule
    image = kv(1, 24, 4096, 128)
    assert plan(384, 152, 32, TAIL) == (304, 17, False)
    assert plan(384, 152, 32, kv_bytes=image) == (0, 81, True)
    assert plan(384, 152, 32, ALL) == (0, 81, True)
    assert plan(384, 152, 32, kv_bytes=image, l2=64 * 2**20) == (384, 0, False)  # a smaller L2: no split
    # joint: 432 items of 36 blocks -> 128 in the last wave; 103-block ranges would save
    # 5 of 108, fewer than the 8 the automatic choice asks for: not split
    assert plan(432, 152, 36, kv_bytes=kv(1, 24, 4608, 128)) == (432, 0, False)
    assert plan(432, 152, 36, ALL) == (0, 103, True)
    # video: 5120 items of 256 blocks -> 104 in the last wave, 176-block ranges (80 saved);
    # K and V (671 MB) far beyond L2
    assert plan(5120, 152, 256, kv_bytes=kv(1, 40, 32768, 128)) == (5016, 176, False)
    # long: 11840 items of 591 blocks -> 136 in the last wave, 529-block ranges (62 saved)
    assert plan(11840, 152, 591, kv_bytes=kv(1, 40, 75600, 128)) == (11704, 529, False)
    # a full last wave is not split by the tail kinds
    assert plan(304, 152, 32) == (304, 0, False)
    assert plan(304, 152, 32, TAIL) == (304, 0, False)
    assert plan(304, 152, 32, NONE) == (304, 0, False)


# The library's own decision (attn_a2a_split_plan, host-only) against the
# restatement above, for whole problems (B x H heads of length S) on a GPU of
# 152 SMs and a GB300-sized L2.
PROBLEMS = [(1, 24, 4096), (1, 24, 4608), (1, 40, 32768), (1, 40, 75600), (1, 40, 4096), (2, 3, 5000),
            (1, 4, 8192), (1, 2, 8192), (1, 3, 8320), (1, 1, 256), (3, 7, 1000), (1, 8, 16384)]


@pytest.mark.parametrize("B,H,S", PROBLEMS)
@pytest.mark.parametrize("grid", [0, 24, 100])
@pytest.mark.parametrize("split", [AUTO, TAIL, ALL, NONE])
def test_library_plan_matches_restatement(B, H, S, grid, split):
    bd = pytest.importorskip("attention_all_layout_gb300.binding")
    try:
        bd.load()
    except Exception as e:  # the library must have been built for this test
        pytest.skip(f"library not loadable: {e}")
    d, n_sm = 128, 152
    nblk = (S + 127) // 128
    total = B * H * ((nblk + 1) // 2)
    g = min(grid or n_sm, total)
    first, length, whole = plan(total, g, nblk, split, kv_bytes=kv(B, H, S, d), l2=L2)
    kind, c_first, c_len = bd.attn_a2a_split_plan(B, H, S, d, grid, split, num_sms=n_sm, l2_bytes=L2)
    want_kind = 0 if first >= total else (ALL if whole else TAIL)
    assert (kind, c_first if kind else total, c_len) == (want_kind, first, length)
