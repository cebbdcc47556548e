"""CPU model check of the bulk-store epilogue's staging-buffer protocol (the
kernel's store_role and softmax_role: owners of query tile t stage their tile
into the one staging buffer and arrive on STGW + t; warp 3 waits for that,
reads the buffer - the tensor stores' shared-memory reads - and releases it).

mbarrier parity waits are modelled exactly: a barrier of arrival count 1 has
completed `n` phases after `n` arrivals, and a wait for phase k with parity
k & 1 returns as soon as the current phase's parity differs from k & 1 - so a
waiter that is two phases ahead is let through. Every interleaving of the
three actors (tile 0's owners, tile 1's owners, warp 3) over a few work items
is explored:

* with a release barrier per tile (STG + t; tile 1 waits for tile 0's release
  of the same item, tile 0 for tile 1's of the previous one) no owner ever
  stages while warp 3 is reading another use, and every interleaving ends with
  all uses stored, none stuck;
* with one release barrier for both tiles, waited on for "use u - 1", some
  interleaving lets tile 0 overwrite a buffer warp 3 is still reading - the
  race this layout removes (owners of use u + 2 waiting for phase u + 1 while
  their own use u was still unreleased).
"""
import functools

import pytest

ITEMS = 4


def parity_done(completed: int, phase: int) -> bool:
    """mbarrier.try_wait.parity for `phase` when `completed` phases have completed."""
    return (completed & 1) != (phase & 1)


def explore(per_tile: bool, items: int = ITEMS):
    """Returns (corrupted, deadlocked, finished) over all interleavings."""
    uses = [(it, t) for it in range(items) for t in (0, 1)]
    found = {"corrupt": False, "dead": False, "done": False}

    # state: next use index per owner tile, warp 3's next use and phase ("wait"
    # or "read"), buffer content, completed phases of STG (one or per tile) and
    # of STGW per tile
    @functools.lru_cache(maxsize=None)
    def step(o0, o1, w_use, w_reading, buf, stg, stgw):
        if w_use == len(uses) and o0 == items and o1 == items:
            found["done"] = True
            return
        moves = []
        # owners of tile t at item `it` (= their next use)
        for t, it in ((0, o0), (1, o1)):
            if it >= items:
                continue
            if per_tile:
                ok = (it == 0 or parity_done(stg[1], it - 1)) if t == 0 else parity_done(stg[0], it)
            else:
                u = 2 * it + t
                ok = u == 0 or parity_done(stg[0], u - 1)
            if ok:
                if w_reading and buf != (it, t):
                    found["corrupt"] = True  # stages over a use warp 3 is reading
                nstgw = list(stgw)
                nstgw[t] += 1
                no = (it + 1, o1) if t == 0 else (o0, it + 1)
                moves.append((no[0], no[1], w_use, w_reading, (it, t), stg, tuple(nstgw)))
        # warp 3
        if w_use < len(uses):
            it, t = uses[w_use]
            if not w_reading:
                if parity_done(stgw[t], it):  # the owners of (it, t) have staged
                    if buf != (it, t):
                        found["corrupt"] = True  # reads another use's rows
                    moves.append((o0, o1, w_use, True, buf, stg, stgw))
            else:
                nstg = list(stg)
                nstg[t if per_tile else 0] += 1
                moves.append((o0, o1, w_use + 1, False, buf, tuple(nstg), stgw))
        if not moves:
            found["dead"] = True
            return
        for m in moves:
            step(*m)

    step(0, 0, 0, False, None, (0, 0), (0, 0))
    return found["corrupt"], found["dead"], found["done"]


def test_parity_model():
    # a fresh barrier: phase 0 not complete; after one arrival it is
    assert not parity_done(0, 0)
    assert parity_done(1, 0)
    # two phases ahead aliases: waiting for phase 2 after one completed phase
    assert parity_done(1, 2)


@pytest.mark.parametrize("items", [1, 2, 3, ITEMS])
def test_per_tile_release_tokens_are_exact(items):
    corrupt, dead, done = explore(per_tile=True, items=items)
    assert not corrupt
    assert not dead
    assert done


def test_one_token_for_both_tiles_can_alias():
    corrupt, _, _ = explore(per_tile=False, items=3)
    assert corrupt
