"""GPU tests of the split schedule (attn_a2a_opts.workspace and .split): work
items' key blocks divided over all CTAs in equal ranges - those of a partial
last wave in a second kernel (SPLIT_TAIL; the automatic choice where that
saves at least 32 key blocks per CTA), or those of every item in one kernel
(SPLIT_ALL) - and partial results merged through the workspace.

* Every row of every split item against the float64 oracle (row by row: each
  output row depends only on its query row), on geometries chosen through the
  grid option so that items are cut in two, three or many pieces, ragged, with
  batch > 1 and d = 64, both store kinds, both split kinds, and on the video
  preset at full size with one CTA per SM (the bench's launch).
* Items that are not cut are untouched: byte-identical to the unsplit call.
* Layout: the fused call with the split equals attention alone with the same
  split followed by the separate permute, byte for byte.
* The workspace is reused: two calls in a row give the same bytes.
"""
import numpy as np
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import workloads
from oracle import attention as orc

from gpu_helpers import REL_FRO, GuardedPartitions, abs_tolerance, rel_fro

pytestmark = pytest.mark.gpu

MIN_SAVED = 32  # key blocks per CTA the automatic tail split must save (the launcher's rule)
MIN_SAVED_ALL = 8  # the same for the whole-schedule split, which needs K and V in half of L2

# (B, H, S, d, P, grid); items = B * H * ceil(ceil(S/128)/2)
CASES = [
    (1, 4, 8192, 128, 4, 24),   # 128 items of 64 blocks: last wave 8 of 24, 22-block ranges
    (1, 2, 8192, 64, 2, 20),    # 64 items: last wave 4 of 20, 13-block ranges
    (2, 3, 5000, 128, 3, 59),   # 120 items of 40 blocks (ragged S): last wave 2 of 59, 2-block ranges
    (1, 3, 8320, 128, 3, 49),   # 99 items of 65 blocks (odd): last wave 1 of 49, one item in 33 pieces
]
# the same over every item in one kernel: 342, 205, 82 and 132-block ranges (the
# grid never exceeds the items, so a range is at least one item long)
CASES_ALL = CASES


def geometry(B, H, S, grid, split=bd.SPLIT_AUTO, d=128):
    """(first split item, pairs per head, items, cut items) as the launcher plans them."""
    nblk = (S + 127) // 128
    npair = (nblk + 1) // 2
    total = B * H * npair
    grid = min(grid, total)
    waves = (total + grid - 1) // grid
    if split == bd.SPLIT_AUTO:
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        all_len = (total * nblk + grid - 1) // grid
        if 2 * 4 * B * H * S * d <= l2 and waves * nblk - all_len >= MIN_SAVED_ALL:
            split = bd.SPLIT_ALL
    if split == bd.SPLIT_ALL:
        length = (total * nblk + grid - 1) // grid
        cut = sorted({u // nblk for u in range(0, total * nblk, length) if u % nblk}
                     | {(u - 1) // nblk for u in range(length, total * nblk, length) if u % nblk})
        return 0, npair, total, cut
    r = total - (waves - 1) * grid
    length = (r * nblk + grid - 1) // grid
    do = r < grid and (split == bd.SPLIT_TAIL or nblk - length >= MIN_SAVED)
    first = (waves - 1) * grid if do else total
    return first, npair, total, list(range(first, total))


def item_rows(item, H, npair, S):
    b, h, pair = item // (H * npair), (item // npair) % H, item % npair
    return b, h, list(range(pair * 256, min(pair * 256 + 256, S)))


def run_fused(q, k, v, cfg, grid, workspace, store_kind, split=bd.SPLIT_AUTO):
    g = GuardedPartitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, g.parts, dev_status=status, grid=grid, workspace=workspace,
                    store_kind=store_kind, split=split)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert g.guards_intact()
    return g


def check_rows(q, k, v, cfg, parts, items, npair):
    bounds = orc.chunk_bounds(cfg.S, cfg.P)
    host = [p.cpu() for p in parts]
    for item in items:
        b, h, rows = item_rows(item, cfg.H, npair, cfg.S)
        if not rows:
            continue
        want = orc.attention_rows_fp64(q, k, v, cfg.scale, b, h, rows)
        got = np.empty_like(want)
        for i, s in enumerate(rows):
            j = next(jj for jj, (st, c) in enumerate(bounds) if st <= s < st + c)
            got[i] = orc.as_f64(host[j][b, s - bounds[j][0], h])
        assert np.all(np.abs(got - want) <= abs_tolerance(want)), f"split item {item}: max|err| {np.abs(got - want).max()}"
        assert rel_fro(got, want) <= REL_FRO, f"split item {item}"


def assert_same_bytes(a_parts, b_parts):
    for a, b in zip(a_parts, b_parts):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def split_and_check(case, store_kind, split):
    B, H, S, d, P, grid = case
    first, npair, total, cut = geometry(B, H, S, grid, split, d)
    assert first < total and cut, "the case must split items"
    cfg = workloads.AttnConfig("split", B=B, H=H, S=S, d=d, P=P)
    q, k, v = workloads.make_qkv(cfg, seed=7)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    ws = bd.alloc_workspace(d, grid)
    g = run_fused(dq, dk, dv, cfg, grid, ws, store_kind, split)
    check_rows(q, k, v, cfg, g.parts, range(first, total), npair)
    # items not cut are the unsplit call's, byte for byte
    plain = run_fused(dq, dk, dv, cfg, grid, None, store_kind)
    bounds = orc.chunk_bounds(S, P)
    for item in sorted(set(range(total)) - set(cut)):
        b, h, rows = item_rows(item, H, npair, S)
        for s in (rows[0], rows[-1]):
            j = next(jj for jj, (st, c) in enumerate(bounds) if st <= s < st + c)
            x, y = g.parts[j][b, s - bounds[j][0], h], plain.parts[j][b, s - bounds[j][0], h]
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), f"item {item}, not cut, changed"
    # the same call again: the workspace keeps the previous call's flags
    assert_same_bytes(g.parts, run_fused(dq, dk, dv, cfg, grid, ws, store_kind, split).parts)
    # attention alone with the same split, then the permute: the same bytes
    o = torch.empty((B, H, S, d), dtype=torch.bfloat16, device="cuda")
    bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o, grid=grid, workspace=ws, store_kind=store_kind, split=split)
    parts = bd.alloc_partitions(B, S, H, d, P)
    bd.attn_a2a_permute(o, P, parts)
    torch.cuda.synchronize()
    assert_same_bytes(g.parts, parts)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}S{}d{}P{}g{}".format(*c))
@pytest.mark.parametrize("store_kind", [1, 2])
def test_split_tail_rows_and_layout(case, store_kind):
    split_and_check(case, store_kind, bd.SPLIT_TAIL)


@pytest.mark.parametrize("case", CASES_ALL, ids=lambda c: "B{}H{}S{}d{}P{}g{}".format(*c))
@pytest.mark.parametrize("store_kind", [1, 2])
def test_split_all_rows_and_layout(case, store_kind):
    split_and_check(case, store_kind, bd.SPLIT_ALL)


@pytest.mark.parametrize("name,split", [("image", bd.SPLIT_ALL), ("image", bd.SPLIT_TAIL), ("joint", bd.SPLIT_ALL)])
def test_short_presets_split_full_size(name, split):
    # one CTA per SM, as the bench launches them: the cut items' rows against the oracle
    cfg = workloads.CONFIGS[name]
    grid = bd.num_sms()
    first, npair, total, cut = geometry(cfg.B, cfg.H, cfg.S, grid, split)
    assert cut
    q, k, v = workloads.make_qkv(cfg, seed=3)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    g = run_fused(dq, dk, dv, cfg, 0, bd.alloc_workspace(cfg.d), 0, split)
    check_rows(q, k, v, cfg, g.parts, cut[:: max(1, len(cut) // 6)], npair)
    plain = run_fused(dq, dk, dv, cfg, 0, None, 0)
    bounds = orc.chunk_bounds(cfg.S, cfg.P)
    for item in sorted(set(range(total)) - set(cut))[::7]:
        b, h, rows = item_rows(item, cfg.H, npair, cfg.S)
        for s in (rows[0], rows[-1]):
            j = next(jj for jj, (st, c) in enumerate(bounds) if st <= s < st + c)
            x, y = g.parts[j][b, s - bounds[j][0], h], plain.parts[j][b, s - bounds[j][0], h]
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), f"item {item}, not cut, changed"


@pytest.mark.slow
def test_video_preset_split_tail_full_size():
    cfg = workloads.CONFIGS["video"]
    grid = bd.num_sms()
    tail_first, npair, total, _ = geometry(cfg.B, cfg.H, cfg.S, grid)
    assert tail_first < total  # 5120 items on 152 SMs: a last wave of 104, 176 of 256 blocks per CTA
    q, k, v = workloads.make_qkv(cfg, seed=0)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    g = run_fused(dq, dk, dv, cfg, 0, bd.alloc_workspace(cfg.d), 0)
    check_rows(q, k, v, cfg, g.parts, range(tail_first, tail_first + 3), npair)
    o = torch.empty((cfg.B, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")
    bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o, workspace=bd.alloc_workspace(cfg.d))
    parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    bd.attn_a2a_permute(o, cfg.P, parts)
    torch.cuda.synchronize()
    assert_same_bytes(g.parts, parts)


def test_automatic_choice_on_the_presets():
    # image: K and V fit in half of L2 and the whole-schedule split saves CTAs 15
    # key blocks, so the automatic choice is SPLIT_ALL (the same bytes); joint: it
    # would save 5, too few, so the call is the unsplit one; SPLIT_NONE with a
    # workspace is the call without one
    for name, want in (("image", bd.SPLIT_ALL), ("joint", 0)):
        cfg = workloads.CONFIGS[name]
        assert bd.attn_a2a_split_plan(cfg.B, cfg.H, cfg.S, cfg.d)[0] == want
        first, _, total, cut = geometry(cfg.B, cfg.H, cfg.S, bd.num_sms(), bd.SPLIT_AUTO, cfg.d)
        assert (first == 0 and cut) if want else first == total
        dq, dk, dv = (t.cuda() for t in workloads.make_qkv(cfg, seed=1))
        a = run_fused(dq, dk, dv, cfg, 0, bd.alloc_workspace(cfg.d), 0)
        b = run_fused(dq, dk, dv, cfg, 0, bd.alloc_workspace(cfg.d), 0, want or bd.SPLIT_NONE)
        assert_same_bytes(a.parts, b.parts)
        c = run_fused(dq, dk, dv, cfg, 0, bd.alloc_workspace(cfg.d), 0, bd.SPLIT_NONE)
        e = run_fused(dq, dk, dv, cfg, 0, None, 0)
        assert_same_bytes(c.parts, e.parts)


def test_workspace_validation():
    cfg = workloads.AttnConfig("split", B=1, H=2, S=512, d=128, P=2)
    dq, dk, dv = (t.cuda() for t in workloads.make_qkv(cfg, seed=0))
    parts = bd.alloc_partitions(1, 512, 2, 128, 2)
    small = torch.zeros(bd.workspace_bytes(4, 128) - 256, dtype=torch.uint8, device="cuda")
    assert bd.attn_a2a_fwd(dq, dk, dv, 2, cfg.scale, parts, grid=4, workspace=small, check=False) == bd.EINVAL
    ws = bd.alloc_workspace(128, 4)
    assert bd.attn_a2a_fwd(dq, dk, dv, 2, cfg.scale, parts, grid=4, workspace=ws[1:], check=False) == bd.EINVAL
    for bad in (-1, 4):
        assert bd.attn_a2a_fwd(dq, dk, dv, 2, cfg.scale, parts, grid=4, workspace=ws, split=bad, check=False) == bd.EINVAL
