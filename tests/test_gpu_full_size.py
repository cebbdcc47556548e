"""Full-size parity at the video (S=32768) and long ragged (S=75600) presets,
in the launch configuration the benchmark times.

The whole output is too large for the float64 oracle, but every output row
depends only on its own query row, so the oracle computes exact rows for a
stratified sample on every head: the first and last two rows of every
sequence chunk, every row of the query blocks that straddle a chunk boundary
or end the sequence, and 256 seeded random rows. Layout is checked in full:
the fused partitions equal attention-then-permute byte for byte, and the
guard bands around every partition are untouched."""
import numpy as np
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import workloads
from oracle import attention as orc

from gpu_helpers import REL_FRO, GuardedPartitions, abs_tolerance, rel_fro

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def sample_rows(S, P, seed):
    bounds = orc.chunk_bounds(S, P)
    rows = set()
    for start, c in bounds:
        rows.update(r for r in (start, start + 1, start + c - 2, start + c - 1) if 0 <= r < S)
    blocks = set()
    for start, _ in bounds[1:]:
        if start % 128:
            blocks.add(start // 128)
    if S % 128:
        blocks.add(S // 128)
    for m in blocks:
        rows.update(range(m * 128, min(S, m * 128 + 128)))
    gen = torch.Generator().manual_seed(seed)
    rows.update(torch.randint(0, S, (256,), generator=gen).tolist())
    return sorted(rows), sorted(blocks)


@pytest.mark.parametrize("name", ["video", "long"])
def test_full_size_sampled_rows_and_layout(name):
    cfg = workloads.CONFIGS[name]
    q, k, v = workloads.make_qkv(cfg, seed=0)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    g = GuardedPartitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd(dq, dk, dv, cfg.P, cfg.scale, g.parts, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert g.guards_intact()

    # layout: bit-exact against attention alone followed by the separate permute
    o = torch.empty((cfg.B, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")
    bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o)
    serial = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    bd.attn_a2a_permute(o, cfg.P, serial)
    torch.cuda.synchronize()
    for a, b in zip(g.parts, serial):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    del o, serial

    rows, blocks = sample_rows(cfg.S, cfg.P, seed=7)
    if name == "long":
        assert len(blocks) == 8  # seven chunk-straddling blocks and the 80-row last block
    bounds = orc.chunk_bounds(cfg.S, cfg.P)
    host_parts = [p.cpu() for p in g.parts]
    worst_abs, worst_rf = 0.0, 0.0
    for h in range(cfg.H):
        want = orc.attention_rows_fp64(q, k, v, cfg.scale, 0, h, rows)
        got = np.empty_like(want)
        for i, s in enumerate(rows):
            j = next(jj for jj, (st, c) in enumerate(bounds) if st <= s < st + c)
            got[i] = orc.as_f64(host_parts[j][0, s - bounds[j][0], h])
        err = float(np.abs(got - want).max())
        rf = rel_fro(got, want)
        worst_abs, worst_rf = max(worst_abs, err), max(worst_rf, rf)
        assert np.all(np.abs(got - want) <= abs_tolerance(want)), f"{name} head {h}: max|err| {err:.3e}"
        assert rf <= REL_FRO, f"{name} head {h}: rel-Frobenius {rf:.3e}"
    print(f"{name}: {len(rows)} rows x {cfg.H} heads, max|err| {worst_abs:.3e}, worst rel-Fro {worst_rf:.3e}")


def _seq_shards(t, P):
    """[B, H, S, d] device tensor -> P contiguous [B, c_j, H, d] partitions (test-side data prep)."""
    out, start = [], 0
    for c in bd.chunk_sizes(t.shape[2], P):
        out.append(t[:, :, start:start + c].permute(0, 2, 1, 3).contiguous())
        start += c
    return out


@pytest.mark.parametrize("name", ["video", "long"])
def test_full_size_whole_layer(name):
    # the whole Ulysses layer (sequence-sharded q, k, v in) at full size: the
    # video preset's whole-tile partitions give the fused call's bytes; the
    # long preset's ragged partitions (9450 rows) are tiled per partition, so
    # they are checked against the oracle on sampled rows of a few heads
    cfg = workloads.CONFIGS[name]
    q, k, v = workloads.make_qkv(cfg, seed=0)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    g = GuardedPartitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd_s2s(_seq_shards(dq, cfg.P), _seq_shards(dk, cfg.P), _seq_shards(dv, cfg.P), cfg.P, cfg.scale,
                        g.parts, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert g.guards_intact()
    if name == "video":
        ref = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
        bd.attn_a2a_fwd(dq, dk, dv, cfg.P, cfg.scale, ref)
        torch.cuda.synchronize()
        for a, b in zip(g.parts, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        return
    rows, _ = sample_rows(cfg.S, cfg.P, seed=8)
    bounds = orc.chunk_bounds(cfg.S, cfg.P)
    host_parts = [p.cpu() for p in g.parts]
    for h in (0, 17, cfg.H - 1):
        want = orc.attention_rows_fp64(q, k, v, cfg.scale, 0, h, rows)
        got = np.empty_like(want)
        for i, s in enumerate(rows):
            j = next(jj for jj, (st, c) in enumerate(bounds) if st <= s < st + c)
            got[i] = orc.as_f64(host_parts[j][0, s - bounds[j][0], h])
        assert np.all(np.abs(got - want) <= abs_tolerance(want)), f"{name} head {h}"
        assert rel_fro(got, want) <= REL_FRO, f"{name} head {h}"
