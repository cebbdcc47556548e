"""GPU parity of attn_a2a_fwd_s2s: the Ulysses layer with both exchanges
folded in (sequence-sharded q, k, v partitions in, sequence-sharded output
out) against the float64 oracle, guard bands intact, and bit-identical to
attn_a2a_fwd when every chunk is a whole number of 128-row tiles, or when the
chunks are equal multiples of 64 rows (each tile then loaded as two halves),
also with the split schedule (attn_a2a_fwd_s2s_ex with a workspace), where
both calls run the same pieces."""
import numpy as np
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import workloads
from oracle import attention as orc

from gpu_helpers import GuardedPartitions, compare

pytestmark = pytest.mark.gpu


def seq_shard(t, P):
    """[B, H, S, d] -> P contiguous [B, c_j, H, d] device partitions (test-side data prep)."""
    out, start = [], 0
    for c in bd.chunk_sizes(t.shape[2], P):
        out.append(t[:, :, start:start + c].permute(0, 2, 1, 3).contiguous().cuda())
        start += c
    return out


CASES = [
    ("tiny", 1, 4, 256, 64, 2),
    ("joint_like_c576", 1, 8, 4608, 128, 8),
    ("ragged_c375", 1, 4, 1500, 128, 4),
    ("ragged_c125_d64", 2, 8, 1000, 64, 8),
    ("S_lt_P", 1, 8, 5, 128, 8),
    # equal chunks of 64 (mod 128) rows: tiles loaded as two 64-row halves
    ("halves_c64_P3_tail", 1, 3, 192, 128, 3),
    ("halves_c192_d64_batch2", 2, 4, 384, 64, 2),
    # one partition: the layer is attention in the sequence-major layout
    ("P1_halves_c320", 1, 2, 320, 128, 1),
    ("P1_whole_c256_d64", 1, 2, 256, 64, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_s2s_matches_oracle(case):
    name, B, H, S, d, P = case
    cfg = workloads.CONFIGS[name] if name in workloads.CONFIGS else workloads.AttnConfig(name, B, H, S, d, P)
    q, k, v = workloads.make_qkv(cfg, seed=3)
    g = GuardedPartitions(B, S, H, d, P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd_s2s(seq_shard(q, P), seq_shard(k, P), seq_shard(v, P), P, cfg.scale, g.parts, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert g.guards_intact()
    want = orc.head_to_seq_partitions(orc.attention_fp64(q, k, v, cfg.scale), P)
    for j, (got, w) in enumerate(zip(g.parts, want)):
        compare(orc.as_f64(got), w, f"{name} partition {j}")


EXTRA = {
    "halves_c192_d64": dict(B=2, H=4, S=384, d=64, P=2),
    # whole-tile partitions past S = 16384: row stores, per-partition tiles
    "whole_c8320_rows": dict(B=1, H=2, S=16640, d=128, P=2),
}


@pytest.mark.parametrize("name", ["tiny", "image", "joint", "halves_c192_d64", "whole_c8320_rows"])
def test_s2s_bit_identical_to_fused_on_whole_or_half_tiles(name):
    cfg = workloads.CONFIGS[name] if name in workloads.CONFIGS else workloads.AttnConfig(name, **EXTRA[name])
    q, k, v = workloads.make_qkv(cfg, seed=4)
    a = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    b = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    bd.attn_a2a_fwd(q.cuda(), k.cuda(), v.cuda(), cfg.P, cfg.scale, a)
    bd.attn_a2a_fwd_s2s(seq_shard(q, cfg.P), seq_shard(k, cfg.P), seq_shard(v, cfg.P), cfg.P, cfg.scale, b)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


# The split schedule in the whole layer (attn_a2a_fwd_s2s_ex with a workspace):
# the same pieces, partials and merges as the fused call's with the same
# workspace setting, so the same bytes; and against the oracle.
SPLIT_CASES = [
    ("image", None, bd.SPLIT_AUTO, 0),                                    # automatic: the whole schedule
    ("tail_h8_s8192", dict(B=1, H=8, S=8192, d=128, P=8), bd.SPLIT_TAIL, 0),
    ("all_h8_s8192", dict(B=1, H=8, S=8192, d=128, P=8), bd.SPLIT_ALL, 0),
    ("all_halves_c576", dict(B=1, H=8, S=4608, d=128, P=8), bd.SPLIT_ALL, 0),   # 64-row halves, row stores
    ("tail_d64_grid40", dict(B=2, H=4, S=2048, d=64, P=4), bd.SPLIT_TAIL, 40),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_s2s_split_schedule_same_bytes_as_fused(case):
    name, shape, split, grid = case
    cfg = workloads.CONFIGS[name] if shape is None else workloads.AttnConfig(name, **shape)
    B, H, S, d, P = cfg.B, cfg.H, cfg.S, cfg.d, cfg.P
    q, k, v = workloads.make_qkv(cfg, seed=21)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    ws = bd.alloc_workspace(d, grid)
    g = GuardedPartitions(B, S, H, d, P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd_s2s(seq_shard(q, P), seq_shard(k, P), seq_shard(v, P), P, cfg.scale, g.parts, dev_status=status,
                        workspace=ws, split=split, grid=grid)
    ref = GuardedPartitions(B, S, H, d, P)
    bd.attn_a2a_fwd(dq, dk, dv, P, cfg.scale, ref.parts, dev_status=status, workspace=bd.alloc_workspace(d, grid),
                    split=split, grid=grid)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert g.guards_intact()
    for a, b in zip(g.parts, ref.parts):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    if B * H * S * S <= 8 * 4608 * 4608:  # the oracle where it takes seconds
        want = orc.head_to_seq_partitions(orc.attention_fp64(q, k, v, cfg.scale), P)
        for j, (got, w) in enumerate(zip(g.parts, want)):
            compare(orc.as_f64(got), w, f"{name} partition {j}")
