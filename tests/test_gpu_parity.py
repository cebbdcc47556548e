"""GPU parity: the fused tcgen05 kernel (through the C ABI) against the
float64 oracle, the partition layout bit-exact against attention-then-permute
on the GPU, guard bands intact, ragged and degenerate shapes, strided
inputs, the host-memory entry point, and the bounded-wait failure path."""
import math

import numpy as np
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import workloads
from oracle import attention as orc

from gpu_helpers import GuardedPartitions, compare, fused, partitions_to_bhsd

pytestmark = pytest.mark.gpu


def cuda_qkv(cfg, seed=0):
    q, k, v = workloads.make_qkv(cfg, seed=seed)
    return q, k, v, q.cuda(), k.cuda(), v.cuda()


# (name, B, H, S, d, P): the small presets run in full against the oracle,
# plus ragged shapes that span several tiles and end in a partial tile,
# chunks that straddle tiles, and degenerate sizes.
FULL_CASES = [
    ("tiny", 1, 4, 256, 64, 2),
    ("image", 1, 24, 4096, 128, 4),
    ("joint", 1, 24, 4608, 128, 8),
    ("ragged_200_P2", 1, 2, 200, 128, 2),
    ("ragged_300_P3", 1, 3, 300, 128, 3),
    ("ragged_1000_P8_d64", 1, 8, 1000, 64, 8),
    ("ragged_4608_P8_H8", 1, 8, 4608, 128, 8),
    ("batch2_odd_blocks", 2, 2, 640, 128, 2),
    ("one_row", 1, 1, 1, 128, 1),
    ("S_lt_P", 1, 8, 5, 64, 8),
    ("one_tile_plus_one", 1, 1, 129, 64, 1),
    # the partition maximum: 64 ranks of 10-11 rows, so every 128-row tile
    # straddles a dozen destination partitions
    ("P64_max_partitions", 1, 64, 700, 64, 64),
    ("batch3_ragged", 3, 4, 333, 128, 4),
]


def case_cfg(name, B, H, S, d, P):
    if name in workloads.CONFIGS:
        return workloads.CONFIGS[name]
    return workloads.AttnConfig(name, B=B, H=H, S=S, d=d, P=P)


@pytest.mark.parametrize("case", FULL_CASES, ids=[c[0] for c in FULL_CASES])
def test_fused_matches_oracle(case):
    cfg = case_cfg(*case)
    q, k, v, dq, dk, dv = cuda_qkv(cfg)
    g = fused(dq, dk, dv, cfg.P, cfg.scale)
    assert g.guards_intact(), "epilogue wrote outside a partition"
    want = orc.head_to_seq_partitions(orc.attention_fp64(q, k, v, cfg.scale), cfg.P)
    for j, (got, w) in enumerate(zip(g.parts, want)):
        compare(orc.as_f64(got), w, f"{cfg.name} partition {j}")
    # per head, so that one wrong head cannot hide in the global norm
    o = partitions_to_bhsd(g.parts)
    ref = orc.seq_to_head(want)
    for h in range(cfg.H):
        compare(o[:, h], ref[:, h], f"{cfg.name} head {h}")


@pytest.mark.parametrize("case", FULL_CASES[:7], ids=[c[0] for c in FULL_CASES[:7]])
def test_layout_bit_exact_vs_attention_then_permute(case):
    cfg = case_cfg(*case)
    _, _, _, dq, dk, dv = cuda_qkv(cfg, seed=1)
    g = fused(dq, dk, dv, cfg.P, cfg.scale)
    o = torch.empty((cfg.B, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")
    bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o)
    serial = GuardedPartitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    bd.attn_a2a_permute(o, cfg.P, serial.parts)
    torch.cuda.synchronize()
    assert serial.guards_intact()
    for a, b in zip(g.parts, serial.parts):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_contig_matches_oracle():
    cfg = workloads.config("image", H=4, S=1000)
    q, k, v, dq, dk, dv = cuda_qkv(cfg, seed=2)
    o = torch.empty((cfg.B, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")
    bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o)
    torch.cuda.synchronize()
    compare(orc.as_f64(o), orc.attention_fp64(q, k, v, cfg.scale), "contig")


def test_simt_debug_path_matches_oracle():
    cfg = workloads.CONFIGS["tiny"]
    q, k, v, dq, dk, dv = cuda_qkv(cfg)
    g = GuardedPartitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    bd.attn_a2a_fwd_simt(dq, dk, dv, cfg.P, cfg.scale, g.parts)
    torch.cuda.synchronize()
    assert g.guards_intact()
    want = orc.head_to_seq_partitions(orc.attention_fp64(q, k, v, cfg.scale), cfg.P)
    for got, w in zip(g.parts, want):
        compare(orc.as_f64(got), w, "simt")


def test_strided_inputs():
    # q, k, v are views of [B, S, H, d] buffers (sequence-major memory), as a
    # Ulysses pre-attention exchange would leave them.
    B, H, S, d, P = 1, 4, 700, 128, 2
    gen = torch.Generator().manual_seed(3)
    base = [torch.randn((B, S, H, d), generator=gen).to(torch.bfloat16) for _ in range(3)]
    q, k, v = (t.permute(0, 2, 1, 3) for t in base)
    dq, dk, dv = (t.cuda().permute(0, 2, 1, 3) for t in base)
    assert dq.stride(2) == H * d
    scale = 1 / math.sqrt(d)
    g = fused(dq, dk, dv, P, scale)
    want = orc.head_to_seq_partitions(orc.attention_fp64(q, k, v, scale), P)
    for got, w in zip(g.parts, want):
        compare(orc.as_f64(got), w, "strided")


def test_scale_zero_and_constant_v():
    B, H, S, d, P = 1, 2, 333, 64, 2
    gen = torch.Generator().manual_seed(4)
    q = torch.randn((B, H, S, d), generator=gen).to(torch.bfloat16).cuda()
    k = torch.randn((B, H, S, d), generator=gen).to(torch.bfloat16).cuda()
    v = torch.randn((B, H, S, d), generator=gen).to(torch.bfloat16).cuda()
    g = fused(q, k, v, P, 0.0)  # uniform weights: every row is the mean of V
    got = partitions_to_bhsd(g.parts)
    mean = orc.as_f64(v).mean(axis=2, keepdims=True)
    compare(got, np.broadcast_to(mean, got.shape), "scale 0")
    vc = torch.full_like(v, 0.75)
    g = fused(q, k, vc, P, 1.0)
    got = partitions_to_bhsd(g.parts)
    compare(got, np.full(got.shape, 0.75), "constant V")
    # the rows sum bf16-rounded probabilities against an fp32 row sum, so a
    # constant comes back within P's rounding (2^-8 relative), not exactly
    assert np.abs(got - 0.75).max() <= 0.75 * 2.0 ** -8 + 2.0 ** -10


def test_empty_sequence_launches_nothing():
    q = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    assert bd.attn_a2a_fwd(q, q, q, 2, 0.1, [None, None]) == bd.OK


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("B,H,S", [(1, 4, 1500), (2, 16, 640), (1, 40, 300)])
def test_host_entry_point_matches_device_path(B, H, S, pinned):
    # head chunks: one head each for H = 4; a ramp (1, 3, 8, 3, 1 heads) per
    # batch entry for H = 16; the video head count (1, 3, 8, 20, 7, 1) for H = 40.
    # Pinned host partitions receive the rows straight from the kernels (the
    # device partitions stay untouched); pageable ones by copies from dparts
    cfg = workloads.config("image", B=B, H=H, S=S)
    q, k, v = workloads.make_qkv(cfg, seed=5)
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    dparts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=7.0)
    hparts = [torch.zeros(p.shape, dtype=p.dtype, pin_memory=pinned) for p in dparts]
    bd.attn_a2a_fwd_host(hq, hk, hv, cfg.P, cfg.scale, dq, dk, dv, dparts, hparts)
    torch.cuda.synchronize()
    ref = fused(q.cuda(), k.cuda(), v.cuda(), cfg.P, cfg.scale)
    for a, b in zip(hparts, ref.parts):
        assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16))
    for d in dparts:
        assert bool(torch.all(d == 7.0)) == pinned


def test_bounded_wait_reports_timeout_and_context_survives():
    cfg = workloads.CONFIGS["tiny"]
    _, _, _, dq, dk, dv = cuda_qkv(cfg)
    parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd(dq, dk, dv, cfg.P, cfg.scale, parts, dev_status=status, inject_stall=1,
                    timeout_ns=50_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == bd.ETIMEOUT
    # the context is still usable and a normal call is correct afterwards
    g = fused(dq, dk, dv, cfg.P, cfg.scale)
    assert g.guards_intact()


def test_grid_size_does_not_change_result():
    cfg = workloads.config("image", H=6, S=1111)
    _, _, _, dq, dk, dv = cuda_qkv(cfg, seed=6)
    a = fused(dq, dk, dv, 2, cfg.scale)
    b = fused(dq, dk, dv, 2, cfg.scale, grid=3)
    for x, y in zip(a.parts, b.parts):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("name", ["image", "tiny"])
def test_chunk_interleaved_order_gives_identical_output(name):
    cfg = workloads.CONFIGS[name]
    _, _, _, dq, dk, dv = cuda_qkv(cfg, seed=8)
    a = fused(dq, dk, dv, cfg.P, cfg.scale)
    b = fused(dq, dk, dv, cfg.P, cfg.scale, tile_order=1)
    assert b.guards_intact()
    for x, y in zip(a.parts, b.parts):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_growing_and_jumping_scores_take_the_rescale_path():
    # Key magnitudes grow along the sequence, so the running row maximum is
    # overtaken again and again; one block in the middle has scores large
    # enough that exponentiating it against the stale maximum overflows. Both
    # force the kernel's fallback (take the block maximum, rescale O and l).
    B, H, S, d, P = 1, 2, 1536, 128, 2
    gen = torch.Generator().manual_seed(9)
    q = torch.randn((B, H, S, d), generator=gen)
    growth = 1.0 + 6.0 * torch.arange(S, dtype=torch.float32) / S
    k = torch.randn((B, H, S, d), generator=gen) * growth[None, None, :, None]
    k[:, :, 700:760] *= 6.0
    v = torch.randn((B, H, S, d), generator=gen)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1 / math.sqrt(d)
    g = fused(q.cuda(), k.cuda(), v.cuda(), P, scale)
    assert g.guards_intact()
    want = orc.head_to_seq_partitions(orc.attention_fp64(q, k, v, scale), P)
    for j, (got, w) in enumerate(zip(g.parts, want)):
        compare(orc.as_f64(got), w, f"growing scores, partition {j}")


# The bulk-store epilogue (store_kind = 1, the default where it is built)
# against the register-store one (store_kind = 2): same arithmetic, so the
# partitions must match byte for byte. The cases
# include tiles that straddle two partitions (stored row by row), ragged
# ends (rows past S are clipped by the tensor store), batch 2, d = 64 and
# fewer rows than ranks.
BULK_CASES = [
    ("tiny", 1, 4, 256, 64, 2),
    ("image", 1, 24, 4096, 128, 4),
    ("joint", 1, 24, 4608, 128, 8),
    ("ragged_1000_P8_d64", 1, 8, 1000, 64, 8),
    ("ragged_300_P3", 1, 3, 300, 128, 3),
    ("batch2_odd_blocks", 2, 2, 640, 128, 2),
    ("S_lt_P", 1, 8, 5, 64, 8),
]


@pytest.mark.parametrize("case", BULK_CASES, ids=[c[0] for c in BULK_CASES])
def test_bulk_store_epilogue_matches_register_stores(case):
    cfg = case_cfg(*case)
    _, _, _, dq, dk, dv = cuda_qkv(cfg, seed=7)
    a = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=2)
    b = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=1)
    c = fused(dq, dk, dv, cfg.P, cfg.scale)  # automatic: bulk here
    assert b.guards_intact() and c.guards_intact(), "bulk stores wrote outside a partition"
    for x, y, z in zip(a.parts, b.parts, c.parts):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
        assert torch.equal(y.view(torch.int16), z.view(torch.int16))


@pytest.mark.parametrize("S", [16384, 32768, 32769])
def test_automatic_store_kind_matches_both_kinds(S):
    # the automatic kind (bulk stores at every length, where the partitions
    # are device memory and P <= 8) and both explicit kinds write the same bytes
    cfg = workloads.AttnConfig(f"switch_{S}", B=1, H=2, S=S, d=128, P=2)
    _, _, _, dq, dk, dv = cuda_qkv(cfg, seed=14)
    outs = [fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=kind) for kind in (0, 1, 2)]
    for g in outs:
        assert g.guards_intact()
    for x, y, z in zip(*(g.parts for g in outs)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
        assert torch.equal(x.view(torch.int16), z.view(torch.int16))


def test_bulk_store_epilogue_with_interleaved_order():
    cfg = workloads.CONFIGS["image"]
    _, _, _, dq, dk, dv = cuda_qkv(cfg, seed=9)
    a = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=2)
    b = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=1, tile_order=1)
    assert b.guards_intact()
    for x, y in zip(a.parts, b.parts):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("B,H,S,d", [(1, 4, 1000, 128), (2, 3, 333, 64), (1, 2, 129, 128)])
def test_contiguous_bulk_store_epilogue_matches_row_stores(B, H, S, d):
    # attention alone: bulk tensor stores of [B, H, S, d] (the default) against
    # row stores; rows past S are clipped by the tensor store
    cfg = workloads.AttnConfig("contig", B=B, H=H, S=S, d=d, P=1)
    _, _, _, dq, dk, dv = cuda_qkv(cfg, seed=10)
    pad = 512
    outs = []
    for kind in (2, 1, 0):
        buf = torch.full((B * H * S * d + 2 * pad,), -12345.0, dtype=torch.bfloat16, device="cuda")
        o = buf[pad:pad + B * H * S * d].view(B, H, S, d)
        bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o, store_kind=kind)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == -12345.0) and torch.all(buf[-pad:] == -12345.0)
        outs.append(o.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
