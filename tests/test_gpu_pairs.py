"""GPU tests of the CTA-pair kernel (attn_a2a_opts.cta_pairs = 1): clusters of
two CTAs on two SMs whose tensor cores run every MMA of a work unit (four
128-row query tiles of one head, two per CTA) as one 256-row MMA, each CTA
holding its own query tiles and half of every K and V block.

* Against the float64 oracle element by element, with guard bands around the
  partitions: ragged S, a head with an odd number of query-tile pairs (its last
  unit's second pair lies past S), B = 2, tiles straddling partitions, a grid
  of four clusters running many units each through the K/V ring.
* Byte for byte the same output as one CTA per work item (cta_pairs = 2): each
  row's scores and outputs are the same products summed in the same order, in
  the all-to-all and the contiguous layout, up to the video preset's size.
* Refusals where the pair kernel does not exist (row stores, d = 64, the
  chunk-interleaved order, a trace), and the bounded waits of both CTAs when
  the first probabilities are withheld: ATTN_A2A_ETIMEOUT, and the context
  stays usable.
"""
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import workloads
from oracle import attention as orc

from gpu_helpers import compare, fused, partitions_to_bhsd

pytestmark = pytest.mark.gpu

CASES = [
    (dict(B=1, H=2, S=1024, d=128, P=2), 0),
    (dict(B=1, H=3, S=1000, d=128, P=3), 0),   # ragged, tiles straddling partitions
    (dict(B=2, H=3, S=640, d=128, P=1), 0),    # 3 pairs per head: the last unit half past S
    (dict(B=1, H=8, S=2304, d=128, P=8), 8),   # 4 clusters, 5 units each
    (dict(B=1, H=8, S=4608, d=128, P=8), 0),   # 576-row partitions: tiles stored in 64-row halves
]


def same_bytes(a_parts, b_parts):
    return all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(a_parts, b_parts))


@pytest.mark.parametrize("case,grid", CASES, ids=lambda c: str(c))
def test_pairs_match_oracle_and_single_cta(case, grid):
    cfg = workloads.AttnConfig("pairs", **case)
    q, k, v = workloads.make_qkv(cfg, seed=11)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    g1 = fused(dq, dk, dv, cfg.P, cfg.scale, cta_pairs=bd.PAIRS_ON, grid=grid)
    assert g1.guards_intact()
    compare(partitions_to_bhsd([p.cpu() for p in g1.parts]), orc.attention_fp64(q, k, v, cfg.scale), "pairs")
    g2 = fused(dq, dk, dv, cfg.P, cfg.scale, cta_pairs=bd.PAIRS_OFF, grid=grid)
    assert same_bytes(g1.parts, g2.parts)


def test_pairs_contiguous_layout():
    cfg = workloads.AttnConfig("pairs", B=1, H=2, S=1000, d=128, P=1)
    q, k, v = workloads.make_qkv(cfg, seed=12)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o1 = torch.empty(1, 2, 1000, 128, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o1, cta_pairs=bd.PAIRS_ON)
    bd.attn_a2a_fwd_contig(dq, dk, dv, cfg.scale, o2, cta_pairs=bd.PAIRS_OFF)
    torch.cuda.synchronize()
    compare(o1.float().cpu().numpy(), orc.attention_fp64(q, k, v, cfg.scale), "pairs, contiguous")
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_pairs_image_preset_same_bytes():
    cfg = workloads.CONFIGS["image"]
    q, k, v = workloads.make_qkv(cfg, seed=13, device="cuda")
    g1 = fused(q, k, v, cfg.P, cfg.scale, cta_pairs=bd.PAIRS_ON)
    g2 = fused(q, k, v, cfg.P, cfg.scale, cta_pairs=bd.PAIRS_OFF)
    assert g1.guards_intact()
    assert same_bytes(g1.parts, g2.parts)


@pytest.mark.parametrize("kw,d", [(dict(store_kind=2), 128), (dict(tile_order=1), 128), ({}, 64)])
def test_pairs_refused_where_not_built(kw, d):
    cfg = workloads.AttnConfig("pairs", B=1, H=2, S=1024, d=d, P=2)
    q, k, v = workloads.make_qkv(cfg, seed=1, device="cuda")
    parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    rc = bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, parts, cta_pairs=bd.PAIRS_ON, check=False, **kw)
    assert rc == bd.EUNSUPPORTED


def test_pairs_refused_with_trace():
    cfg = workloads.AttnConfig("pairs", B=1, H=2, S=1024, d=128, P=2)
    q, k, v = workloads.make_qkv(cfg, seed=1, device="cuda")
    parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    tr = torch.zeros(bd.trace_numel(cfg.B, cfg.H, cfg.S), dtype=torch.int64, device="cuda")
    rc = bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, parts, trace=tr, cta_pairs=bd.PAIRS_ON, check=False)
    assert rc == bd.EUNSUPPORTED


def test_pairs_bounded_wait_reports_timeout():
    cfg = workloads.AttnConfig("pairs", B=1, H=2, S=1024, d=128, P=2)
    q, k, v = workloads.make_qkv(cfg, seed=2, device="cuda")
    parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, parts, dev_status=status, inject_stall=1, timeout_ns=50_000_000,
                    cta_pairs=bd.PAIRS_ON)
    torch.cuda.synchronize()
    assert int(status.item()) == bd.ETIMEOUT
    g = fused(q, k, v, cfg.P, cfg.scale, cta_pairs=bd.PAIRS_ON)
    assert g.guards_intact()


def test_pairs_video_preset_same_bytes():
    # the full video shape: 2560 units of 256 key blocks on 76 clusters, the K/V
    # ring of eight half stages wrapping many times per unit
    cfg = workloads.CONFIGS["video"]
    q, k, v = workloads.make_qkv(cfg, seed=14, device="cuda")
    g1 = fused(q, k, v, cfg.P, cfg.scale, cta_pairs=bd.PAIRS_ON)
    g2 = fused(q, k, v, cfg.P, cfg.scale, cta_pairs=bd.PAIRS_OFF, split=bd.SPLIT_NONE)
    assert g1.guards_intact()
    assert same_bytes(g1.parts, g2.parts)
