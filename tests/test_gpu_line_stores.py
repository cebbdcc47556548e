"""GPU tests of the whole-line row-store epilogue (attn_a2a_opts.store_kind = 3)
and of the fused call storing into partitions in host memory.

* Against the float64 oracle element by element (ragged S, d = 64 and 128,
  B = 2, P = 3 with tiles straddling partitions, P = 16), with guard bands
  around every partition.
* Byte for byte the same partitions as the row stores from registers (kind 2)
  - the two kinds compute the same values and only write them differently -
  also for a head-group call into full-width partitions, with the split
  schedule, and in the traced instantiation.
* Bulk tensor stores in two 64-row halves where equal partitions of an odd
  multiple of 64 rows cut tiles in half: against the oracle and byte for byte
  the row stores.
* Into pinned host memory (the device stores straight into the host's
  partitions over the host link): the same bytes as into device memory, for
  kinds 2 and 3, at a small shape and at the image preset's size.
"""
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import ulysses as ul
from attention_all_layout_gb300 import workloads
from oracle import attention as orc

from gpu_helpers import compare, fused, partitions_to_bhsd

pytestmark = pytest.mark.gpu

CASES = [
    dict(B=1, H=2, S=256, d=128, P=2),
    dict(B=1, H=3, S=1000, d=128, P=3),   # ragged, tiles straddling partitions
    dict(B=2, H=3, S=777, d=64, P=3),
    dict(B=1, H=16, S=640, d=64, P=16),   # more partitions than the bulk path's tensor maps
]


def same_bytes(a_parts, b_parts):
    return all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(a_parts, b_parts))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{B}H{H}S{S}d{d}P{P}".format(**c))
def test_line_stores_match_oracle_and_row_stores(case):
    cfg = workloads.AttnConfig("line", **case)
    q, k, v = workloads.make_qkv(cfg, seed=5)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    g3 = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=3)
    assert g3.guards_intact()
    got = partitions_to_bhsd([p.cpu() for p in g3.parts])
    want = orc.attention_fp64(q, k, v, cfg.scale)
    compare(got, want, "line stores")
    g2 = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=2)
    assert same_bytes(g3.parts, g2.parts)


def test_line_stores_head_group_call():
    cfg = workloads.AttnConfig("line", B=1, H=8, S=1000, d=128, P=4)
    q, k, v = workloads.make_qkv(cfg, seed=6, device="cuda")
    ref = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
    got = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, ref, store_kind=2)
    bases = [t.data_ptr() for t in got]
    for r in range(cfg.P):
        p = ul.plan(r, cfg.P, cfg.B, cfg.H, cfg.S, cfg.d)
        ul.rank_forward(p, q[:, p.h0:p.h1], k[:, p.h0:p.h1], v[:, p.h0:p.h1], bases, cfg.scale, store_kind=3)
    torch.cuda.synchronize()
    assert same_bytes(ref, got)


@pytest.mark.parametrize("split", [bd.SPLIT_TAIL, bd.SPLIT_ALL])
def test_line_stores_with_split_schedule(split):
    cfg = workloads.AttnConfig("line", B=1, H=4, S=8192, d=128, P=4)
    q, k, v = workloads.make_qkv(cfg, seed=7, device="cuda")
    ws = bd.alloc_workspace(cfg.d, 24)
    g2 = fused(q, k, v, cfg.P, cfg.scale, store_kind=2, grid=24, workspace=ws, split=split)
    g3 = fused(q, k, v, cfg.P, cfg.scale, store_kind=3, grid=24, workspace=ws, split=split)
    assert g3.guards_intact()
    assert same_bytes(g2.parts, g3.parts)


def test_line_stores_traced():
    cfg = workloads.AttnConfig("line", B=1, H=3, S=1000, d=128, P=3)
    q, k, v = workloads.make_qkv(cfg, seed=8, device="cuda")
    tr = torch.zeros(bd.trace_numel(cfg.B, cfg.H, cfg.S), dtype=torch.int64, device="cuda")
    a = fused(q, k, v, cfg.P, cfg.scale, store_kind=3)
    b = fused(q, k, v, cfg.P, cfg.scale, store_kind=3, trace=tr)
    assert same_bytes(a.parts, b.parts)
    rec = tr.view(-1, bd.TRACE_RECORD).cpu()
    assert bool((rec[:, 3] >= rec[:, 2]).all()) and bool((rec[:, 2] >= rec[:, 1]).all())


@pytest.mark.parametrize("name", ["small", "image", "long"])
@pytest.mark.parametrize("store_kind", [0, 2, 3])
def test_partitions_in_host_memory(name, store_kind):
    # kind 0 (automatic) would take bulk stores for device partitions; for host
    # partitions the library takes the whole-line row stores
    cfg = {"small": workloads.AttnConfig("host", B=1, H=3, S=1000, d=128, P=3), "image": workloads.CONFIGS["image"],
           "long": workloads.AttnConfig("host", B=1, H=2, S=33000, d=64, P=2)}[name]
    q, k, v = workloads.make_qkv(cfg, seed=9, device="cuda")
    dev = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
    host = [torch.zeros(t.shape, dtype=t.dtype, pin_memory=True) for t in dev]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, dev, store_kind=store_kind)
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, [t.data_ptr() for t in host], dev_status=status,
                    store_kind=store_kind)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert same_bytes(host, [t.cpu() for t in dev])


def test_bulk_stores_refused_outside_device_memory():
    cfg = workloads.AttnConfig("host", B=1, H=2, S=512, d=128, P=2)
    q, k, v = workloads.make_qkv(cfg, seed=10, device="cuda")
    host = [torch.zeros(t, dtype=torch.bfloat16, pin_memory=True) for t in
            [(1, c, cfg.H, cfg.d) for c in bd.chunk_sizes(cfg.S, cfg.P)]]
    assert bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, [t.data_ptr() for t in host], store_kind=1,
                           check=False) == bd.EUNSUPPORTED
    o = torch.zeros((1, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, pin_memory=True)
    assert bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o, store_kind=1, check=False) == bd.EUNSUPPORTED
    # the automatic kind stores the contiguous output into host memory with row stores
    dev = torch.empty((1, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")
    bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, dev)
    bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), dev.cpu().view(torch.int16))


# Equal partitions of an odd multiple of 64 rows: every other partition
# boundary cuts a 128-row tile in half, and the bulk-store epilogue stores
# every tile as two 64-row halves, each into the partition holding it.
HALF_CASES = [
    dict(B=1, H=8, S=4608, d=128, P=8),   # the joint preset's partitions (576 rows)
    dict(B=1, H=3, S=192, d=128, P=3),    # 64-row partitions: every tile cut
    dict(B=2, H=4, S=640, d=64, P=2),     # 320-row partitions, d = 64, batch 2
    dict(B=1, H=5, S=320, d=128, P=5),    # 64-row partitions, an odd tile count
]


@pytest.mark.parametrize("case", HALF_CASES, ids=lambda c: "B{B}H{H}S{S}d{d}P{P}".format(**c))
def test_half_tile_bulk_stores_match_oracle_and_row_stores(case):
    cfg = workloads.AttnConfig("halves", **case)
    q, k, v = workloads.make_qkv(cfg, seed=9)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    g1 = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=1)
    assert g1.guards_intact()
    compare(partitions_to_bhsd([p.cpu() for p in g1.parts]), orc.attention_fp64(q, k, v, cfg.scale), "half tiles")
    g2 = fused(dq, dk, dv, cfg.P, cfg.scale, store_kind=2)
    assert same_bytes(g1.parts, g2.parts)
