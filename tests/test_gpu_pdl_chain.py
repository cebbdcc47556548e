"""GPU test of the ordering between consecutive calls on one stream. A call's
first kernel is launched with programmatic stream serialisation behind the
stream's previous kernel: its CTAs run their set-up on SMs that the previous
kernel's CTAs leave and wait for that kernel (griddepcontrol.wait) before
touching global memory; a tail kernel waits for the plain kernel ahead of it
before it exits, so that its completion covers the plain kernel's stores.

Here the second call reads the first call's output as its q, both queued with
no host synchronisation in between, over output buffers filled with NaN
beforehand: reading any row before the first call has stored it would show
up. Both outputs must be byte-identical to the same two calls each followed
by a device synchronisation - for the plain kernel alone (a partial last wave,
so that most CTAs exit early and the next call's CTAs start beside the last
ones), the plain kernel with the tail kernel behind it, and the
whole-schedule split, with both store kinds; the same for the fused call
behind attention alone, and for two whole-layer calls (sequence-sharded in
and out), the second reading the first one's output partitions.
"""
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import workloads

pytestmark = pytest.mark.gpu

# 128 work items of 64 key blocks on 24 CTAs: a last wave of 8
B, H, S, D, GRID = 1, 4, 8192, 128, 24
SPLITS = {"plain": bd.SPLIT_NONE, "tail": bd.SPLIT_TAIL, "all": bd.SPLIT_ALL}


def nan_like(x):
    return torch.full_like(x, float("nan"))


@pytest.mark.parametrize("store_kind", [1, 2])
@pytest.mark.parametrize("schedule", list(SPLITS))
def test_second_call_reads_the_first_calls_output(schedule, store_kind):
    split = SPLITS[schedule]
    cfg = workloads.AttnConfig("chain", B=B, H=H, S=S, d=D, P=1)
    q, k, v = (t.cuda() for t in workloads.make_qkv(cfg, seed=11))
    ws = bd.alloc_workspace(D, GRID)

    def call(qq, out):
        bd.attn_a2a_fwd_contig(qq, k, v, cfg.scale, out, grid=GRID, workspace=ws, store_kind=store_kind,
                               split=split)

    # each call on its own
    ref1 = nan_like(q)
    call(q, ref1)
    torch.cuda.synchronize()
    ref2 = nan_like(q)
    call(ref1, ref2)
    torch.cuda.synchronize()
    assert not torch.isnan(ref1).any() and not torch.isnan(ref2).any()

    for _ in range(3):
        o1, o2 = nan_like(q), nan_like(q)
        torch.cuda.synchronize()
        call(q, o1)
        call(o1, o2)  # queued right behind the call that writes its q
        torch.cuda.synchronize()
        assert torch.equal(o1.view(torch.int16), ref1.view(torch.int16))
        assert torch.equal(o2.view(torch.int16), ref2.view(torch.int16)), f"{schedule}: second call read early"


def test_fused_call_behind_attention_alone():
    """The fused call's partitions from q that attention alone writes just before."""
    cfg = workloads.AttnConfig("chain", B=B, H=H, S=S, d=D, P=4)
    q, k, v = (t.cuda() for t in workloads.make_qkv(cfg, seed=12))
    ws = bd.alloc_workspace(D, GRID)
    o = nan_like(q)
    bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o, grid=GRID, workspace=ws)
    torch.cuda.synchronize()
    ref = bd.alloc_partitions(B, S, H, D, cfg.P)
    bd.attn_a2a_fwd(o, k, v, cfg.P, cfg.scale, ref, grid=GRID, workspace=ws)
    torch.cuda.synchronize()
    o2 = nan_like(q)
    parts = bd.alloc_partitions(B, S, H, D, cfg.P)
    for p in parts:
        p.fill_(float("nan"))
    torch.cuda.synchronize()
    bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o2, grid=GRID, workspace=ws)
    bd.attn_a2a_fwd(o2, k, v, cfg.P, cfg.scale, parts, grid=GRID, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(parts, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("split", [bd.SPLIT_NONE, bd.SPLIT_ALL])
def test_layer_call_reads_the_previous_layer_calls_output(split):
    """The whole layer (sequence-sharded q, k, v in and out): a second call whose q
    partitions are the first call's output partitions, queued right behind it."""
    cfg = workloads.AttnConfig("chain", B=B, H=H, S=S, d=D, P=4)
    q, k, v = (t.cuda() for t in workloads.make_qkv(cfg, seed=13))
    qp, kp, vp = (bd.alloc_partitions(B, S, H, D, cfg.P) for _ in range(3))
    for src, dst in ((q, qp), (k, kp), (v, vp)):
        bd.attn_a2a_permute(src, cfg.P, dst)
    ws = bd.alloc_workspace(D, GRID)
    torch.cuda.synchronize()

    def layer(qparts, out):
        bd.attn_a2a_fwd_s2s(qparts, kp, vp, cfg.P, cfg.scale, out, grid=GRID, workspace=ws, split=split)

    def nan_parts():
        parts = bd.alloc_partitions(B, S, H, D, cfg.P)
        for p in parts:
            p.fill_(float("nan"))
        return parts

    ref1, ref2 = nan_parts(), nan_parts()
    layer(qp, ref1)
    torch.cuda.synchronize()
    layer(ref1, ref2)
    torch.cuda.synchronize()
    assert not any(bool(torch.isnan(p).any()) for p in ref1 + ref2)
    for _ in range(3):
        o1, o2 = nan_parts(), nan_parts()
        torch.cuda.synchronize()
        layer(qp, o1)
        layer(o1, o2)
        torch.cuda.synchronize()
        for a, b in zip(o1 + o2, ref1 + ref2):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
