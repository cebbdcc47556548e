"""GPU test of the Ulysses head-group call (attn_a2a_opts.part_heads, used by
ulysses.rank_forward): P calls, one per rank's head group, each storing into
all P partitions at its heads' slots, give the partitions of one call over all
heads byte for byte. On one GPU the P "ranks" run in turn into partitions on
the same device; on several GPUs the same calls store into peer partitions."""
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import ulysses as ul
from attention_all_layout_gb300 import workloads

pytestmark = pytest.mark.gpu

CASES = [
    dict(B=1, H=8, S=1024, d=128, P=4),
    dict(B=1, H=6, S=1000, d=64, P=3),   # ragged chunks, tiles straddling them
    dict(B=2, H=4, S=300, d=128, P=2),
    dict(B=1, H=16, S=4608, d=128, P=8),  # joint-preset chunks of 576 rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{B}H{H}S{S}d{d}P{P}".format(**c))
@pytest.mark.parametrize("store_kind", [0, 1, 2])
def test_head_group_calls_fill_partitions_like_one_call(case, store_kind):
    cfg = workloads.AttnConfig("ulysses", **case)
    q, k, v = workloads.make_qkv(cfg, seed=11, device="cuda")
    ref = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
    got = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, ref, store_kind=store_kind)
    bases = [t.data_ptr() if t.numel() else 0 for t in got]
    for r in range(cfg.P):
        p = ul.plan(r, cfg.P, cfg.B, cfg.H, cfg.S, cfg.d)
        # the rank's head group is a strided view of the full tensors
        ul.rank_forward(p, q[:, p.h0:p.h1], k[:, p.h0:p.h1], v[:, p.h0:p.h1], bases, cfg.scale,
                        dev_status=status, store_kind=store_kind)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_head_group_call_leaves_other_heads_alone():
    cfg = workloads.AttnConfig("ulysses", B=1, H=8, S=512, d=128, P=4)
    q, k, v = workloads.make_qkv(cfg, seed=2, device="cuda")
    parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=7.0)
    p = ul.plan(1, cfg.P, cfg.B, cfg.H, cfg.S, cfg.d)
    ul.rank_forward(p, q[:, p.h0:p.h1], k[:, p.h0:p.h1], v[:, p.h0:p.h1], [t.data_ptr() for t in parts],
                    cfg.scale)
    torch.cuda.synchronize()
    for t in parts:
        other = torch.cat([t[:, :, :p.h0], t[:, :, p.h1:]], dim=2)
        assert torch.all(other == 7.0)
        assert not torch.any(t[:, :, p.h0:p.h1] == 7.0)
