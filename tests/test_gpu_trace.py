"""GPU tests of the traced attention kernel (per-tile stamps for the store-span
and tensor-core-timeline views of the X-Stage pages' "Results"): the traced
call writes the same partitions, byte for byte, as the untraced call; every
tile's record is written; the stamps of a tile are ordered; spans are
non-negative; each record names the CTA that the static schedule gives its
item and the tile's first row."""
import numpy as np
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import tile_trace as tt
from attention_all_layout_gb300 import workloads

pytestmark = pytest.mark.gpu

# ragged: S not a multiple of 128 (last tile partial), an odd block count (the
# last item's second tile has no rows), chunks straddled by tiles
CASES = [
    dict(B=1, H=6, S=1100, d=128, P=3),
    dict(B=2, H=4, S=600, d=64, P=2),
]


def check_records(rec, S, grid):
    items = rec.shape[0]
    assert np.all(rec[:, :, :, 0] > 0), "record not written"
    for w in range(4):
        assert np.all(rec[:, :, w, 0] <= rec[:, :, w, 1])
        assert np.all(rec[:, :, w, 1] <= rec[:, :, w, 2])
        assert np.all(rec[:, :, w, 2] <= rec[:, :, w, 3])
        assert np.all(rec[:, :, w, 4] >= 0)
    nsm = bd.num_sms()
    assert np.all((rec[:, :, :, 5] >= 0) & (rec[:, :, :, 5] < nsm))
    item = np.arange(items)[:, None, None]
    assert np.all(rec[:, :, :, 6] == item % grid)
    pairs = ((S + 127) // 128 + 1) // 2
    t = np.arange(2)[None, :, None]
    assert np.all(rec[:, :, :, 7] == (2 * (item % pairs) + t) * 128)
    assert np.all(tt.store_span_ns(rec) >= 0)
    # a CTA runs its items in order: each tile's Q loop starts after the
    # previous item's tile of the same index has finished its Q loop
    for c in range(grid):
        mine = rec[c::grid]
        for t_ in range(2):
            assert np.all(mine[1:, t_, 0, 0] >= mine[:-1, t_, 0, 1])


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{B}H{H}S{S}d{d}P{P}".format(**c))
@pytest.mark.parametrize("store_kind", [1, 2])
@pytest.mark.parametrize("layout", ["a2a", "contig"])
def test_traced_call_matches_untraced(case, store_kind, layout):
    cfg = workloads.AttnConfig("trace", **case)
    q, k, v = workloads.make_qkv(cfg, seed=3, device="cuda")
    trace = torch.full((bd.trace_numel(cfg.B, cfg.H, cfg.S),), -1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if layout == "a2a":
        ref = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
        got = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
        bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, ref, store_kind=store_kind)
        bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, got, dev_status=status, store_kind=store_kind, trace=trace)
    else:
        ref = [torch.zeros((cfg.B, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")]
        got = [torch.zeros_like(ref[0])]
        bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, ref[0], store_kind=store_kind)
        bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, got[0], dev_status=status, store_kind=store_kind, trace=trace)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    pairs = ((cfg.S + 127) // 128 + 1) // 2
    grid = min(bd.num_sms(), cfg.B * cfg.H * pairs)
    rec = tt.records(trace, cfg.B, cfg.H, cfg.S)
    check_records(rec, cfg.S, grid)
    s = tt.summary(rec, cfg.S, grid)
    assert s["store_span_ns"]["n"] > 0


def test_trace_rejects_short_buffer():
    cfg = workloads.AttnConfig("trace", B=1, H=2, S=256, d=64, P=2)
    q, k, v = workloads.make_qkv(cfg, seed=0, device="cuda")
    parts = bd.alloc_partitions(1, cfg.S, cfg.H, cfg.d, cfg.P)
    short = torch.zeros(bd.trace_numel(1, 2, 256) - 1, dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, parts, trace=short)
