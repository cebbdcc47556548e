"""The allocation-free probe entry point, xstage_probe_run_noalloc.

It exists for callers that may not call cudaMalloc when they want to measure
(their device memory belongs to another allocator, or their runtime forbids
allocation after start-up): the burst target is a fixed 16 MiB array inside
the library instead of a caller buffer. This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process, where its first call does the per-device
set-up.

The probe's output is timing, so "the same output" means the same measurement:
two calls in a row of the new entry point are each compared with the existing
entry point given a caller-owned target of the same 16 MiB, same producers,
burst and gap; the stamps must be well formed and the median issue time and
period must agree within the 15 % the probe's model checks use.
"""
import statistics

import pytest
import torch

from attention_all_layout_gb300 import binding as bd

pytestmark = pytest.mark.gpu

REL_TOL = 0.15


def summary(stamps, K, rounds):
    s = stamps.view(K, rounds, 3).cpu()
    assert torch.all(s[:, :, 1] >= s[:, :, 0])
    assert torch.all(s[:, 1:, 0] >= s[:, :-1, 2])
    half = s[:, rounds // 2:, :].double()
    t_iss = statistics.median((half[:, :, 1] - half[:, :, 0]).mean(dim=0).tolist())
    period = statistics.median((half[:, :, 2] - half[:, :, 0]).mean(dim=0).tolist())
    return s, t_iss, period


# (store kind, gap kind, gap iterations): idle gaps with both store kinds, a
# dependent-FMA gap, and tensor-core work as the gap (needs the larger dynamic
# shared memory and TMEM).
CASES = [(0, 0, 0), (1, 0, 0), (0, 1, 4000), (1, 2, 200)]


@pytest.mark.parametrize("kind,gap_kind,iters", CASES, ids=lambda x: str(x))
def test_noalloc_probe_matches_caller_buffer_probe(kind, gap_kind, iters):
    K = bd.num_sms()
    rounds, G_ns = 32, 10_000
    V = (8 * 2**20 // (4096 * K)) * 4096 * K
    target = torch.empty(bd.NOALLOC_MAX_BYTES, dtype=torch.uint8, device="cuda")
    ref_st = torch.zeros(K * rounds * 3, dtype=torch.int64, device="cuda")
    bd.xstage_probe_run(K, rounds, V, G_ns, target, ref_st, store_kind=kind, gap_kind=gap_kind, fma_iters=iters)
    torch.cuda.synchronize()
    _, ref_iss, ref_period = summary(ref_st, K, rounds)
    for call in range(2):  # two calls in a row share the library's array
        st = torch.zeros(K * rounds * 3, dtype=torch.int64, device="cuda")
        bd.xstage_probe_run_noalloc(K, rounds, V, G_ns, st, store_kind=kind, gap_kind=gap_kind, fma_iters=iters)
        torch.cuda.synchronize()
        s, t_iss, period = summary(st, K, rounds)
        if gap_kind == 0:
            assert torch.all(s[:, :, 2] - s[:, :, 1] >= G_ns), f"call {call}: gap not honoured"
        else:
            assert torch.all(s[:, :, 2] >= s[:, :, 1]), f"call {call}: gap stamps out of order"
        assert abs(t_iss - ref_iss) <= REL_TOL * ref_iss, f"call {call}: issue time {t_iss} vs {ref_iss} ns"
        assert abs(period - ref_period) <= REL_TOL * ref_period, f"call {call}: period {period} vs {ref_period} ns"


def test_noalloc_probe_rejects_bursts_beyond_its_array():
    K = bd.num_sms()
    st = torch.zeros(K * 3, dtype=torch.int64, device="cuda")
    V = (bd.NOALLOC_MAX_BYTES // (4096 * K) + 1) * 4096 * K
    assert bd.xstage_probe_run_noalloc(K, 1, V, 0, st, check=False) == bd.ETOOLARGE
    assert "scratch" in bd.strerror(bd.ETOOLARGE)
