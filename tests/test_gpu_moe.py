"""GPU parity of the synthetic MegaMoE-style grouped GEMM (moe_gemm_scatter)
against its float64 oracle, for the Expert-Wave and the interleaved task
orders (bit-identical to each other), plus malformed input handling."""
import numpy as np
import pytest
import torch

from attention_all_layout_gb300 import binding as bd
from attention_all_layout_gb300 import moe_sched as ms
from oracle import moe as om

from gpu_helpers import compare

pytestmark = pytest.mark.gpu


def run(x, w1, w2, tasks_np, rm, rows, N, status=None):
    h = torch.full((x.shape[0], x.shape[1], N), -7.0, dtype=torch.bfloat16, device="cuda")
    dst = [torch.full((r, N), -7.0, dtype=torch.bfloat16, device="cuda") for r in rows]
    bd.moe_gemm_scatter(x, w1, w2, torch.from_numpy(tasks_np).cuda(), h, torch.from_numpy(rm).cuda(), dst,
                        dev_status=status)
    torch.cuda.synchronize()
    return h, dst


@pytest.mark.parametrize("E,T,K,N,P,epw", [(4, 256, 256, 256, 4, 2), (3, 384, 128, 256, 2, 2), (6, 128, 512, 768, 8, 4)])
def test_moe_matches_oracle_both_orders(E, T, K, N, P, epw):
    x, w1, w2 = ms.make_inputs(E, T, K, N, seed=E + K, device="cpu")
    xd, w1d, w2d = x.cuda(), w1.cuda(), w2.cuda()
    rm, rows = ms.round_robin_row_map(E, T, P)
    tw = ms.expert_wave_tasks(E, T, N, epw)
    ti = ms.interleaved_tasks(E, T, N, epw)
    hw, dw = run(xd, w1d, w2d, tw, rm, rows, N)
    hi, di = run(xd, w1d, w2d, ti, rm, rows, N)
    href, dref = om.grouped_gemm_scatter(x, w1, w2, tw, rm, rows)
    compare(om.as_f64(hw), href, "h")
    for j, (a, b) in enumerate(zip(dw, dref)):
        compare(om.as_f64(a), b, f"dst {j}")
    assert torch.equal(hw.view(torch.int16), hi.view(torch.int16))
    for a, b in zip(dw, di):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_malformed_tasks_and_row_map_are_flagged_and_skipped():
    E, T, K, N, P = 2, 128, 128, 256, 2
    x, w1, w2 = ms.make_inputs(E, T, K, N, seed=3, device="cpu")
    rm, rows = ms.round_robin_row_map(E, T, P)
    tasks = ms.expert_wave_tasks(E, T, N, 2)
    bad = np.concatenate([tasks, np.array([[0, 5, 0, 0], [1, 0, 9, 0], [3, 0, 0, 0]], dtype=np.int32)])
    rm_bad = rm.copy()
    rm_bad[5] = (7 << 24) | 0  # rank 7 does not exist
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h, dst = run(x.cuda(), w1.cuda(), w2.cuda(), bad, rm_bad, rows, N, status)
    assert int(status.item()) == bd.EINVAL
    href, _ = om.grouped_gemm_scatter(x, w1, w2, tasks, rm, rows)
    compare(om.as_f64(h), href, "h with bad tasks skipped")
