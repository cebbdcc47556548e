"""CPU tests of the synthetic MegaMoE-style workload: the task-list builders
(both orders hold exactly the same tasks; waves are ordered as described) and
pins of its oracle (pure-Python brute force, identity and one-hot weights)."""
import numpy as np
import torch

from attention_all_layout_gb300 import moe_sched as ms
from oracle import moe as om


def test_orders_hold_the_same_tasks():
    for E, epw in ((8, 2), (5, 3), (4, 4)):
        a = ms.expert_wave_tasks(E, 256, 512, epw)
        b = ms.interleaved_tasks(E, 256, 512, epw)
        assert a.shape == b.shape == (E * 2 * 2 * 2, 4)
        assert sorted(map(tuple, a)) == sorted(map(tuple, b))
        assert len(set(map(tuple, a))) == len(a)


def test_expert_wave_groups_kinds_and_interleaved_alternates():
    a = ms.expert_wave_tasks(4, 128, 256, 2)
    assert [int(t[0]) for t in a] == [0, 0, 1, 1, 0, 0, 1, 1]
    b = ms.interleaved_tasks(4, 128, 256, 2)
    assert [(int(t[0]), int(t[1])) for t in b] == [(0, 0), (0, 1), (1, 0), (0, 2), (1, 1), (0, 3), (1, 2), (1, 3)]
    # tasks are 128 x 256 output tiles: N = 768 gives column blocks 0..2
    assert sorted({int(t[3]) for t in ms.expert_wave_tasks(1, 128, 768, 1)}) == [0, 1, 2]


def test_round_robin_row_map():
    rm, rows = ms.round_robin_row_map(2, 6, 4)
    assert rows == [4, 4, 2, 2]
    assert list(rm >> 24) == [0, 1, 2, 3, 0, 1, 0, 1, 2, 3, 0, 1]
    assert list(rm & 0xFFFFFF) == [0, 0, 0, 0, 1, 1, 2, 2, 1, 1, 3, 3]


def brute(x, w1, w2, tasks, rm, rows):
    E, T, K = x.shape
    N = w1.shape[1]
    h = [[[0.0] * N for _ in range(T)] for _ in range(E)]
    dst = [[[0.0] * N for _ in range(r)] for r in rows]
    for kind, e, m, n in tasks.tolist():
        w = w1 if kind == 0 else w2
        for r in range(128 * m, 128 * m + 128):
            for c in range(256 * n, 256 * n + 256):
                acc = sum(float(x[e, r, k]) * float(w[e, c, k]) for k in range(K))
                if kind == 0:
                    h[e][r][c] = acc
                else:
                    code = int(rm[e * T + r])
                    dst[code >> 24][code & 0xFFFFFF][c] = acc
    return np.array(h), [np.array(d) for d in dst]


def test_oracle_against_brute_force():
    g = torch.Generator().manual_seed(0)
    E, T, K, N, P = 2, 128, 3, 256, 2
    x = torch.randn((E, T, K), generator=g).to(torch.bfloat16)
    w1 = torch.randn((E, N, K), generator=g).to(torch.bfloat16)
    w2 = torch.randn((E, N, K), generator=g).to(torch.bfloat16)
    tasks = ms.interleaved_tasks(E, T, N, 1)
    rm, rows = ms.round_robin_row_map(E, T, P)
    h, dst = om.grouped_gemm_scatter(x, w1, w2, tasks, rm, rows)
    hb, db = brute(om.as_f64(x), om.as_f64(w1), om.as_f64(w2), tasks, rm, rows)
    np.testing.assert_allclose(h, hb, rtol=1e-12, atol=1e-12)
    for a, b in zip(dst, db):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_oracle_identity_and_one_hot_weights():
    E, T, K, N, P = 1, 128, 256, 256, 4
    x = torch.randn((E, T, K), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    eye = torch.eye(K).reshape(1, N, K).to(torch.bfloat16)
    tasks = ms.expert_wave_tasks(E, T, N, 1)
    rm, rows = ms.round_robin_row_map(E, T, P)
    h, dst = om.grouped_gemm_scatter(x, eye, eye, tasks, rm, rows)
    xs = om.as_f64(x)
    np.testing.assert_array_equal(h[0], xs[0])  # identity weights copy the rows
    for r in range(T):  # and the scatter sends row r to rank r mod P, slot r // P
        np.testing.assert_array_equal(dst[r % P][r // P], xs[0, r])
