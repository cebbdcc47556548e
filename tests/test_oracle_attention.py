"""Pins for the attention + layout oracle, independent of the oracle's own code.

Each test checks the oracle against something the mathematics fixes: a
pure-Python brute force, closed forms, invariances of softmax attention, a
library routine (torch SDPA in float64, numpy/torch split rules), and the
inverse layout change. A dropped term, a wrong sign or index, a missing scale,
a softmax over the wrong axis or a transposed operand fails at least one.
"""
import math

import numpy as np
import pytest
import torch

from attention_all_layout_gb300 import workloads
from oracle import attention as orc


def brute_force(q, k, v, scale):
    """Triple loop over plain Python floats, straight from the definition."""
    B, H, S, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    out = [[[[0.0] * d for _ in range(S)] for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(S):
                scores = []
                for j in range(S):
                    acc = 0.0
                    for t in range(d):
                        acc += q[b][h][i][t] * k[b][h][j][t]
                    scores.append(scale * acc)
                m = max(scores)
                w = [math.exp(s - m) for s in scores]
                z = sum(w)
                for t in range(d):
                    out[b][h][i][t] = sum(w[j] * v[b][h][j][t] for j in range(S)) / z
    return np.array(out)


def rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("B,H,S,d,scale", [(1, 2, 7, 4, 0.5), (2, 1, 16, 8, 1 / math.sqrt(8)), (1, 1, 32, 3, 1.7)])
def test_brute_force(B, H, S, d, scale):
    q, k, v = rand((B, H, S, d), 1), rand((B, H, S, d), 2), rand((B, H, S, d), 3)
    want = brute_force(orc.as_f64(q).tolist(), orc.as_f64(k).tolist(), orc.as_f64(v).tolist(), scale)
    got = orc.attention_fp64(q, k, v, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_two_key_closed_form():
    # softmax over two keys is a logistic: w0 = 1/(1+exp(s1-s0)).
    q = np.array([[[[1.0, 2.0]]]])
    k = np.array([[[[0.5, -1.0], [2.0, 0.25]]]])
    v = np.array([[[[3.0, -1.0], [-2.0, 5.0]]]])
    scale = 0.75
    s0 = scale * (1.0 * 0.5 + 2.0 * -1.0)
    s1 = scale * (1.0 * 2.0 + 2.0 * 0.25)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    want = w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1]
    got = orc.attention_fp64(np.repeat(q, 1, axis=2), k, v, scale)[0, 0, 0]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_sdpa_float64_cross_check():
    q, k, v = rand((1, 3, 64, 16), 4), rand((1, 3, 64, 16), 5), rand((1, 3, 64, 16), 6)
    scale = 0.3
    want = torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double(), v.double(), scale=scale
    ).numpy()
    np.testing.assert_allclose(orc.attention_fp64(q, k, v, scale), want, rtol=1e-12, atol=1e-13)


def test_constant_v_gives_constant():
    q, k = rand((1, 2, 40, 8), 7, 3.0), rand((1, 2, 40, 8), 8, 3.0)
    v = torch.full((1, 2, 40, 8), 1.25, dtype=torch.bfloat16)
    np.testing.assert_allclose(orc.attention_fp64(q, k, v, 0.9), 1.25, rtol=0, atol=1e-14)


def test_zero_q_gives_mean_of_v():
    k, v = rand((1, 2, 33, 8), 9), rand((1, 2, 33, 8), 10)
    q = torch.zeros_like(k)
    out = orc.attention_fp64(q, k, v, 1.0)
    want = orc.as_f64(v).mean(axis=2, keepdims=True)
    np.testing.assert_allclose(out, np.broadcast_to(want, out.shape), rtol=0, atol=1e-14)


def test_scale_zero_gives_mean_of_v():
    q, k, v = rand((1, 1, 20, 4), 11), rand((1, 1, 20, 4), 12), rand((1, 1, 20, 4), 13)
    out = orc.attention_fp64(q, k, v, 0.0)
    np.testing.assert_allclose(out, np.broadcast_to(orc.as_f64(v).mean(axis=2, keepdims=True), out.shape), atol=1e-14)


def test_softmax_rows_sum_to_one():
    a = orc.as_f64(rand((50, 70), 14, 30.0))
    w = orc.softmax_rows(a)
    assert np.all(w >= 0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # the row maximum gets the largest weight in every row
    assert np.array_equal(w.argmax(axis=1), a.argmax(axis=1))


def test_one_hot_dominant_key():
    S, d = 24, 8
    k = torch.zeros(1, 1, S, d)
    k[0, 0, 5, 0] = 1.0
    q = torch.zeros(1, 1, S, d)
    q[0, 0, :, 0] = 200.0
    v = rand((1, 1, S, d), 15)
    out = orc.attention_fp64(q, k, v, 1.0)
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(orc.as_f64(v)[0, 0, 5], (S, d)), atol=1e-12)


def test_key_shift_and_permutation_invariance():
    q, k, v = rand((1, 1, 30, 8), 16), rand((1, 1, 30, 8), 17), rand((1, 1, 30, 8), 18)
    base = orc.attention_fp64(q, k, v, 0.6)
    # the same vector added to every key shifts each score row by a constant
    u = torch.randn(8, generator=torch.Generator().manual_seed(19)).double()
    shifted = orc.attention_fp64(q.double(), k.double() + u, v.double(), 0.6)
    np.testing.assert_allclose(shifted, base, rtol=1e-11, atol=1e-12)
    # permuting keys and values together leaves the output unchanged
    perm = torch.randperm(30, generator=torch.Generator().manual_seed(20))
    np.testing.assert_allclose(orc.attention_fp64(q, k[:, :, perm], v[:, :, perm], 0.6), base, atol=1e-13)


def test_large_scores_stay_finite():
    q, k, v = rand((1, 1, 16, 4), 21, 100.0), rand((1, 1, 16, 4), 22, 100.0), rand((1, 1, 16, 4), 23)
    out = orc.attention_fp64(q, k, v, 1.0)
    assert np.all(np.isfinite(out))


def test_rows_subset_matches_full():
    q, k, v = rand((1, 2, 48, 8), 24), rand((1, 2, 48, 8), 25), rand((1, 2, 48, 8), 26)
    full = orc.attention_fp64(q, k, v, 0.4)
    rows = [0, 5, 47, 13]
    np.testing.assert_allclose(orc.attention_rows_fp64(q, k, v, 0.4, 0, 1, rows), full[0, 1, rows], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("S,P", [(256, 2), (4096, 4), (4608, 8), (75600, 8), (200, 3), (7, 7), (10, 4)])
def test_chunk_bounds_match_array_split(S, P):
    bounds = orc.chunk_bounds(S, P)
    sizes = [len(a) for a in np.array_split(np.arange(S), P)]
    assert [c for _, c in bounds] == sizes
    assert [s for s, _ in bounds] == list(np.cumsum([0] + sizes[:-1]))


@pytest.mark.parametrize("B,H,S,d,P", [(1, 4, 12, 3, 2), (2, 3, 10, 2, 4), (1, 2, 9, 4, 3)])
def test_partitions_match_tensor_split(B, H, S, d, P):
    o = np.arange(B * H * S * d, dtype=np.float64).reshape(B, H, S, d)
    parts = orc.head_to_seq_partitions(o, P)
    want = torch.tensor_split(torch.from_numpy(o).permute(0, 2, 1, 3), P, dim=1)
    assert len(parts) == P
    for got, w in zip(parts, want):
        assert np.array_equal(got, w.numpy())


def test_partition_round_trip_and_p1_transpose():
    o = np.random.default_rng(0).standard_normal((2, 5, 23, 4))
    for P in (1, 2, 5, 8):
        assert np.array_equal(orc.seq_to_head(orc.head_to_seq_partitions(o, P)), o)
    (only,) = orc.head_to_seq_partitions(o, 1)
    assert np.array_equal(only, o.transpose(0, 2, 1, 3))


def test_rank_of_row():
    S, P = 75600, 8
    assert orc.rank_of_row(S, P, 0) == (0, 0)
    assert orc.rank_of_row(S, P, 9449) == (0, 9449)
    assert orc.rank_of_row(S, P, 9450) == (1, 0)
    assert orc.rank_of_row(S, P, S - 1) == (7, 9449)
    assert orc.rank_of_row(10, 4, 2) == (0, 2) and orc.rank_of_row(10, 4, 3) == (1, 0)


def test_workload_recipe_shapes_and_text_rows():
    cfg = workloads.config("joint", S=640, H=2)
    q, k, v = workloads.make_qkv(cfg, seed=0)
    assert q.shape == (1, 2, 640, 128) and q.dtype == torch.bfloat16
    for t in (q, k, v):
        text = t[:, :, :512].float().std().item()
        image = t[:, :, 512:].float().std().item()
        assert 1.9 < text < 2.1 and 0.9 < image < 1.1
    q2, _, _ = workloads.make_qkv(cfg, seed=0)
    assert torch.equal(q, q2)
