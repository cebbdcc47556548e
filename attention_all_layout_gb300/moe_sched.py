"""Task lists and measurement for the synthetic MegaMoE-style workload
(moe_gemm_scatter). X-Stage pages, "Key Contributions", MegaMoE reshaping:
Expert-Wave runs each wave of experts' Linear-1 work, then its Linear-2 work,
so every SM stores at the same time; the interleaved scheduler mixes the next
wave's Linear-1 tiles with the current wave's Linear-2 tiles so that each
burst of stores has compute behind it.

Task = (kind, expert, row block, column block) for a 128 x 256 output tile; kind 0 = Linear-1-like
(output kept), kind 1 = Linear-2-like (output rows scattered to the ranks).
"""
from __future__ import annotations

import argparse
import json
import sys

import numpy as np
import torch

TILE_M, TILE_N = 128, 256  # output tile of one task


def _wave_tasks(kind, experts, T, N):
    return [(kind, e, m, n) for e in experts for m in range(T // TILE_M) for n in range(N // TILE_N)]


def expert_wave_tasks(E: int, T: int, N: int, experts_per_wave: int) -> np.ndarray:
    out = []
    for w0 in range(0, E, experts_per_wave):
        wave = range(w0, min(E, w0 + experts_per_wave))
        out += _wave_tasks(0, wave, T, N) + _wave_tasks(1, wave, T, N)
    return np.asarray(out, dtype=np.int32).reshape(-1, 4)


def interleaved_tasks(E: int, T: int, N: int, experts_per_wave: int) -> np.ndarray:
    waves = [range(w0, min(E, w0 + experts_per_wave)) for w0 in range(0, E, experts_per_wave)]
    out = _wave_tasks(0, waves[0], T, N)
    for i, wave in enumerate(waves):
        l2 = _wave_tasks(1, wave, T, N)
        l1 = _wave_tasks(0, waves[i + 1], T, N) if i + 1 < len(waves) else []
        for a in range(max(len(l2), len(l1))):
            if a < len(l2):
                out.append(l2[a])
            if a < len(l1):
                out.append(l1[a])
    return np.asarray(out, dtype=np.int32).reshape(-1, 4)


def round_robin_row_map(E: int, T: int, P: int):
    """Token row t of every expert goes to rank t mod P, in arrival order.
    Returns (row_map int32 [E*T] with (rank << 24) | slot, rows per rank)."""
    rank = np.tile(np.arange(T) % P, E)
    slot = np.zeros(E * T, dtype=np.int64)
    counts = np.zeros(P, dtype=np.int64)
    for i, r in enumerate(rank):
        slot[i] = counts[r]
        counts[r] += 1
    return ((rank.astype(np.int64) << 24) | slot).astype(np.int32), [int(c) for c in counts]


def make_inputs(E, T, K, N, seed=0, device="cuda"):
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn((E, T, K), generator=g, device=device).to(torch.bfloat16)
    w1 = (torch.randn((E, N, K), generator=g, device=device) / K**0.5).to(torch.bfloat16)
    w2 = (torch.randn((E, N, K), generator=g, device=device) / K**0.5).to(torch.bfloat16)
    return x, w1, w2


def time_orders(E=32, T=512, K=1024, N=512, P=8, experts_per_wave=None, reps=20):
    """CUDA-event time of the Expert-Wave and interleaved orders of the same tasks."""
    from . import binding as bd

    if experts_per_wave is None:  # one wave of Linear-1 tasks fills the GPU about once
        per_expert = (T // TILE_M) * (N // TILE_N)
        experts_per_wave = max(1, round(bd.num_sms() / per_expert))
    x, w1, w2 = make_inputs(E, T, K, N)
    rm, rows = round_robin_row_map(E, T, P)
    row_map = torch.from_numpy(rm).cuda()
    h = torch.empty((E, T, N), dtype=torch.bfloat16, device="cuda")
    dst = [torch.empty((r, N), dtype=torch.bfloat16, device="cuda") for r in rows]
    res = {"E": E, "T": T, "K": K, "N": N, "P": P, "experts_per_wave": experts_per_wave}
    for name, fn in (("expert_wave", expert_wave_tasks), ("interleaved", interleaved_tasks)):
        tasks = torch.from_numpy(fn(E, T, N, experts_per_wave)).cuda()
        call = lambda: bd.moe_gemm_scatter(x, w1, w2, tasks, h, row_map, dst)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[name + "_ms"] = ms
        res[name + "_tflops"] = 2.0 * 2 * E * T * N * K / (ms * 1e-3) / 1e12
    res["interleaved_speedup"] = res["expert_wave_ms"] / res["interleaved_ms"]
    return res


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    ap.add_argument("--shape", default=None, help="E,T,K,N: time this one problem instead of the K sweep")
    ap.add_argument("--reps", type=int, default=20)
    a = ap.parse_args(argv)
    if a.shape:
        E, T, K, N = (int(v) for v in a.shape.split(","))
        rows = [time_orders(E=E, T=T, K=K, N=N, reps=a.reps)]
    else:
        rows = [time_orders(K=K, reps=a.reps) for K in (128, 256, 512, 1024, 2048)]
    text = json.dumps(rows, indent=1)
    if a.out:
        with open(a.out, "w") as fh:
            fh.write(text)
    print(text)
    return 0


if __name__ == "__main__":
    sys.exit(main())
