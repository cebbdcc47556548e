"""CPU oracle of the synthetic MegaMoE-style grouped GEMM with scattered
outputs (test infrastructure only; shares no code with the CUDA path).

Definition (our own synthetic stand-in for the pages' MegaMoE
workload, X-Stage explanation, "Key Contributions", MegaMoE reshaping): for a
task (kind, e, m, n) the output tile is rows [128m, 128m+128) and columns
[256n, 256n+256) of x[e] @ w^T with w = w1[e] for kind 0 and w2[e] for kind
1; kind 0 tiles land in h[e] at the same rows and columns, kind 1 rows go to
dst[rank][slot] for row_map[e*T + row] = (rank << 24) | slot. float64 from
the exact upcast of the bf16 inputs.
"""
from __future__ import annotations

import numpy as np

from .attention import as_f64

TILE_N = 256  # output columns per task (the pages fix no tile size; this workload's task unit)


def grouped_gemm_scatter(x, w1, w2, tasks, row_map, dst_rows):
    x, w1, w2 = as_f64(x), as_f64(w1), as_f64(w2)
    tasks = np.asarray(tasks)
    row_map = np.asarray(row_map)
    E, T, K = x.shape
    N = w1.shape[1]
    h = np.zeros((E, T, N))
    dst = [np.zeros((r, N)) for r in dst_rows]
    for kind, e, m, n in tasks:
        rows = slice(128 * m, 128 * m + 128)
        cols = slice(TILE_N * n, TILE_N * n + TILE_N)
        w = w1 if kind == 0 else w2
        tile = x[e, rows] @ w[e, cols].T
        if kind == 0:
            h[e, rows, cols] = tile
        else:
            for i, r in enumerate(range(128 * m, 128 * m + 128)):
                rm = int(row_map[e * T + r])
                dst[rm >> 24][rm & 0xFFFFFF, cols] = tile[i]
    return h, dst
