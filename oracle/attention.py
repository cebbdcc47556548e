"""CPU oracle for fused attention + post-attention Ulysses all-to-all layout.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, links or runs
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it. It shares no code with the CUDA path.

What it follows (X-Stage: An Overlooked Pipeline Stage for
Communication-Computation Overlap in DiT Inference, gist.science explanation):

* "Key Contributions", FlashAttention-A2A (piggybacking) item: in Ulysses-style
  sequence-parallel attention the post-attention all-to-all is fused into
  FlashAttention; the owner of each output tile stores it to its destination
  and resumes the Q loop. The fusion changes when the bytes move, not what is
  computed, so the result is the plain definition written out below:

  1. attention per batch b and head h (non-causal, no bias, no dropout):
       A = scale * Q[b,h] @ K[b,h]^T            (S x S)
       W = exp(A - rowmax(A)) / rowsum(...)     (row-wise softmax)
       O[b,h] = W @ V[b,h]                      (S x d)
  2. the post-attention all-to-all (head-sharded -> sequence-sharded): rank j
     ends up with sequence chunk j for every head,
       part_j[b, l, h, :] = O[b, h, start_j + l, :]   for 0 <= l < c_j.

Readings where the pages are silent: non-causal attention with one scale
(1/sqrt(d) in the presets); the same head count for Q, K, V; chunks of a
sequence that P does not divide follow the tensor_split convention (the first
S mod P chunks hold one extra row); partitions are laid out [B, c_j, H, d].

Arithmetic is float64 from the exact upcast of the bf16 input bits. The matrix
products are numpy matmuls (a library primitive); nothing is blocked, fused or
reordered beyond the definition: rows are computed independently, exactly as
the definition states, so a subset of rows is the definition restricted to
those rows.
"""
from __future__ import annotations

import numpy as np


def as_f64(x) -> np.ndarray:
    """Exact float64 copy of a bf16/fp32 torch tensor or array-like.

    bf16 -> fp32 -> fp64 is exact (both widenings keep every bit of the value).
    """
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    return np.asarray(x, dtype=np.float64)


def chunk_bounds(S: int, P: int) -> list[tuple[int, int]]:
    """(start_j, c_j) of the P sequence chunks; the first S mod P get one more row."""
    if P < 1:
        raise ValueError("P must be >= 1")
    base, rem = divmod(S, P)
    out, start = [], 0
    for j in range(P):
        c = base + (1 if j < rem else 0)
        out.append((start, c))
        start += c
    return out


def softmax_rows(a: np.ndarray) -> np.ndarray:
    """Row-wise softmax of a float64 matrix, max-subtracted."""
    a = a - a.max(axis=-1, keepdims=True)
    e = np.exp(a)
    return e / e.sum(axis=-1, keepdims=True)


def attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q k^T) v for one head: q [Sq,d], k [S,d], v [S,d] -> [Sq,d]."""
    a = scale * (q @ k.T)
    return softmax_rows(a) @ v


def attention_fp64(q, k, v, scale: float) -> np.ndarray:
    """O[b,h] = softmax(scale Q K^T) V for every (b, h); inputs [B,H,S,d]."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, H, S, d = q.shape
    out = np.empty((B, H, S, v.shape[-1]), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            out[b, h] = attention_head(q[b, h], k[b, h], v[b, h], scale)
    return out


def attention_rows_fp64(q, k, v, scale: float, b: int, h: int, rows) -> np.ndarray:
    """The definition restricted to query rows ``rows`` of head (b, h): [len(rows), d]."""
    rows = np.asarray(rows, dtype=np.int64)
    qb = as_f64(q[b, h])[rows]
    return attention_head(qb, as_f64(k[b, h]), as_f64(v[b, h]), scale)


def head_to_seq_partitions(o: np.ndarray, P: int) -> list[np.ndarray]:
    """Post-attention all-to-all: [B,H,S,d] -> P partitions [B, c_j, H, d].

    Written as the explicit element-row loop of the definition,
    part_j[b, l, h, :] = O[b, h, start_j + l, :].
    """
    B, H, S, d = o.shape
    parts = []
    for start, c in chunk_bounds(S, P):
        part = np.empty((B, c, H, d), dtype=o.dtype)
        for b in range(B):
            for l in range(c):
                for h in range(H):
                    part[b, l, h, :] = o[b, h, start + l, :]
        parts.append(part)
    return parts


def seq_to_head(parts: list[np.ndarray]) -> np.ndarray:
    """Inverse layout change: P partitions [B, c_j, H, d] -> [B, H, S, d]."""
    B, _, H, d = parts[0].shape
    S = sum(p.shape[1] for p in parts)
    o = np.empty((B, H, S, d), dtype=parts[0].dtype)
    start = 0
    for part in parts:
        c = part.shape[1]
        for b in range(B):
            for l in range(c):
                for h in range(H):
                    o[b, h, start + l, :] = part[b, l, h, :]
        start += c
    return o


def rank_of_row(S: int, P: int, s: int) -> tuple[int, int]:
    """(destination rank j, local row l) of global sequence row s."""
    for j, (start, c) in enumerate(chunk_bounds(S, P)):
        if start <= s < start + c:
            return j, s - start
    raise IndexError(s)
