"""Shared pieces of the GPU tests: guard-banded output partitions, error
metrics, and the oracle comparison of full or sampled outputs."""
from __future__ import annotations

import numpy as np
import torch

from attention_all_layout_gb300 import binding as bd
from oracle import attention as orc

SENTINEL = -12345.0  # exactly representable in bf16
GUARD = 256  # elements of guard band before and after each partition (16-byte multiple)

# Tolerances of the fused path against the float64 oracle: max-abs 2e-2 on
# top of the bf16 output format's own rounding (half a bf16 ulp of the exact
# value; the exact result rounded to bf16 already differs from it by up to that
# much, e.g. 0.029 at |O| = 8.16 in the joint preset), and relative
# Frobenius 1e-2.
MAX_ABS = 2e-2
REL_FRO = 1e-2


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def abs_tolerance(want: np.ndarray) -> np.ndarray:
    return MAX_ABS + half_ulp_bf16(want)


class GuardedPartitions:
    """P output partitions [B, c_j, H, d], each inside a buffer whose margins hold a sentinel."""

    def __init__(self, B, S, H, d, P, device="cuda"):
        self.buffers, self.parts = [], []
        for c in bd.chunk_sizes(S, P):
            n = B * c * H * d
            buf = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.bfloat16, device=device)
            self.buffers.append(buf)
            self.parts.append(buf[GUARD:GUARD + n].view(B, c, H, d))

    def guards_intact(self) -> bool:
        for buf in self.buffers:
            if not (torch.all(buf[:GUARD] == SENTINEL) and torch.all(buf[-GUARD:] == SENTINEL)):
                return False
        return True


def rel_fro(got: np.ndarray, want: np.ndarray) -> float:
    return float(np.linalg.norm((got - want).ravel()) / max(np.linalg.norm(want.ravel()), 1e-300))


def compare(got: np.ndarray, want: np.ndarray, what: str):
    """Max-abs and relative Frobenius error, asserted against the tolerances."""
    err = np.abs(got - want)
    mx = float(err.max()) if err.size else 0.0
    rf = rel_fro(got, want) if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if err.size:
        excess = err - abs_tolerance(want)
        i = np.unravel_index(int(np.argmax(excess)), err.shape)
        assert excess[i] <= 0, (f"{what}: |err| {err[i]:.3e} at |ref| {abs(want[i]):.3f} exceeds "
                                f"{MAX_ABS} + half bf16 ulp")
    assert rf <= REL_FRO, f"{what}: rel-Frobenius {rf:.3e} > {REL_FRO}"
    return mx, rf


def partitions_to_bhsd(parts) -> np.ndarray:
    """Reassemble device partitions into a float64 [B, H, S, d] array (test-side inverse)."""
    host = [orc.as_f64(p) for p in parts]
    return orc.seq_to_head(host)


def fused(q, k, v, P, scale, **kw):
    B, H, S, d = q.shape
    g = GuardedPartitions(B, S, H, d, P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.attn_a2a_fwd(q, k, v, P, scale, g.parts, dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return g
