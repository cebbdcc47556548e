"""Ulysses sequence-parallel attention across P ranks: which heads a rank
computes, where each of its output rows goes, and the rank's fused call that
stores them there.

X-Stage pages, "Key Contributions" (FlashAttention-A2A: in Ulysses sequence
parallelism the post-attention all-to-all is fused into the attention
kernel, the owner of each output tile storing it to its destination) and
"Problem Statement" (device-initiated one-sided stores to another rank).

Layouts. Before attention (after the pre-attention exchange), rank r holds
heads [h0, h1) = [r*H/P, (r+1)*H/P) of q, k and v over the whole sequence:
[B, H/P, S, d]. After it, rank j holds sequence chunk j of every head:
partition j = [B, c_j, H, d], chunk sizes by the torch.tensor_split rule
(c_j = floor(S/P) + (j < S mod P)). Output row s of head h0 + h therefore
goes to rank j = chunk(s), local row s - start_j, head slot h0 + h.

Data path. Every rank's partition is mapped into every other rank's address
space (peer memory); `exchange_bases` collects the P base addresses through
the process group. Rank r then runs one fused call over its head group with
`part_heads = H`, the partition pointers offset to its first head
(`RankPlan.store_addresses`): its tile owners store straight into the
destination ranks' partitions with plain stores, no second pass. A partition
is complete when all P ranks' kernels have finished: each rank synchronises
its stream, then the ranks meet at a barrier.

The GPU side of one head-group call is the library's own (tests run the P
calls in turn on one GPU into shared partitions, which gives the same bytes as
one call over all heads). Opening another GPU's memory is the caller's
`open_peer`; nothing here calls CUDA's inter-process API.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Sequence


def chunk_sizes(S: int, P: int) -> list[int]:
    """Rows of each of the P sequence chunks (torch.tensor_split rule: larger chunks first)."""
    base, rem = divmod(S, P)
    return [base + (1 if j < rem else 0) for j in range(P)]


@dataclass(frozen=True)
class RankPlan:
    """Rank `rank` of `world` in one Ulysses attention layer of B, H, S, d."""

    rank: int
    world: int
    B: int
    H: int
    S: int
    d: int

    @property
    def heads_per_rank(self) -> int:
        return self.H // self.world

    @property
    def h0(self) -> int:
        return self.rank * self.heads_per_rank

    @property
    def h1(self) -> int:
        return self.h0 + self.heads_per_rank

    @property
    def chunks(self) -> list[tuple[int, int]]:
        """(start_j, c_j) of every destination rank's sequence chunk."""
        out, st = [], 0
        for c in chunk_sizes(self.S, self.world):
            out.append((st, c))
            st += c
        return out

    def destination(self, s: int) -> tuple[int, int]:
        """Destination rank and its local row of output sequence row s."""
        if not 0 <= s < self.S:
            raise IndexError(s)
        for j, (st, c) in enumerate(self.chunks):
            if s < st + c:
                return j, s - st
        raise AssertionError("unreachable")

    def partition_shape(self, j: int) -> tuple[int, int, int, int]:
        """Shape of rank j's output partition (all heads of its chunk)."""
        return (self.B, self.chunks[j][1], self.H, self.d)

    def store_addresses(self, part_bases: Sequence[int], elem_bytes: int = 2) -> list[int]:
        """Device addresses this rank's call stores to: every rank's partition
        base offset to this rank's first head (rows hold H heads of d values).
        Partitions without rows stay 0 (NULL)."""
        if len(part_bases) != self.world:
            raise ValueError("one partition base per rank")
        off = self.h0 * self.d * elem_bytes
        return [(int(b) + off) if c > 0 else 0 for b, (_, c) in zip(part_bases, self.chunks)]


def plan(rank: int, world: int, B: int, H: int, S: int, d: int) -> RankPlan:
    """The plan of one rank; H must split evenly over the ranks (head sharding)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank out of range")
    if H % world != 0:
        raise ValueError("H must be a multiple of the rank count")
    return RankPlan(rank, world, B, H, S, d)


def exchange_bases(local_handle, open_peer: Callable, all_gather: Callable, rank: int) -> list[int]:
    """Base addresses of every rank's partition in this rank's address space.

    Each rank publishes the handle of its own partition (`local_handle`);
    `all_gather(obj)` returns the list of every rank's object (e.g.
    torch.distributed.all_gather_object); `open_peer(handle)` maps another
    rank's partition and returns its address here. A rank's own partition is
    used as it is."""
    handles = all_gather(local_handle)
    return [int(h if j == rank else open_peer(h)) for j, h in enumerate(handles)]


def rank_forward(p: RankPlan, q, k, v, part_bases: Sequence[int], scale: float, dev_status=None,
                 stream=None, store_kind: int = 0) -> int:
    """This rank's fused call: its head group (q, k, v [B, H/P, S, d], bf16,
    head dim contiguous) into every rank's partition. Asynchronous on `stream`."""
    from . import binding as bd

    if tuple(q.shape) != (p.B, p.heads_per_rank, p.S, p.d):
        raise ValueError("q must be this rank's head group [B, H/P, S, d]")
    return bd.attn_a2a_fwd(q, k, v, p.world, scale, p.store_addresses(part_bases), dev_status=dev_status,
                           stream=stream, store_kind=store_kind, part_heads=p.H)
