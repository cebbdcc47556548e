"""CPU tests of the Ulysses multi-rank plan (attention_all_layout_gb300.ulysses):
which heads each rank computes, the destination rank and local row of every
output row against the oracle's chunk rule, the exchange of partition base
addresses with fake pointers, and - on gloo ranks (world size 2 and 3) - that
the ranks' head-group outputs, routed by the plan, assemble into the oracle's
partitions. The per-rank outputs here come from the oracle (test
infrastructure); the GPU side of a head-group call is tested in
tests/test_gpu_ulysses.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from attention_all_layout_gb300 import ulysses as ul
from attention_all_layout_gb300 import workloads
from oracle import attention as orc


def test_head_groups_partition_the_heads():
    for world in (1, 2, 4, 8):
        heads = []
        for r in range(world):
            p = ul.plan(r, world, 1, 40, 1000, 128)
            heads += list(range(p.h0, p.h1))
        assert heads == list(range(40))
    with pytest.raises(ValueError):
        ul.plan(0, 3, 1, 40, 1000, 128)  # 40 heads do not split over 3 ranks
    with pytest.raises(ValueError):
        ul.plan(2, 2, 1, 8, 100, 64)


@pytest.mark.parametrize("S,P", [(75600, 8), (1000, 3), (10, 4), (3, 8), (4096, 4)])
def test_destination_matches_oracle_chunk_rule(S, P):
    p = ul.plan(0, P, 1, 8 * P, S, 64)
    bounds = orc.chunk_bounds(S, P)
    assert p.chunks == bounds
    rows = range(S) if S <= 2000 else list(range(0, S, 97)) + [S - 1]
    for s in rows:
        j, l = p.destination(s)
        st, c = bounds[j]
        assert st <= s < st + c and l == s - st
        assert orc.rank_of_row(S, P, s) == (j, l)
    with pytest.raises(IndexError):
        p.destination(S)


def test_store_addresses_offset_to_the_head_group():
    B, H, S, d, P = 2, 8, 10, 64, 4  # chunks 3, 3, 2, 2
    bases = [0x10000 * (j + 1) for j in range(P)]
    for r in range(P):
        p = ul.plan(r, P, B, H, S, d)
        addrs = p.store_addresses(bases)
        assert addrs == [b + r * (H // P) * d * 2 for b in bases]
        assert all(a % 16 == 0 for a in addrs)
    # a chunk without rows gets no address
    p = ul.plan(1, 8, 1, 8, 3, 64)
    assert p.store_addresses([0x1000 * (j + 1) for j in range(8)])[3:] == [0] * 5


def test_exchange_bases_opens_every_peer_but_itself():
    handles = [f"h{j}" for j in range(4)]
    opened = []

    def open_peer(h):
        opened.append(h)
        return 0x100000 + int(h[1:]) * 0x1000

    got = ul.exchange_bases(7, open_peer, lambda obj: [7 if j == 2 else handles[j] for j in range(4)], rank=2)
    assert got == [0x100000, 0x101000, 7, 0x103000]
    assert opened == ["h0", "h1", "h3"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, cfg, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v = workloads.make_qkv(cfg, seed=5)
        p = ul.plan(rank, world, cfg.B, cfg.H, cfg.S, cfg.d)
        # bookkeeping: every rank learns every partition's base (fake addresses)
        def all_gather(obj):
            lst = [None] * world
            dist.all_gather_object(lst, obj)
            return lst

        bases = ul.exchange_bases(0x7000000 * (rank + 1), lambda h: h + 0x100, all_gather, rank)
        want = [0x7000000 * (j + 1) + (0x100 if j != rank else 0) for j in range(world)]
        assert bases == want, (bases, want)
        # this rank's head group, computed by the oracle: [B, H/P, S, d]
        o = orc.attention_fp64(q[:, p.h0:p.h1], k[:, p.h0:p.h1], v[:, p.h0:p.h1], cfg.scale)
        # route every output row to its destination rank by the plan
        send = []
        for j, (st, c) in enumerate(p.chunks):
            blk = np.zeros((cfg.B, c, p.heads_per_rank, cfg.d))
            for s in range(st, st + c):
                jj, l = p.destination(s)
                assert jj == j
                blk[:, l] = o[:, :, s]
            send.append(torch.from_numpy(blk).reshape(-1))
        recv = [torch.empty(cfg.B * p.chunks[rank][1] * p.heads_per_rank * cfg.d, dtype=torch.float64)
                for _ in range(world)]
        # the exchange (gloo has no all_to_all: point-to-point per peer)
        reqs = []
        for j in range(world):
            if j == rank:
                recv[j].copy_(send[j])
            else:
                reqs.append(dist.isend(send[j], j))
                reqs.append(dist.irecv(recv[j], j))
        for rq in reqs:
            rq.wait()
        # my partition: all heads of my chunk, head group i from rank i
        c = p.chunks[rank][1]
        part = np.zeros((cfg.B, c, cfg.H, cfg.d))
        for i in range(world):
            pi = ul.plan(i, world, cfg.B, cfg.H, cfg.S, cfg.d)
            part[:, :, pi.h0:pi.h1] = recv[i].numpy().reshape(cfg.B, c, pi.heads_per_rank, cfg.d)
        ref = orc.head_to_seq_partitions(orc.attention_fp64(q, k, v, cfg.scale), world)[rank]
        out[rank] = float(np.abs(part - ref).max())
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,S", [(2, 300), (3, 257)])
def test_ranks_assemble_oracle_partitions_gloo(world, S):
    cfg = workloads.AttnConfig("ulysses", B=2, H=2 * world, S=S, d=64, P=world)
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cfg, out)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=180)
        assert pr.exitcode == 0
    for r in range(world):
        assert out[r] == 0.0
