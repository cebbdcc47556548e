#!/usr/bin/env python3
"""Benchmark of the fused attention + post-attention all-to-all hot path.

One step = one call of the fused kernel (attention forward with the
head-to-sequence all-to-all stored by the tile owners) over one batch of the
video DiT workload (B=1, H=40, S=32768, d=128, P=8 virtual ranks), inputs
resident in HBM (1.0 GB of q, k, v: larger than L2, so no flush is needed).

Prints one JSON line. Legs:
  value        device-timed fused call, TFLOP/s = 4*B*H*S^2*d / time
  e2e          the host-memory C-ABI call (pinned host q, k, v copied to the
               device, fused kernels whose tile owners store the output rows
               straight into the pinned host partitions) timed end to end;
               d2h_bytes_per_step counts the output those stores carry
  roofline     the fused kernel against the measured bf16 tensor peak
  cpu_baseline the float64 oracle on a bounded row sample, on host cores
  attention-alone, serial (attention, then a separate permute) and whole-layer
               times, taken in turns with the fused call over three rounds
  other_presets_fused  the fused call on the image, joint and long presets
               (CUDA events; context, not the headline): image and joint
               before the headline, long after every other leg
`--impl reference` times the oracle arm instead (CPU, rank 0 only).
Multi-GPU (torchrun): every rank runs an independent replica of the workload
(no data-path collective); value is the sum over ranks / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused attn+A2A-layout TFLOP/s and % of bf16 dense tensor peak, 1 GB300"
WORKLOAD = "video DiT attention + Ulysses post-attention A2A layout: B=1, H=40, S=32768, d=128, P=8 virtual ranks"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
KERNEL_SOURCES = ["fa_tc.cuh", "ptx.cuh", "epilogue.cuh", "tmem_ops.cuh", "fa_tc.cu", "fa_tc_launch.cuh",
                  "fa_tc_split.cu"]


def device_split_plan(cfg):
    """How a call with a workspace and the automatic split divides cfg's work items on this
    GPU (the library's own decision, attn_a2a_split_plan): "all" (every item's key blocks in
    equal ranges, one kernel), "tail" (the partial last wave's, in a second kernel) or None."""
    from attention_all_layout_gb300 import binding as bd

    kind, _, _ = bd.attn_a2a_split_plan(cfg.B, cfg.H, cfg.S, cfg.d)
    return {bd.SPLIT_ALL: "all", bd.SPLIT_TAIL: "tail"}.get(kind)


def fused_kernel_label(cfg, split: bool) -> str:
    """The kernel instantiation the fused call launches for cfg (the ncu name)."""
    from attention_all_layout_gb300 import binding as bd

    bulk = bd.attn_a2a_store_kind(cfg.S, cfg.P, 1) == 1
    plan = device_split_plan(cfg) if split else None
    what = {"tail": ", split tail", "all": ", whole schedule split", None: ""}[plan]
    return (f"fa_fwd_tc_kernel<{cfg.d}, {3 if bulk else 1}, 1, false, {'true' if plan else 'false'}> "
            f"(all-to-all layout, {'bulk-store' if bulk else 'row-store'} epilogue{what})")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and whitespace: what the compiler sees."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_hash() -> str:
    """Hash of the fused kernel's code (comments and whitespace excluded), so a
    recorded ncu traffic figure is reused only for the kernel it was taken on."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "attention_all_layout_gb300", "csrc", name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu summary, if current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_hash") != kernel_hash():
        return None
    return rec.get("dram_bytes_per_launch_full_workload")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1]
        if not rows:  # a short region: take the samples nearest to it
            rows = [s for (t, s) in self.samples if t0 - 0.3 <= t <= t1 + 0.3]
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 7:
                continue
            try:
                mhz.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def _starts(S: int, P: int):
    base, rem = divmod(S, P)
    out, st = [], 0
    for j in range(P):
        out.append(st)
        st += base + (1 if j < rem else 0)
    return out


def max_over_ranks(ms: float, world: int, device) -> float:
    """Slowest rank's time: the job finishes when its last replica does."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: the work of every replica over the slowest rank's time."""
    return flops_per_rank * world / (max_ms * 1e-3) / 1e12


def time_events(fn, steps, warmup, stream):
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def cpu_oracle_sample(q, k, v, cfg, rows_per_head: int, heads: int, seed: int):
    """Times the float64 oracle on `rows_per_head` query rows of `heads` heads."""
    import numpy as np
    import torch

    from oracle import attention as orc

    gen = torch.Generator().manual_seed(seed)
    t_total, n_rows = 0.0, 0
    for h in range(heads):
        rows = torch.randint(0, cfg.S, (rows_per_head,), generator=gen).tolist()
        qh = q[0, h][rows].cpu()
        kh, vh = k[0, h].cpu(), v[0, h].cpu()
        t0 = time.perf_counter()
        out = orc.attention_head(orc.as_f64(qh), orc.as_f64(kh), orc.as_f64(vh), cfg.scale)
        for r in rows:  # the layout change of these rows
            orc.rank_of_row(cfg.S, cfg.P, r)
        t_total += time.perf_counter() - t0
        n_rows += len(rows)
        assert np.all(np.isfinite(out))
    flops = 4.0 * cfg.S * cfg.d * n_rows
    return flops / t_total / 1e12, n_rows, t_total


def reference_arm(args):
    """The oracle as it stands, timed on host cores (rank 0 only)."""
    import numpy as np

    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch

    from attention_all_layout_gb300 import workloads
    from oracle import attention as orc

    cfg = workloads.CONFIGS[args.config]
    cores = os.cpu_count() or 1
    torch.set_num_threads(cores)
    rows_per_head, heads = 64, min(cfg.H, 8)
    gen = torch.Generator().manual_seed(0)

    def draw(shape):
        return torch.randn(shape, generator=gen).to(torch.bfloat16)

    kh = [orc.as_f64(draw((cfg.S, cfg.d))) for _ in range(heads)]
    vh = [orc.as_f64(draw((cfg.S, cfg.d))) for _ in range(heads)]
    qh = [orc.as_f64(draw((rows_per_head, cfg.d))) for _ in range(heads)]

    def step():
        for h in range(heads):
            out = orc.attention_head(qh[h], kh[h], vh[h], cfg.scale)
            assert np.isfinite(out).all()

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    flops = 4.0 * cfg.S * cfg.d * rows_per_head * heads
    value = flops / dt / 1e12
    sample = (f"{rows_per_head} query rows x {heads} heads per step of the {cfg.name} config "
              f"(full key length {cfg.S}), float64 numpy oracle; TFLOP/s = 4*S*d per row / time")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD if cfg.name == "video" else cfg.name, "B": cfg.B, "H": cfg.H,
                   "S": cfg.S, "d": cfg.d, "P": cfg.P},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="video")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-only", action="store_true",
                    help="time only the fused call (no attention-alone, serial or e2e legs); for profiling")
    ap.add_argument("--H", type=int, default=None, help="override the head count (smaller profiling cases)")
    ap.add_argument("--S", type=int, default=None, help="override the sequence length (smaller profiling cases)")
    ap.add_argument("--no-presets", action="store_true", help="skip timing the image, joint and long presets")
    ap.add_argument("--no-split", action="store_true",
                    help="no split-tail workspace: a partial last wave of work items leaves CTAs idle")
    ap.add_argument("--cta-pairs", action="store_true",
                    help="with --fused-only: run the fused call on CTA pairs (cta_group::2 MMAs), no split")
    args = ap.parse_args()
    if args.cta_pairs and not args.fused_only:
        ap.error("--cta-pairs times the fused call alone: give --fused-only too")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)

    import torch

    from attention_all_layout_gb300 import binding as bd
    from attention_all_layout_gb300 import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    bd.load()
    cfg = workloads.CONFIGS[args.config]
    overrides = {k: v for k, v in (("H", args.H), ("S", args.S)) if v is not None}
    if overrides:
        cfg = workloads.config(args.config, name=f"{args.config}_" + "_".join(f"{k}{v}" for k, v in overrides.items()),
                               **overrides)
    stream = torch.cuda.current_stream()

    q, k, v = workloads.make_qkv(cfg, seed=rank, device="cuda")
    parts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    o = torch.empty((cfg.B, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # split-tail workspace (a partial last wave of work items is divided over all CTAs)
    ws = None if args.no_split or args.cta_pairs else bd.alloc_workspace(cfg.d)
    pairs = bd.PAIRS_ON if args.cta_pairs else bd.PAIRS_AUTO

    def fused():
        bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, parts, dev_status=status, stream=stream, workspace=ws,
                        cta_pairs=pairs)

    def contig():
        bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o, dev_status=status, stream=stream, workspace=ws)

    def serial():
        contig()
        bd.attn_a2a_permute(o, cfg.P, parts, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    time.sleep(0.3)
    # ---- the other presets' fused call (context beside the headline; not the
    # metric). The short ones (image, joint: milliseconds of work) first, so
    # that they are not timed at the clock the long legs leave behind
    presets = {}

    def time_preset(name, when):
        pc = workloads.CONFIGS[name]
        pq, pk, pv = workloads.make_qkv(pc, seed=rank, device="cuda")
        pparts = bd.alloc_partitions(pc.B, pc.S, pc.H, pc.d, pc.P)
        pws = None if args.no_split else bd.alloc_workspace(pc.d)
        n = 50 if pc.flops < 1e12 else 5
        # median of three windows
        pms = statistics.median(
            time_events(lambda: bd.attn_a2a_fwd(pq, pk, pv, pc.P, pc.scale, pparts, dev_status=status,
                                                stream=stream, workspace=pws), n, 3, stream) for _ in range(3))
        l2_note = ("back to back, no flush: q,k,v and the output (%.0f MB) fit in the 129 MB L2, so calls after "
                   "the first find them there" % ((pc.qkv_bytes + pc.qkv_bytes / 3) / 1e6)
                   if pc.qkv_bytes * 4 / 3 < 129e6 else
                   "no flush: q,k,v inputs (%.2f GB) exceed the 129 MB L2" % (pc.qkv_bytes / 1e9))
        presets[name] = {"ms": pms, "tflops": pc.flops / (pms * 1e-3) / 1e12, "steps": n, "timed": when,
                         "l2": l2_note, "shape": {"B": pc.B, "H": pc.H, "S": pc.S, "d": pc.d, "P": pc.P}}
        del pq, pk, pv, pparts, pws
        torch.cuda.empty_cache()

    if cfg.name == "video" and not args.no_presets and not args.fused_only:
        for name in ("image", "joint"):
            time_preset(name, "before the headline")
    # ---- headline: the fused call, inputs resident in HBM
    for _ in range(args.warmup):
        fused()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        fused()
    e1.record(stream)
    barrier()
    t_wall1 = time.time()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, "cuda")
    clocks = sampler.summary(t_wall0, t_wall1)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the timed region")

    if args.fused_only:
        sampler.stop()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": cfg.flops / (ms * 1e-3) / 1e12 * world,
                              "unit": "TFLOP/s", "ms_per_step": ms, "steps": args.steps,
                              "config": {"workload": cfg.name, "B": cfg.B, "H": cfg.H, "S": cfg.S,
                                         "d": cfg.d, "P": cfg.P,
                                         "split": device_split_plan(cfg) if ws is not None else None,
                                         "cta_pairs": bool(args.cta_pairs)},
                              "clocks": clocks, "fused_only": True}),
                  flush=True)
        return 0
    # ---- comparison legs, taking turns over three rounds (median per leg), so
    # that a clock drift under the power cap does not favour the leg timed
    # first: the fused call again, attention alone and the serial baseline
    # (same kernel, contiguous epilogue, then the separate permute), and the
    # whole Ulysses layer (sequence-sharded q, k, v in: the pre-attention
    # exchange folded into the loads; sequence-sharded output out)
    legs = {
        "fused": fused,
        "contig": contig,
        "permute": lambda: bd.attn_a2a_permute(o, cfg.P, parts, stream=stream),
        "serial": serial,
    }
    if cfg.P <= 8:
        sq, sk, sv = ([t[:, :, st:st + c].permute(0, 2, 1, 3).contiguous()
                       for st, c in zip(_starts(cfg.S, cfg.P), bd.chunk_sizes(cfg.S, cfg.P))] for t in (q, k, v))
        legs["s2s"] = lambda: bd.attn_a2a_fwd_s2s(sq, sk, sv, cfg.P, cfg.scale, parts, dev_status=status,
                                                  stream=stream, workspace=ws)
    turns = {name: [] for name in legs}
    for _ in range(3):
        for name, fn in legs.items():
            turns[name].append(time_events(fn, max(5, args.steps // 3), 1, stream))
    med = {name: statistics.median(v) for name, v in turns.items()}
    ms_turns, ms_contig, ms_permute, ms_serial = med["fused"], med["contig"], med["permute"], med["serial"]
    ms_s2s = med.get("s2s")
    if cfg.P <= 8:
        del sq, sk, sv

    # ---- e2e: host buffers through the C-ABI host entry point
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    dparts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P)
    hparts = [torch.empty(p.shape, dtype=p.dtype).pin_memory() for p in dparts]

    def e2e_step():
        bd.attn_a2a_fwd_host(hq, hk, hv, cfg.P, cfg.scale, dq, dk, dv, dparts, hparts,
                             dev_status=status, stream=stream)

    e2e_steps = max(3, args.steps // 3)
    for _ in range(2):
        e2e_step()
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    f1.record(stream)
    barrier()
    ms_e2e = f0.elapsed_time(f1) / e2e_steps
    # ---- the output partitions in host memory: the tile owners store every row
    # straight into the host's partitions over the host link (whole-line row
    # stores), against attention alone, the permute and a copy of the device
    # partitions to the host (context: the remote-destination case; not the metric)
    haddr = [t.data_ptr() if t.numel() else 0 for t in hparts]

    def copy_back():
        with torch.cuda.stream(stream):
            for a, b_ in zip(hparts, dparts):
                a.copy_(b_, non_blocking=True)

    def serial_to_host():
        contig()
        bd.attn_a2a_permute(o, cfg.P, dparts, stream=stream)
        copy_back()

    host_legs = {"fused": lambda: bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, haddr, dev_status=status,
                                                  stream=stream, store_kind=3),
                 "serial": serial_to_host}
    host_turns = {name: [] for name in host_legs}
    for _ in range(3):
        for name, fn in host_legs.items():
            host_turns[name].append(time_events(fn, 3, 1, stream))
    host_med = {name: statistics.median(v) for name, v in host_turns.items()}
    host_dest = {"fused_into_host_ms": host_med["fused"], "serial_to_host_ms": host_med["serial"],
                 "speedup_vs_serial": host_med["serial"] / host_med["fused"], "store_kind": 3,
                 "serial": "attention alone, permute, copy of the partitions to pinned host memory"}
    del hq, hk, hv, dq, dk, dv, dparts, hparts

    # ---- the long preset, last: seconds of full load that would heat the headline
    if cfg.name == "video" and not args.no_presets:
        time_preset("long", "after the other legs")
    sampler.stop()

    peaks, peak_src = load_peaks()
    flops = cfg.flops
    tflops = flops / (ms * 1e-3) / 1e12
    total_value = job_throughput(flops, world, ms)
    peak = peaks["bf16_tflops"]
    traffic = recorded_traffic()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        torch.set_num_threads(cores)
        # a bounded sample: about 10-15 s of float64 work on the host's cores
        rows_per_head = 1024
        val, nrows, secs = cpu_oracle_sample(q, k, v, cfg, rows_per_head=rows_per_head, heads=cfg.H, seed=0)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{nrows} query rows ({rows_per_head} random rows x {cfg.H} heads) of this workload at full key "
                         f"length, float64 numpy oracle incl. the row's layout destination; "
                         f"{secs:.1f} s of CPU work; TFLOP/s = 4*S*d per row / time"}
    line = {
        "metric": METRIC,
        "value": total_value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if cfg.name == "video" else cfg.name, "B": cfg.B, "H": cfg.H,
                   "S": cfg.S, "d": cfg.d, "P": cfg.P,
                   "l2": "no flush: q,k,v inputs (%.2f GB) exceed the 129 MB L2" % (cfg.qkv_bytes / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU, P virtual ranks",
                   "split": device_split_plan(cfg) if ws is not None else None},
        "pct_of_bf16_peak": 100.0 * tflops / peak,
        "pct_of_bf16_peak_sustained": 100.0 * tflops / peaks.get("bf16_tflops_sustained", peak),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "traffic": traffic,
                     "kernel": fused_kernel_label(cfg, ws is not None),
                     "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "fused_in_turns_ms": ms_turns,
        "attention_alone_ms": ms_contig,
        "permute_ms": ms_permute,
        "serial_ms": ms_serial,
        "epilogue_overhead": ms_turns / ms_contig - 1.0,
        "speedup_vs_serial": ms_serial / ms_turns,
        "ulysses_layer_s2s_ms": ms_s2s,
        "ulysses_layer_s2s_tflops": (flops / (ms_s2s * 1e-3) / 1e12) if ms_s2s else None,
        "e2e": {"value": flops / (ms_e2e * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "h2d_bytes_per_step": cfg.qkv_bytes, "d2h_bytes_per_step": cfg.out_bytes,
                "ms_per_step": ms_e2e},
        "clocks": clocks,
        # the split tail runs as a second kernel behind the first one
        "gpu_launches": args.steps * (2 if ws is not None and device_split_plan(cfg) == "tail" else 1),
        "cpu_baseline": cpu,
        "other_presets_fused": presets or None,
        "host_destination": host_dest,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
