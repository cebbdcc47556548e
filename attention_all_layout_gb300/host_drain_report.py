"""The fused call storing its output partitions into host memory: a
destination behind a link far slower than the GPU's own memory, the regime
in which the X-Stage pages' Burst-Gap equation predicts a cost the issuer
sees (Technical Summary, "Methodology": T_iss = max(T0, V/R - G), R the drain
rate of the path downstream of the stores; "Problem Statement": one-sided
stores from the tile owner into memory across a link; "Results": the fused
kernel's gains over attention followed by a separate all-to-all, largest at
short sequences).

On a system with one GPU, the host's memory, which the GPU stores to over
the host link (NVLink-C2C on GB300 systems), stands in for a peer GPU's
memory: the tile owners store every output row straight into the host-side
partition where it belongs (whole-line row stores, store_kind 3), while the
next tiles compute.

1. Probe fits with the burst destination in pinned host memory: contiguous
   lines (probe store_kind 0) and scattered whole rows (store_kind 2, the
   epilogue's pattern), idle gaps, each with held-out residuals.
2. Per workload, legs taking turns over several rounds (median per leg):
   fused into host partitions (fh), the same with a workspace so that the
   library's automatic split schedule applies (fhs: where it splits, CTAs
   finish their tiles at staggered times instead of in waves), the same with
   every item's key blocks split into equal ranges whatever the automatic
   choice (fha), the same into device partitions (fd),
   attention alone into device memory (c), the separate permute (p), and the
   copy of the device partitions to the host (x, one contiguous copy per
   partition). Serial baseline = c + p + x; fused then copy = fd + x. And one
   Ulysses rank's view: its own partition in device memory, the other P - 1 in
   host memory, automatic store kind (fr), against c + p + the copy of the
   P - 1 partitions (xr). The host partitions are checked byte for byte
   against the device ones.
3. The equation's prediction of fh, per wave of work items (all CTAs finish
   an item together; the last wave may be partial): the wave's stores,
   V_w = items_w * 2 * 128 * 2d bytes, cost the issuers max(0, V_w/R - G)
   beyond what a fast destination costs, G = one item's compute time
   (attention alone / waves), never less than the link bound (all output
   bytes / R). Next to it the two counterfactuals: completion-coupled (every
   wave also waits V_w/R) and unbounded-asynchronous (no cost; only the link
   bound). Two values of R: the probe's scattered-row fit, and the drain rate
   the fused call itself reaches at the shortest sequence (where its time is
   all drain), used to predict the other workloads.
4. Traced calls into the host partitions: the per-tile store spans (first warp
   starting to issue a tile's stores to the last warp resuming).

Usage: python -m attention_all_layout_gb300.host_drain_report [--out FILE] [--quick]
"""
from __future__ import annotations

import argparse
import json
import sys

import torch

from . import binding as bd
from . import probe_sweep as ps
from . import tile_trace as tt
from . import workloads

S_LIST = (1024, 2048, 4096, 8192, 16384, 32768)
PRESETS = ("image", "joint")
ROUNDS = 3
PROBE_V_MB = (2, 4, 8, 16, 32, 64)
PROBE_G_US = (0, 5, 10, 20, 40, 100, 200, 400)


def time_ms(fn, n):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def probe_fit(kind: int, host: bool = True, quick: bool = False, seed: int = 0) -> dict:
    """Probe sweep into pinned host memory (or device memory), fitted on a
    calibration split; returns R, Q, the T0 table and the held-out residuals."""
    K = bd.num_sms()
    vs = PROBE_V_MB if not quick else (4, 16, 64)
    gs = PROBE_G_US if not quick else (0, 10, 40, 100, 400)
    dst_bytes = (4 * max(vs) * 2**20 // (4096 * K) + 1) * 4096 * K
    pr = ps.Prober(dst_bytes, K * 16 * 3, host=host)
    pts = [pr.run(K, ps.round_volume(v * 2**20, K), g * 1000, 16, store_kind=kind, discard=8) for v in vs for g in gs]
    f, held = ps.split_fit(pts, seed=seed, g_max=max(gs) * 1e-6)
    return {"kind": kind, "host": host, "R_GBps": f.R / 1e9, "Q_MB": None if f.Q is None else f.Q / 2**20,
            "T0_us": {f"{V / 2**20:.1f}": t * 1e6 for (_k, V, _kd), t in sorted(f.T0.items())},
            "heldout": held, "points": [{"V_MB": p.V / 2**20, "G_us": p.G * 1e6, "t_iss_us": p.t_iss_med * 1e6}
                                        for p in pts]}


def waves_of(items: int, n_sm: int) -> list[int]:
    """Items in each wave of a persistent grid of n_sm CTAs."""
    full, rest = divmod(items, n_sm)
    return [n_sm] * full + ([rest] if rest else [])


def predict(fd_ms: float, c_ms: float, items: int, n_sm: int, v_item: int, out_bytes: int, R: float) -> dict:
    """Burst-Gap prediction of the fused call into the slow destination, and
    the two counterfactuals, in ms."""
    waves = waves_of(items, n_sm)
    g = c_ms * 1e-3 / len(waves)  # one item's compute time
    burst_gap = sum(max(0.0, w * v_item / R - g) for w in waves)
    coupled = sum(w * v_item / R for w in waves)
    link = out_bytes / R
    return {"burst_gap_ms": max(fd_ms + burst_gap * 1e3, link * 1e3),
            "completion_coupled_ms": fd_ms + coupled * 1e3,
            "unbounded_async_ms": max(fd_ms, link * 1e3),
            "waves": len(waves), "gap_item_us": g * 1e6, "burst_MB": waves[0] * v_item / 2**20}


def measure(cfg, R: float, n_sm: int, trace: bool = True) -> dict:
    q, k, v = workloads.make_qkv(cfg, seed=0, device="cuda")
    dparts = bd.alloc_partitions(cfg.B, cfg.S, cfg.H, cfg.d, cfg.P, fill=0.0)
    hparts = [torch.zeros(t.shape, dtype=t.dtype, pin_memory=True) for t in dparts]
    haddr = [t.data_ptr() if t.numel() else 0 for t in hparts]
    o = torch.empty((cfg.B, cfg.H, cfg.S, cfg.d), dtype=torch.bfloat16, device="cuda")
    # same bytes in the host partitions as in the device ones
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, dparts, store_kind=3)
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, haddr, store_kind=3)
    torch.cuda.synchronize()
    same = all(torch.equal(a.view(torch.int16), b.cpu().view(torch.int16)) for a, b in zip(hparts, dparts))
    own = dparts[0].clone()
    for t in hparts:
        t.zero_()
    dparts[0].zero_()
    bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, [dparts[0].data_ptr()] + haddr[1:])
    torch.cuda.synchronize()
    same = same and torch.equal(own.view(torch.int16), dparts[0].view(torch.int16)) and all(
        torch.equal(a.view(torch.int16), b.cpu().view(torch.int16)) for a, b in zip(hparts[1:], dparts[1:]))

    def copy_back():
        for a, b in zip(hparts, dparts):
            a.copy_(b, non_blocking=True)

    # one Ulysses rank's view: its own partition in device memory, the other
    # P - 1 (the other ranks') in host memory; the automatic store kind
    raddr = [dparts[0].data_ptr()] + haddr[1:]

    def copy_back_remote():
        for a, b in zip(hparts[1:], dparts[1:]):
            a.copy_(b, non_blocking=True)

    ws = bd.alloc_workspace(cfg.d)
    legs = {
        "fh": lambda: bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, haddr, store_kind=3),
        "fhs": lambda: bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, haddr, store_kind=3, workspace=ws),
        "fha": lambda: bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, haddr, store_kind=3, workspace=ws,
                                       split=bd.SPLIT_ALL),
        "fd": lambda: bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, dparts, store_kind=3),
        "c": lambda: bd.attn_a2a_fwd_contig(q, k, v, cfg.scale, o),
        "p": lambda: bd.attn_a2a_permute(o, cfg.P, dparts),
        "x": copy_back,
        "fr": lambda: bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, raddr),
        "xr": copy_back_remote,
    }
    n = max(3, min(50, int(5e11 / cfg.flops))) if cfg.flops < 5e12 else 3
    samples = {name: [] for name in legs}
    for _ in range(ROUNDS):
        for name, fn in legs.items():
            samples[name].append(time_ms(fn, n))
    med = {name: sorted(x)[len(x) // 2] for name, x in samples.items()}
    items = cfg.B * cfg.H * (((cfg.S + 127) // 128 + 1) // 2)
    out_bytes = cfg.B * cfg.S * cfg.H * cfg.d * 2
    serial = med["c"] + med["p"] + med["x"]
    row = {"workload": cfg.name, "B": cfg.B, "H": cfg.H, "S": cfg.S, "d": cfg.d, "P": cfg.P,
           "bytes_equal": same, "out_MB": out_bytes / 2**20,
           "fused_host_ms": med["fh"], "fused_host_split_ms": med["fhs"], "fused_host_split_all_ms": med["fha"],
           "split": split_kind(cfg, n_sm), "fused_device_ms": med["fd"], "attention_alone_ms": med["c"],
           "permute_ms": med["p"], "copy_to_host_ms": med["x"], "serial_ms": serial,
           "fused_then_copy_ms": med["fd"] + med["x"], "speedup_vs_serial": serial / med["fh"],
           "speedup_vs_fused_then_copy": (med["fd"] + med["x"]) / med["fh"],
           "host_over_device": med["fh"] / med["fd"] - 1,
           "effective_drain_GBps": out_bytes / (med["fh"] * 1e-3) / 1e9,
           "rank_fused_ms": med["fr"], "rank_serial_ms": med["c"] + med["p"] + med["xr"],
           "rank_speedup_vs_serial": (med["c"] + med["p"] + med["xr"]) / med["fr"]}
    row["model"] = predict(med["fd"], med["c"], items, min(n_sm, items), 2 * 128 * 2 * cfg.d, out_bytes, R)
    row["model"]["burst_gap_rel_err"] = row["model"]["burst_gap_ms"] / med["fh"] - 1
    if trace:
        tr = torch.zeros(bd.trace_numel(cfg.B, cfg.H, cfg.S), dtype=torch.int64, device="cuda")
        for _ in range(2):  # the second call's stamps
            bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, haddr, store_kind=3, trace=tr)
        torch.cuda.synchronize()
        rec = tt.records(tr, cfg.B, cfg.H, cfg.S)
        row["traced_host"] = tt.summary(rec, cfg.S, min(n_sm, items))
        bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, dparts, store_kind=3, trace=tr)
        bd.attn_a2a_fwd(q, k, v, cfg.P, cfg.scale, dparts, store_kind=3, trace=tr)
        torch.cuda.synchronize()
        row["traced_device"] = tt.summary(tt.records(tr, cfg.B, cfg.H, cfg.S), cfg.S, min(n_sm, items))
        del tr
    del q, k, v, dparts, hparts, o, ws
    torch.cuda.empty_cache()
    return row


def split_kind(cfg, n_sm: int):
    """The split the library picks automatically for cfg with a workspace
    (attn_a2a_split_plan): "all", "tail" or None."""
    kind, _, _ = bd.attn_a2a_split_plan(cfg.B, cfg.H, cfg.S, cfg.d, grid=n_sm)
    return {bd.SPLIT_ALL: "all", bd.SPLIT_TAIL: "tail"}.get(kind)


def report(H=40, d=128, P=8, s_list=S_LIST, presets=PRESETS, quick=False) -> dict:
    fits = {"host_lines": probe_fit(0, quick=quick), "host_rows": probe_fit(2, quick=quick, seed=1)}
    R = fits["host_rows"]["R_GBps"] * 1e9
    n_sm = bd.num_sms()
    rows = [measure(workloads.AttnConfig(f"S{S}", B=1, H=H, S=S, d=d, P=P), R, n_sm) for S in s_list]
    rows += [measure(workloads.CONFIGS[name], R, n_sm) for name in presets]
    # The drain rate the fused call itself reaches where its time is all drain
    # (the shortest sequence: the output crossing the link takes twice the
    # compute), used as R for the other workloads (held out from it).
    cal = rows[0]
    R_app = cal["out_MB"] * 2**20 / (cal["fused_host_ms"] * 1e-3)
    for r in rows:
        items = r["B"] * r["H"] * (((r["S"] + 127) // 128 + 1) // 2)
        m = predict(r["fused_device_ms"], r["attention_alone_ms"], items, min(n_sm, items), 2 * 128 * 2 * r["d"],
                    int(r["out_MB"] * 2**20), R_app)
        m["burst_gap_rel_err"] = m["burst_gap_ms"] / r["fused_host_ms"] - 1
        m["held_out"] = r is not cal
        r["model_app_R"] = m
    return {"fits": fits, "R_app_GBps": R_app / 1e9, "R_app_from": cal["workload"], "rows": rows, "sm": n_sm}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    ap.add_argument("--quick", action="store_true", help="fewer probe points and sequence lengths")
    a = ap.parse_args(argv)
    res = report(s_list=(1024, 4096, 32768) if a.quick else S_LIST, quick=a.quick)
    txt = json.dumps(res, indent=1)
    if a.out:
        with open(a.out, "w") as fh:
            fh.write(txt)
    for r in res["rows"]:
        m, ma = r["model"], r["model_app_R"]
        print(f"{r['workload']:>7} S={r['S']:>6}: fused->host {r['fused_host_ms']:.3f} ms, ->device "
              f"{r['fused_device_ms']:.3f}, serial {r['serial_ms']:.3f} ({r['speedup_vs_serial']:.2f}x); "
              f"Burst-Gap probe R {m['burst_gap_ms']:.3f} ({100 * m['burst_gap_rel_err']:+.0f} %), app R "
              f"{ma['burst_gap_ms']:.3f} ({100 * ma['burst_gap_rel_err']:+.0f} %); coupled "
              f"{ma['completion_coupled_ms']:.3f}, async {ma['unbounded_async_ms']:.3f}; bytes equal {r['bytes_equal']}")
    print(f"R from the fused call at {res['R_app_from']}: {res['R_app_GBps']:.1f} GB/s")
    for r in res["rows"]:
        print(f"{r['workload']:>7}: one rank's view (own partition local, P - 1 in host memory): fused "
              f"{r['rank_fused_ms']:.3f} ms, serial {r['rank_serial_ms']:.3f} ({r['rank_speedup_vs_serial']:.2f}x)")
    for r in res["rows"]:
        print(f"{r['workload']:>7}: fused->host with the automatic split ({r['split']}) {r['fused_host_split_ms']:.3f} ms, "
              f"whole schedule split {r['fused_host_split_all_ms']:.3f} ms, without {r['fused_host_ms']:.3f} ms")
    for k, f in res["fits"].items():
        print(f"fit {k}: R {f['R_GBps']:.1f} GB/s, Q {f['Q_MB']} MB, held-out {f['heldout']}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
