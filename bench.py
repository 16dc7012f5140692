#!/usr/bin/env python
"""Benchmark of one cascade decode step (shared-prefix attention, one layer).

Workload (default): the Llama-3-8B attention shape -- B=64 sequences, 32
query heads / 8 KV heads, head dim 128, bf16, a 4096-token prefix shared by
all sequences, private suffixes of U[1,256] tokens in a paged cache with
16-token pages in shuffled physical order; q/K/V ~ N(0,1) from seeded
generators.  A step is one hp_cascade_decode call: every sequence and head,
the batched prefix pass, the paged suffix pass and the merge.

Metric: microseconds per step and effective KV TB/s = unique KV bytes (each
stored token once) / step time; also as a fraction of the roofline
max(prefix FLOPs / bf16 peak, unique KV bytes / HBM peak).

Timing: inputs resident in HBM; R distinct input sets (own pools, tables, q
and plan each) are rotated so that R x working set exceeds 3x the L2 size
read at run time, which keeps every step's KV cold in L2; the sets share one
workspace (partial states), as a decode loop reuses one.  One CUDA graph
holds 4R consecutive steps (four rounds of the input sets), as a decode loop
captures its whole forward pass (so steps follow one another kernel to
kernel, not graph launch to graph launch); a remainder replays one-step
graphs.  CUDA events on the launching stream, W warm-up steps, exactly K
timed steps, barrier + synchronize on both sides, max over ranks.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hp|reference]
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/step and effective KV TB/s, Llama-3-8B shape B=64 P=4K; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["hp", "reference"], default="hp")
    ap.add_argument("--config", default="llama3_8b")
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0: enough for 3x L2)")
    ap.add_argument("--graph-steps", type=int, default=0,
                    help="steps per CUDA graph: 0 = four rounds of the input sets, 1 = one graph per step")
    ap.add_argument("--no-naive", action="store_true")
    ap.add_argument("--loop-steps", type=int, default=64,
                    help="decode-loop measurement: steps per input set in one graph (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


# ------------------------------------------------------------------ peaks
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str, interval_ms: int = 100):
        self.uuid = uuid
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.interval_ms)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0] and parts[0] not in self.uuid:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 <= ts <= t1]
        use = inside if inside else [p for _, p in rows]
        sm = [float(p[1]) for p in use if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_max": max((float(p[3]) for p in use if p[3].replace(".", "").isdigit()), default=None)}


# ------------------------------------------------------------- reference
def run_reference(args, rank: int):
    """The oracle, as it stands, timed on this host's cores on the same
    workload: each step is a bounded sample of the step's output rows."""
    if rank != 0:
        return
    import numpy as np  # noqa: F401
    import oracle
    from shared_prefix_decode_gb300.workloads import make_config

    cores = len(os.sched_getaffinity(0))
    oracle.build()
    oracle.set_num_threads(cores)
    wl = make_config(args.config, seed=0)
    rows_all = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
    # calibrate the cost of one row (all cores busy on a batch of rows)
    t = time.perf_counter()
    oracle.cascade(wl, rows_all[:cores * 4])
    t_row = (time.perf_counter() - t) / (cores * 4)
    budget = 90.0
    n = max(1, min(len(rows_all), int(budget / max(t_row, 1e-9) / max(args.steps + args.warmup, 1))))
    sample = rows_all[:: max(1, len(rows_all) // n)][:n]
    for _ in range(args.warmup):
        oracle.cascade(wl, sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.cascade(wl, sample)
    el = time.perf_counter() - t0
    frac = len(sample) / len(rows_all)
    t_step = el / args.steps / frac  # full-step equivalent
    bytes_step = wl.unique_kv_bytes()
    val = bytes_step / t_step / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "us_per_step": t_step * 1e6,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, None),
        "cpu_baseline": {"value": val, "unit": "TB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{len(sample)} of {len(rows_all)} output rows per step (seed 0), "
                                   f"scaled to the full step"},
        "e2e": {"value": val, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, l2_note):
    suf = [int(n[2]) for n in wl.levels[-1].nodes.tolist()]
    cfg = {"workload": f"{wl.name}: cascade decode, B={wl.B}, Hq={wl.Hq}, Hkv={wl.Hkv}, d={wl.d}, "
                       f"shared prefix {int(wl.levels[0].nodes[0, 2]) if len(wl.levels) > 1 else 0}, "
                       f"paged suffixes, page {wl.page_size}, shuffled pages",
           "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d, "page_size": wl.page_size,
           "suffix_len_mean": sum(suf) / len(suf), "unique_kv_bytes": wl.unique_kv_bytes(),
           "prefix_flops": wl.shared_flops()}
    if l2_note:
        cfg["l2"] = l2_note
    return cfg


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, used only while the
    kernel source is unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[kernel]
        if d["source_hash"] == source_hash(d["sources"]):
            return d
    except Exception:
        pass
    return None


# ------------------------------------------------------------ multi-rank
# One independent replica per rank (the step needs no exchange): the job's
# time is the slowest rank's, its throughput the units all ranks processed.
def job_time_ms(local_ms: float, dist, device) -> float:
    """Max over ranks of a timed region (ms); `dist` is None on one rank."""
    if dist is None:
        return local_ms
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tbs(world: int, bytes_per_step: float, us_step: float) -> float:
    """Whole-job effective KV TB/s: every rank's replica moves bytes_per_step
    per step of us_step microseconds."""
    return world * bytes_per_step / (us_step * 1e-6) / 1e12


# -------------------------------------------------------------------- main
def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import numpy as np
    import torch
    from shared_prefix_decode_gb300 import binding as hb
    from shared_prefix_decode_gb300.workloads import full_page_tables, make_config

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()

    # ---------------------------------------------------------- inputs
    wl0 = make_config(args.config, seed=1000 * rank)
    set_bytes = wl0.unique_kv_bytes() + wl0.q.numel() * 2 * 2
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 2 ** 20
    R = args.sets or max(2, math.ceil(3 * l2 / set_bytes))
    sets = []
    for i in range(R):
        wl = wl0 if i == 0 else make_config(args.config, seed=1000 * rank + i)
        wg = wl.to(dev)
        plan = hb.CascadePlan.from_workload(wg)
        # O and LSE share one buffer, so a host read of the result is one copy
        n_o = wl.B * wl.Hq * wl.d * 2
        res = torch.empty(n_o + wl.B * wl.Hq * 4, dtype=torch.uint8, device=dev)
        out = res[:n_o].view(torch.bfloat16).view(wl.B, wl.Hq, wl.d)
        lse = res[n_o:].view(torch.float32).view(wl.B, wl.Hq)
        sets.append({"wl": wl, "wg": wg, "plan": plan, "out": out, "lse": lse, "res": res})
    l2_note = (f"rotating {R} input sets, {R * set_bytes / 1e6:.0f} MB >= 3x L2 ({l2 / 2**20:.0f} MiB); "
               f"no flush")
    # steps per graph: whole rounds of the input sets when at least one round
    gsteps = 4 * R if args.graph_steps <= 0 else args.graph_steps
    if gsteps > R:
        gsteps = (gsteps + R - 1) // R * R
    # one workspace for every input set, as a decode loop reuses one buffer
    ws_shared = hb.alloc_workspace(max(s["plan"].info.ws_bytes for s in sets), dev)
    for s in sets:
        s["plan"].ws = ws_shared
    info = sets[0]["plan"].info
    kernels_per_step = int(info.n_tc_items + info.n_small_items > 0) + 1
    stream = torch.cuda.Stream(device=dev)

    def step(s, st=None):
        hb.hp_cascade_decode(s["plan"], s["wg"].q, s["wl"].scale, out=s["out"], lse=s["lse"], stream=st)

    # warm up eagerly, check status, then capture one graph per input set
    with torch.cuda.stream(stream):
        for s in sets:
            step(s, stream)
    torch.cuda.synchronize(dev)
    for s in sets:
        st = hb.hp_read_device_status(s["plan"].ws)
        if st != 0:
            raise RuntimeError(f"device status {hb.status_str(st)}")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def capture_runs(fn, items):
        """One-step graphs and, when gsteps > 1, graphs of gsteps consecutive
        steps in rotation order: {first item: graph}."""
        singles = [capture(lambda it=it: fn(it)) for it in items]
        runs = {}
        if gsteps > 1:
            for k in range(0, max(1, len(items) - gsteps + 1), gsteps):
                runs[k] = capture(lambda k=k: [fn(items[(k + i) % len(items)]) for i in range(gsteps)])
        return singles, runs

    graphs = capture_runs(lambda s: step(s, stream), sets)
    torch.cuda.synchronize(dev)

    # parity spot check on rank 0 (oracle on a few rows of set 0)
    parity = None
    if rank == 0:
        import oracle
        oracle.build()
        rows = [(b, h) for b in range(0, wl0.B, max(1, wl0.B // 8)) for h in range(0, wl0.Hq, max(1, wl0.Hq // 4))]
        O, L = oracle.cascade(wl0, rows)
        o = sets[0]["out"].float().cpu().numpy()
        l = sets[0]["lse"].cpu().numpy()
        ob = np.stack([o[b, h] for b, h in rows])
        lb = np.array([l[b, h] for b, h in rows])
        parity = {"rows": len(rows), "max_abs_o": float(np.abs(ob - O).max()),
                  "max_abs_lse": float(np.abs(lb - L).max())}

    def barrier():
        if dist is not None:
            dist.barrier()

    def replay(graph_runs, n):
        """Replays exactly n steps in rotation order: whole multi-step graphs
        where they fit, one-step graphs for the rest."""
        singles, runs = graph_runs
        i = 0
        while i < n:
            k = i % len(singles)
            if k in runs and n - i >= gsteps:
                runs[k].replay()
                i += gsteps
            else:
                singles[k].replay()
                i += 1

    def timed(graph_runs, steps, warmup):
        replay(graph_runs, warmup)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t_wall0 = time.time()
        e0.record(stream)
        with torch.cuda.stream(stream):
            replay(graph_runs, steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t_wall1 = time.time()
        barrier()
        ms = job_time_ms(e0.elapsed_time(e1), dist, dev)
        return ms, t_wall0, t_wall1

    clocks = ClockSampler(getattr(props, "uuid", "") and str(props.uuid))
    clocks.start()
    time.sleep(0.3)
    ms, tw0, tw1 = timed(graphs, args.steps, args.warmup)
    clock_summary = clocks.summary(tw0, tw1)
    clocks.stop()

    us_step = ms * 1e3 / args.steps
    bytes_per_step = statistics.mean(s["wl"].unique_kv_bytes() for s in sets)
    flops_per_step = statistics.mean(s["wl"].shared_flops() for s in sets)
    value = whole_job_tbs(world, bytes_per_step, us_step)
    t_bytes = bytes_per_step / (peaks["hbm_gbs"] * 1e9)
    t_flops = flops_per_step / (peaks["bf16_tflops"] * 1e12)
    roof_us = max(t_bytes, t_flops) * 1e6

    # ------------------------------------------- per-kernel event pass
    ev_sets = []
    for s in sets:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
        for e in evs:
            e.record(stream)  # creates the CUDA event behind the handle
        g = capture(lambda s=s, evs=evs: hb.hp_cascade_decode_profiled(
            s["plan"], s["wg"].q, s["wl"].scale, s["out"], s["lse"], evs, stream=stream))
        ev_sets.append((g, evs))
    torch.cuda.synchronize(dev)
    k_ms = {"cascade": [], "merge": []}
    passes = max(1, min(200, args.steps // max(R, 1)))
    for _ in range(passes):
        for g, _ in ev_sets:
            g.replay()
        torch.cuda.synchronize(dev)
        for _, evs in ev_sets:
            k_ms["cascade"].append(evs[0].elapsed_time(evs[1]))
            k_ms["merge"].append(evs[1].elapsed_time(evs[2]))
    k_us = {k: statistics.mean(v) * 1e3 for k, v in k_ms.items()}

    # algorithmic bytes per launch of each kernel
    def level_bytes(wl, shared):
        tot = 0
        for lv in wl.levels:
            for sb, se, kl, _ in lv.nodes.tolist():
                rows = (se - sb) * wl.G
                if (rows > 16) == shared:
                    tot += kl * wl.Hkv * wl.d * 4
        return tot

    tc_bytes = statistics.mean(level_bytes(s["wl"], True) for s in sets)
    small_bytes = statistics.mean(level_bytes(s["wl"], False) for s in sets)
    merge_bytes = statistics.mean(
        s["plan"].info.n_part_rows * (s["wl"].d * 2 + 4) + s["wl"].B * s["wl"].Hq * (s["wl"].d * 2 + 4)
        for s in sets)
    kb = {"cascade": tc_bytes + small_bytes, "merge": merge_bytes}
    kname = {"cascade": "hp_cascade_kernel", "merge": "hp_merge_kernel"}
    dom = max(k_us, key=lambda k: k_us[k])
    achieved = kb[dom] / (k_us[dom] * 1e-6) / 1e9
    tr = load_traffic(kname[dom])
    roofline = {"bound": "hbm", "kernel": kname[dom], "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "peak_source": peak_src,
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "algorithmic_bytes": kb[dom], "avg_launch_us": k_us[dom]}
    if tr:
        roofline["traffic_note"] = tr.get("note", "")

    # --------------------------------------------------------------- e2e
    h2d = sets[0]["wl"].q.numel() * 2
    d2h = sets[0]["res"].numel()
    for s in sets:
        s["q_host"] = s["wl"].q.pin_memory()
        s["res_host"] = torch.empty(s["res"].shape, dtype=s["res"].dtype).pin_memory()

    def e2e_step(s):
        s["wg"].q.copy_(s["q_host"], non_blocking=True)
        step(s, stream)
        s["res_host"].copy_(s["res"], non_blocking=True)  # O and LSE

    e2e_graphs = capture_runs(e2e_step, sets)
    e2e_steps = args.steps
    ms_e2e, _, _ = timed(e2e_graphs, e2e_steps, min(args.warmup, 50))
    us_e2e = ms_e2e * 1e3 / e2e_steps
    e2e = {"value": whole_job_tbs(world, bytes_per_step, us_e2e), "unit": "TB/s", "us_per_step": us_e2e,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "path": "pinned host q -> device, hp_cascade_decode, device O and LSE (one buffer) -> pinned host"}

    # ------------------------------------------------ naive baseline
    naive = None
    if not args.no_naive:
        nsets = []
        for s in sets:
            pt, sl = full_page_tables(s["wl"])
            pt, sl = pt.to(dev), sl.to(dev)
            ws = hb.alloc_workspace(hb.suffix_workspace_bytes(s["wl"].B, s["wl"].Hq, s["wl"].d, pt.shape[1],
                                                              s["wl"].page_size), dev)
            nsets.append((s, pt, sl, ws))

        def nstep(n):
            s, pt, sl, ws = n
            hb.hp_suffix_decode_paged(s["wg"].q, s["wg"].k_pool, s["wg"].v_pool, pt, sl, s["wl"].scale,
                                      out=s["out"], lse=s["lse"], ws=ws, stream=stream)

        with torch.cuda.stream(stream):
            for n in nsets:
                nstep(n)
        torch.cuda.synchronize(dev)
        ngraphs = capture_runs(nstep, nsets)
        nk = max(R, min(args.steps, 2000))
        ms_n, _, _ = timed(ngraphs, nk, min(args.warmup, 20))
        naive = {"us_per_step": ms_n * 1e3 / nk, "steps": nk,
                 "kernel": "per-sequence paged decode over the whole context (prefix pages aliased, "
                           "re-read per sequence)",
                 "speedup_of_cascade": (ms_n / nk) / (ms / args.steps)}

    # ------------------------------------------------------ decode loop
    # The same workload as a decode loop: each step appends one token per
    # sequence (hp_cascade_append_kv) and decodes over the grown suffixes
    # (hp_cascade_decode_loop) with a plan built once.  One graph holds
    # loop_steps steps of every input set in rotation, after resetting the
    # suffix lengths; the pools are not reset (each replay rewrites the same
    # slots).
    loop = None
    if args.loop_steps > 0:
        from shared_prefix_decode_gb300.workloads import decode_tokens, with_suffix_capacity
        T = args.loop_steps
        lsets = []
        for i, s in enumerate(sets):
            cap = int(s["wl"].levels[-1].nodes[:, 2].max()) + T
            host = with_suffix_capacity(s["wl"], cap, seed=1000 * rank + i)
            lg = host.to(dev)
            lp = hb.LoopPlan.from_workload(lg, cap)
            lp.ws = ws_shared
            toks = decode_tokens(host, T, seed=1000 * rank + i)
            qs, ks, vs = (torch.stack([t[j] for t in toks]).to(dev) for j in range(3))
            lsets.append({"wl": host, "wg": lg, "plan": lp, "n0": lp.suffix_len.clone(), "qs": qs, "ks": ks,
                          "vs": vs, "out": s["out"], "lse": s["lse"]})

        def loop_run(fused=False):
            for ls in lsets:
                ls["plan"].suffix_len.copy_(ls["n0"], non_blocking=True)
            for t in range(T):
                for ls in lsets:
                    if fused:
                        hb.hp_cascade_decode_append(ls["plan"], ls["qs"][t], ls["ks"][t], ls["vs"][t],
                                                    ls["wl"].scale, out=ls["out"], lse=ls["lse"], stream=stream)
                        continue
                    hb.hp_cascade_append_kv(ls["plan"], ls["ks"][t], ls["vs"][t], stream=stream)
                    hb.hp_cascade_decode_loop(ls["plan"], ls["qs"][t], ls["wl"].scale, out=ls["out"],
                                              lse=ls["lse"], stream=stream)

        with torch.cuda.stream(stream):
            loop_run()
            loop_run(fused=True)
        torch.cuda.synchronize(dev)
        st = hb.hp_read_device_status(ws_shared)
        if st != 0:
            raise RuntimeError(f"decode loop: device status {hb.status_str(st)}")
        n_loop = T * len(lsets)
        reps = max(3, min(200, args.steps // n_loop))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def time_graph(g):
            for _ in range(2):
                g.replay()
            torch.cuda.synchronize(dev)
            e0.record(stream)
            with torch.cuda.stream(stream):
                for _ in range(reps):
                    g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            st = hb.hp_read_device_status(ws_shared)
            if st != 0:
                raise RuntimeError(f"decode loop: device status {hb.status_str(st)}")
            return job_time_ms(e0.elapsed_time(e1), dist, dev) * 1e3 / (reps * n_loop)

        # the append fused into the step (two launches per step): headline
        us_loop = time_graph(capture(lambda: loop_run(fused=True)))
        us_sep = time_graph(capture(loop_run))

        # the same steps without the appends, at the loop's mean suffix
        # lengths (the slots hold tokens of the replays above)
        def decode_only_run():
            for ls in lsets:
                ls["plan"].suffix_len.copy_(ls["n0"] + T // 2, non_blocking=True)
            for t in range(T):
                for ls in lsets:
                    hb.hp_cascade_decode_loop(ls["plan"], ls["qs"][t], ls["wl"].scale, out=ls["out"],
                                              lse=ls["lse"], stream=stream)

        us_dec = time_graph(capture(decode_only_run))
        # keys grow by one token per sequence per step: mean over the loop
        grow = lsets[0]["wl"].B * (T + 1) / 2 * wl0.Hkv * wl0.d * 4
        loop_bytes = bytes_per_step + grow
        loop = {"us_per_step": us_loop, "value": whole_job_tbs(world, loop_bytes, us_loop), "unit": "TB/s",
                "steps_per_graph": n_loop, "graph_replays": reps, "loop_steps": T,
                "kernels_per_step": 2, "mean_kv_bytes_per_step": loop_bytes,
                "separate_append_us_per_step": us_sep, "decode_only_us_per_step": us_dec,
                "step": "hp_cascade_decode_append: the token written by the persistent kernel, the length advanced "
                        "by the merge (plan built once; suffix lengths on the device)"}

    # ---------------------------------------------------- cpu baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        cores = len(os.sched_getaffinity(0))
        oracle.set_num_threads(cores)
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds or reps < 1:
            oracle.cascade(wl0)
            reps += 1
        t_cpu = (time.perf_counter() - t0) / reps
        cpu = {"value": wl0.unique_kv_bytes() / t_cpu / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
               "sample": f"the full step of input set 0 ({wl0.B * wl0.Hq} output rows), {reps} repeats",
               "us_per_step": t_cpu * 1e6}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us_step / 1e3, "us_per_step": us_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": dict(workload_config(wl0, l2_note), graph_steps=gsteps),
            "roofline_step": {"bound": "hbm" if t_bytes >= t_flops else "tensor", "roofline_us": roof_us,
                              "frac": roof_us / us_step, "t_bytes_us": t_bytes * 1e6, "t_flops_us": t_flops * 1e6,
                              "unique_kv_bytes": bytes_per_step, "prefix_flops": flops_per_step,
                              "peak_source": peak_src},
            "roofline": roofline,
            "kernels_us": k_us,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": kernels_per_step * args.steps,
            "clocks": clock_summary,
            "naive": naive,
            "decode_loop": loop,
            "parity_spot": parity,
            "plan": {"tc_items": info.n_tc_items, "small_items": info.n_small_items, "grid": info.grid,
                     "part_rows": info.n_part_rows},
            "device": props.name,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
