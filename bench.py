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
workspace (partial states), as a decode loop reuses one.  The K timed steps
are consecutive steps captured in CUDA graphs (one graph of all K steps when
K <= --graph-max; otherwise graphs of --graph-max steps and one of the
remainder), so steps follow one another kernel to kernel, as in a captured
forward pass.  A timed pass is exactly K steps between CUDA events on the
launching stream, bracketed by a barrier and a synchronize; passes repeat
until --min-timed-s seconds of GPU time (at least 20 passes), after W
warm-up steps.  ms_per_step is the median pass / K (min and p90 alongside),
the max over ranks of each pass.

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
    ap.add_argument("--steps", type=int, default=2000, help="K: consecutive steps per timed pass")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["hp", "reference"], default="hp")
    ap.add_argument("--config", default="llama3_8b")
    ap.add_argument("--part", choices=["all", "prefix", "suffix"], default="all",
                    help="time the whole step, or its shared levels / private suffixes alone")
    ap.add_argument("--B", type=int, default=0, help="batch override (a smaller variant of the workload)")
    ap.add_argument("--prefix", type=int, default=-1, help="first-level prefix override")
    ap.add_argument("--e4m3", action="store_true",
                    help="the levels of the per-sequence pass (private suffixes) read E4M3 copies of the pools")
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0: enough for 3x L2)")
    ap.add_argument("--graph-max", type=int, default=256, help="most steps captured in one CUDA graph")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="timed passes repeat until this much GPU time (at least 20 passes)")
    ap.add_argument("--no-naive", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the warm-L2, one-pass, per-workload and one-graph-per-step figures")
    ap.add_argument("--loop-steps", type=int, default=64,
                    help="decode-loop measurement: steps per input set in one graph (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--parallel-prompting-only", action="store_true",
                    help="print only the Parallel Prompting figure (extras.parallel_prompting) as one JSON line")
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
        "config": workload_config(wl, l2_plan(wl, device_l2_bytes())[1]),
        "cpu_baseline": {"value": val, "unit": "TB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{len(sample)} of {len(rows_all)} output rows per step (seed 0), "
                                   f"scaled to the full step"},
        "e2e": {"value": val, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def l2_plan(wl, l2: int, n_sets: int = 0):
    """Input sets to rotate (R x working set >= 3x L2, at least 2) and the
    config note that says so."""
    set_bytes = wl.unique_kv_bytes() + wl.q.numel() * 2 * 2
    R = n_sets or max(2, math.ceil(3 * l2 / set_bytes))
    return R, f"cold: rotating {R} input sets, {R * set_bytes / 1e6:.0f} MB >= 3x L2 ({l2 / 2**20:.0f} MiB); no flush"


def device_l2_bytes() -> int:
    """L2 size of the current CUDA device (GB300's 126 MiB when none)."""
    try:
        import torch
        if torch.cuda.is_available():
            v = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0) or 0)
            if v > 0:
                return v
    except Exception:
        pass
    return 126 * 2 ** 20


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
    if getattr(wl, "part", "all") != "all":
        cfg["part"] = wl.part
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


def plan_summary(hb, s) -> dict:
    """Work items of a set's plan and how the persistent grid is split
    between the two roles (host-side listing of the same plan)."""
    info = s["plan"].info
    wl = s["wl"]
    items = hb.hp_cascade_plan_items(hb._levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d, num_sms=info.grid)
    tc_ctas = {it["cta"] for it in items if it["tc"]}
    sm_ctas = {it["cta"] for it in items if not it["tc"]}
    return {"tc_items": info.n_tc_items, "small_items": info.n_small_items, "grid": info.grid,
            "part_rows": info.n_part_rows, "tc_ctas": len(tc_ctas), "paged_ctas": len(sm_ctas),
            "ctas_with_both": len(tc_ctas & sm_ctas)}


def parallel_prompting_figure(hb, dev, stream, peaks, dist) -> dict:
    """Parallel Prompting rows (Read Once, Answer Many, Section 3): R
    requests of P streams over their own 8K-token documents, decode step 64,
    questions U[32, 64]; each request's row read in place with the stream
    mask (hp_stream_decode) against the same requests in the cascade form
    (the document a node shared by the request's streams, each stream's
    slots a private node) -- both read the same unique bytes -- and against
    one request per question (per-sequence paged decode over the document
    and the question's own slots: the document read once per question, the
    page's prefix-caching baseline)."""
    import torch
    from shared_prefix_decode_gb300 import workloads as W
    R, P, doc, T = 2, 64, 8192, 64
    sets = []
    for i in range(2):
        req = W.stream_requests(R=R, P=P, Hq=32, Hkv=32, d=128, doc_len=doc, q_len_range=(32, 64), T=T, seed=900 + i)
        rows = W.stream_rows_paged(req, seed=i).to(dev)
        tree = W.streams_as_tree(req).to(dev)
        plan = hb.CascadePlan.from_workload(tree)
        q = req.q.to(dev)
        ws = hb.alloc_workspace(hb.stream_workspace_bytes(R, P, 32, 32, 128, rows.row_pages.shape[1], 16), dev)
        out = torch.empty(R * P, 32, 128, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(R * P, 32, dtype=torch.float32, device=dev)
        pt, sl = W.full_page_tables(tree)
        pt, sl = pt.to(dev), sl.to(dev)
        ws_n = hb.alloc_workspace(hb.suffix_workspace_bytes(R * P, 32, 128, pt.shape[1], 16), dev)
        sets.append({"req": req, "rows": rows, "tree": tree, "plan": plan, "q": q, "ws": ws, "out": out, "lse": lse,
                     "pt": pt, "sl": sl, "ws_n": ws_n})
    nbytes = statistics.mean(int(s["rows"].row_len.sum()) * 32 * 128 * 4 for s in sets)

    def in_place(s):
        hb.hp_stream_decode(s["q"], s["rows"], P, s["req"].scale, out=s["out"], lse=s["lse"], ws=s["ws"],
                            stream=stream)

    def cascade(s):
        hb.hp_cascade_decode(s["plan"], s["tree"].q, s["tree"].scale, out=s["out"], lse=s["lse"], stream=stream)

    res = {"requests": R, "streams_per_request": P, "document_tokens": doc, "decode_step": T,
           "unique_kv_bytes": nbytes}
    def per_question(s):
        hb.hp_suffix_decode_paged(s["tree"].q, s["tree"].k_pool, s["tree"].v_pool, s["pt"], s["sl"], s["tree"].scale,
                                  out=s["out"], lse=s["lse"], ws=s["ws_n"], stream=stream)

    for name, fn in (("in_place_masked_rows", in_place), ("cascade_form", cascade),
                     ("one_request_per_question", per_question)):
        with torch.cuda.stream(stream):
            for s in sets:
                fn(s)
        torch.cuda.synchronize(dev)
        g = StepGraphs(fn, sets, 8, 256, stream)
        t, _, _ = timed_passes(g, 4, 0.2, stream, dev, dist)
        st = pass_stats(t, 8)
        res[name] = dict(st, tbs=nbytes / (st["median_us"] * 1e-6) / 1e12,
                         roofline_frac=nbytes / (peaks["hbm_gbs"] * 1e9) / (st["median_us"] * 1e-6))
    for s in sets:
        if hb.hp_read_device_status(s["ws"]) != 0:
            raise RuntimeError("parallel prompting rows: device status")
    return res


# ------------------------------------------------------------ graph timing
class StepGraphs:
    """CUDA graphs of consecutive steps over `items` in rotation order (step i
    uses items[i % R]): a pass of exactly K steps is K // full replays of a
    graph of `full` steps (a multiple of R, so it starts every replay at item
    0) and one replay of a graph of the remaining K % full steps."""

    def __init__(self, fn, items, K: int, graph_max: int, stream):
        import torch
        R = len(items)
        self.K = K
        self.full = R * max(1, graph_max // R)
        self.n_full = K // self.full if K >= self.full else 0
        rem = K - self.n_full * self.full

        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    fn(items[i % R])
            return g

        self.g_full = capture(self.full) if self.n_full > 0 else None
        self.g_rem = capture(rem) if rem > 0 else None

    def run_pass(self):
        for _ in range(self.n_full):
            self.g_full.replay()
        if self.g_rem is not None:
            self.g_rem.replay()


def timed_passes(graphs: StepGraphs, warmup: int, min_s: float, stream, dev, dist, min_passes: int = 20,
                 max_passes: int = 20000):
    """Warm-up passes (at least `warmup` steps), then timed passes of exactly
    K steps each, every pass between CUDA events on `stream`, a barrier and a
    synchronize on both sides; at least `min_passes` and until `min_s` seconds
    of GPU time.  Returns (per-pass ms, max over ranks; wall start; wall end)."""
    import torch
    K = graphs.K

    def barrier():
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / K))):
            graphs.run_pass()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2)]
    times = []
    n_target = min_passes
    t_wall0 = time.time()
    i = 0
    while i < n_target:
        barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = ev[i & 1]
        e0.record(stream)
        with torch.cuda.stream(stream):
            graphs.run_pass()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
        i += 1
        if i == min_passes:
            # passes for min_s of GPU time, the same count on every rank
            med = statistics.median(times)
            want = min(max_passes, max(min_passes, math.ceil(min_s * 1e3 / max(med, 1e-6))))
            n_target = int(job_time_ms(float(want), dist, dev))
    t_wall1 = time.time()
    barrier()
    if dist is not None:
        t = torch.tensor(times, dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        times = t.tolist()
    return times, t_wall0, t_wall1


def pass_stats(times_ms, K: int) -> dict:
    """Per-step microseconds of the timed passes: median, min, p90."""
    per = sorted(t * 1e3 / K for t in times_ms)
    p90 = per[min(len(per) - 1, int(math.ceil(0.9 * len(per))) - 1)]
    return {"median_us": statistics.median(per), "min_us": per[0], "p90_us": p90, "passes": len(per)}


def roofline_step(bytes_step: float, flops_step: float, us_step: float, peaks: dict) -> dict:
    t_bytes = bytes_step / (peaks["hbm_gbs"] * 1e9)
    t_flops = flops_step / (peaks["bf16_tflops"] * 1e12)
    roof_us = max(t_bytes, t_flops) * 1e6
    return {"bound": "hbm" if t_bytes >= t_flops else "tensor", "roofline_us": roof_us, "frac": roof_us / us_step,
            "t_bytes_us": t_bytes * 1e6, "t_flops_us": t_flops * 1e6, "unique_kv_bytes": bytes_step,
            "prefix_flops": flops_step}


# -------------------------------------------------------------------- main
def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")

    import numpy as np
    import torch
    from shared_prefix_decode_gb300 import binding as hb
    from shared_prefix_decode_gb300.workloads import full_page_tables, make_config, with_e4m3_levels

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()
    K = args.steps
    stream = torch.cuda.Stream(device=dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 2 ** 20
    if args.parallel_prompting_only:
        pp = parallel_prompting_figure(hb, dev, stream, peaks, dist)
        if rank == 0:
            print(json.dumps({"parallel_prompting": pp, "device": props.name}))
        return

    def make_sets(name, part, seed0, n_sets=0, device=None, e4m3=False):
        """Input sets of one workload (R of them: R x working set >= 3x L2,
        at least 2), each with its plan and a result buffer; one workspace
        shared by all.  e4m3: the levels of the per-sequence pass read E4M3
        copies of the pools."""
        def gen(seed):
            kw = {}
            if name == args.config and args.B > 0:
                kw["B"] = args.B
            if name == args.config and args.prefix >= 0:
                kw["prefix"] = args.prefix
            wl = make_config(name, seed=seed, part=part, device=device, **kw)
            return with_e4m3_levels(wl) if e4m3 else wl

        first = gen(seed0)
        R, note = l2_plan(first, l2, n_sets)
        out = []
        for i in range(R):
            wl = first if i == 0 else gen(seed0 + i)
            wg = wl.to(dev)
            plan = hb.CascadePlan.from_workload(wg)
            # O and LSE share one buffer, so a host read of the result is one copy
            n_o = wl.B * wl.Hq * wl.d * 2
            res = torch.empty(n_o + wl.B * wl.Hq * 4, dtype=torch.uint8, device=dev)
            o = res[:n_o].view(torch.bfloat16).view(wl.B, wl.Hq, wl.d)
            ls = res[n_o:].view(torch.float32).view(wl.B, wl.Hq)
            out.append({"wl": wl, "wg": wg, "plan": plan, "out": o, "lse": ls, "res": res})
        ws = hb.alloc_workspace(max(s["plan"].info.ws_bytes for s in out), dev)
        for s in out:
            s["plan"].ws = ws
        return out, ws, note

    def step(s, st=None):
        hb.hp_cascade_decode(s["plan"], s["wg"].q, s["wl"].scale, out=s["out"], lse=s["lse"], stream=st)

    def warm_and_check(items, fn, ws):
        with torch.cuda.stream(stream):
            for it in items:
                fn(it)
        torch.cuda.synchronize(dev)
        st = hb.hp_read_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {hb.status_str(st)}")

    # ---------------------------------------------------------- inputs
    sets, ws_shared, l2_note = make_sets(args.config, args.part, 1000 * rank, args.sets, e4m3=args.e4m3)
    R = len(sets)
    wl0 = sets[0]["wl"]
    info = sets[0]["plan"].info
    kernels_per_step = int(info.n_tc_items + info.n_small_items > 0) + 1
    warm_and_check(sets, lambda s: step(s, stream), ws_shared)
    graphs = StepGraphs(lambda s: step(s, stream), sets, K, args.graph_max, stream)
    torch.cuda.synchronize(dev)

    # parity spot check on rank 0 (oracle on a few rows of set 0)
    parity = None
    if rank == 0:
        import oracle
        oracle.build()
        rows = [(b, h) for b in range(0, wl0.B, max(1, wl0.B // 8)) for h in range(0, wl0.Hq, max(1, wl0.Hq // 4))]
        O, L = oracle.cascade(wl0, rows)
        o = sets[0]["out"].float().cpu().numpy()
        lv = sets[0]["lse"].cpu().numpy()
        ob = np.stack([o[b, h] for b, h in rows])
        lb = np.array([lv[b, h] for b, h in rows])
        parity = {"rows": len(rows), "max_abs_o": float(np.abs(ob - O).max()),
                  "max_abs_lse": float(np.abs(lb - L).max())}

    clocks = ClockSampler(getattr(props, "uuid", "") and str(props.uuid))
    clocks.start()
    time.sleep(0.3)
    times, tw0, tw1 = timed_passes(graphs, args.warmup, args.min_timed_s, stream, dev, dist)
    clock_summary = clocks.summary(tw0, tw1)
    clocks.stop()
    stats = pass_stats(times, K)
    us_step = stats["median_us"]
    bytes_per_step = statistics.mean(s["wl"].unique_kv_bytes() for s in sets)
    flops_per_step = statistics.mean(s["wl"].shared_flops() for s in sets)
    value = whole_job_tbs(world, bytes_per_step, us_step)
    roof = dict(roofline_step(bytes_per_step, flops_per_step, us_step, peaks), peak_source=peak_src)
    timing = dict(stats, steps_per_pass=K, graph_steps=min(K, graphs.full), timed_s=sum(times) / 1e3,
                  form="CUDA graphs of the K consecutive steps (rotating input sets), one pass per timed "
                       "region; median / min / p90 over passes")

    # ------------------------------------------- per-kernel event pass
    ev_sets = []
    for s in sets:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
        for e in evs:
            e.record(stream)  # creates the CUDA event behind the handle
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            hb.hp_cascade_decode_profiled(s["plan"], s["wg"].q, s["wl"].scale, s["out"], s["lse"], evs,
                                          stream=stream)
        ev_sets.append((g, evs))
    torch.cuda.synchronize(dev)
    k_ms = {"cascade": [], "merge": []}
    for _ in range(max(3, min(200, 2000 // max(R, 1)))):
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
                rows_ = (se - sb) * wl.G
                if (rows_ > 16) == shared:
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
    # The step as a caller with host-resident queries runs it:
    # hp_cascade_decode_host reads each step's q from pinned host memory
    # (copy-in kernel) and the merge stores O and LSE into pinned host memory.
    h2d = sets[0]["wl"].q.numel() * 2
    d2h = sets[0]["res"].numel()
    ws_host = hb.alloc_workspace(max(hb.host_workspace_bytes(s["plan"]) for s in sets), dev)
    for s in sets:
        wl = s["wl"]
        s["q_host"] = wl.q.pin_memory()
        s["res_host"] = torch.empty(s["res"].shape, dtype=s["res"].dtype).pin_memory()
        n_o = wl.B * wl.Hq * wl.d * 2
        s["o_host"] = s["res_host"][:n_o].view(torch.bfloat16).view(wl.B, wl.Hq, wl.d)
        s["lse_host"] = s["res_host"][n_o:].view(torch.float32).view(wl.B, wl.Hq)

    def e2e_step(s):
        hb.hp_cascade_decode_host(s["plan"], s["q_host"], s["wl"].scale, s["o_host"], s["lse_host"], ws_host,
                                  stream=stream)

    e2e_graphs = StepGraphs(e2e_step, sets, K, args.graph_max, stream)
    t_e2e, _, _ = timed_passes(e2e_graphs, min(args.warmup, 50), min(args.min_timed_s, 0.5), stream, dev, dist)
    st_e2e = pass_stats(t_e2e, K)
    us_e2e = st_e2e["median_us"]
    # the host result equals the device-resident step's, bit for bit
    step(sets[0], stream)
    torch.cuda.synchronize()
    same = bool(torch.equal(sets[0]["res_host"], sets[0]["res"].cpu()))
    st = hb.hp_read_device_status(ws_host)
    if st != hb.HP_OK:
        raise RuntimeError(f"host-memory step: device status {hb.status_str(st)}")
    e2e = {"value": whole_job_tbs(world, bytes_per_step, us_e2e), "unit": "TB/s", "us_per_step": us_e2e,
           "min_us": st_e2e["min_us"], "p90_us": st_e2e["p90_us"],
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "equals_device_step": same,
           "path": "hp_cascade_decode_host: q read from pinned host memory by a copy-in kernel, the step, "
                   "O and LSE stored by the merge into pinned host memory"}

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
        nk = 4 * R
        t_n, _, _ = timed_passes(StepGraphs(nstep, nsets, nk, args.graph_max, stream), min(args.warmup, 20), 0.2,
                                 stream, dev, dist)
        st_n = pass_stats(t_n, nk)
        naive = {"us_per_step": st_n["median_us"], "min_us": st_n["min_us"], "p90_us": st_n["p90_us"],
                 "steps_per_pass": nk, "passes": st_n["passes"],
                 "kernel": "per-sequence paged decode over the whole context (prefix pages aliased, "
                           "re-read per sequence)",
                 "speedup_of_cascade": st_n["median_us"] / us_step}

    # ------------------------------------------------------ decode loop
    # The same workload as a decode loop: each step appends one token per
    # sequence (hp_cascade_append_kv) and decodes over the grown suffixes
    # (hp_cascade_decode_loop) with a plan built once.  One graph holds
    # loop_steps steps of every input set in rotation, after resetting the
    # suffix lengths; the pools are not reset (each replay rewrites the same
    # slots).
    loop = None
    if args.loop_steps > 0 and args.part == "all":
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
        reps = max(3, min(200, 20000 // n_loop))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def capture(fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            return g

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
                "roofline_frac": loop_bytes / (peaks["hbm_gbs"] * 1e9) / (us_loop * 1e-6),
                "steps_per_graph": n_loop, "graph_replays": reps, "loop_steps": T,
                "kernels_per_step": 2, "mean_kv_bytes_per_step": loop_bytes,
                "separate_append_us_per_step": us_sep, "decode_only_us_per_step": us_dec,
                "step": "hp_cascade_decode_append: the token written by the persistent kernel, the length advanced "
                        "by the merge (plan built once; suffix lengths on the device)"}
        del lsets

    # ------------------------------------------------------- extras
    extras = None
    if not args.no_extras:
        extras = {}

        def measure(items, ws, bytes_step, flops_step, k_steps, min_s=0.2):
            warm_and_check(items, lambda s: step(s, stream), ws)
            g = StepGraphs(lambda s: step(s, stream), items, k_steps, args.graph_max, stream)
            t, _, _ = timed_passes(g, 2 * len(items), min_s, stream, dev, dist)
            stt = pass_stats(t, k_steps)
            return dict(stt, steps_per_pass=k_steps, tbs=bytes_step / (stt["median_us"] * 1e-6) / 1e12,
                        roofline=roofline_step(bytes_step, flops_step, stt["median_us"], peaks))

        # the same K steps on one input set over and over (its KV stays in L2)
        extras["warm_l2"] = dict(measure([sets[0]], ws_shared, wl0.unique_kv_bytes(), wl0.shared_flops(), K),
                                 note="WARM L2: input set 0 every step (53 MB < L2), not the cold-L2 headline")
        # the one-graph-per-step form (each step its own graph launch)
        singles = [StepGraphs(lambda s: step(s, stream), [sets[i]], 1, 1, stream) for i in range(R)]

        class _PerStep:
            K = 4 * R

            @staticmethod
            def run_pass():
                for j in range(4 * R):
                    singles[j % R].run_pass()

        t1g, _, _ = timed_passes(_PerStep, R, 0.2, stream, dev, dist)
        extras["graph_per_step"] = dict(pass_stats(t1g, 4 * R),
                                        note="one CUDA graph launch per step (graph launch overhead included)")
        # the step's passes alone (same kernels, same shapes)
        if args.part == "all":
            for part in ("prefix", "suffix"):
                ps_sets, ps_ws, _ = make_sets(args.config, part, 1000 * rank + 500, device=dev)
                b = statistics.mean(s["wl"].unique_kv_bytes() for s in ps_sets)
                f = statistics.mean(s["wl"].shared_flops() for s in ps_sets)
                extras[f"{part}_only"] = measure(ps_sets, ps_ws, b, f, 4 * len(ps_sets))
                del ps_sets, ps_ws
                torch.cuda.empty_cache()
        # the same workload with its private suffixes in E4M3 (bf16 prefix)
        if args.part == "all":
            e_sets, e_ws, e_note = make_sets(args.config, "all", 1000 * rank + 600, device=dev, e4m3=True)
            b = statistics.mean(s["wl"].unique_kv_bytes() for s in e_sets)
            f = statistics.mean(s["wl"].shared_flops() for s in e_sets)
            extras["e4m3_suffix"] = dict(measure(e_sets, e_ws, b, f, 4 * len(e_sets)), l2=e_note,
                                         note="suffix KV as E4M3 codes + f32 scale per (page, KV head); "
                                              "unique bytes count codes and scales")
            del e_sets, e_ws
            torch.cuda.empty_cache()
        # the other workloads at full size, cold L2 (and, for the two that
        # are mostly per-sequence bytes, with those levels in E4M3)
        per_cfg = {}
        for name, e4 in (("codellama13b", False), ("codellama13b", True), ("tree2", False), ("doc_streams", False),
                         ("no_sharing", False), ("no_sharing", True)):
            if name == args.config:
                continue
            c_sets, c_ws, c_note = make_sets(name, "all", 1000 * rank + 700, device=dev, e4m3=e4)
            b = statistics.mean(s["wl"].unique_kv_bytes() for s in c_sets)
            f = statistics.mean(s["wl"].shared_flops() for s in c_sets)
            per_cfg[name + ("_e4m3" if e4 else "")] = dict(
                measure(c_sets, c_ws, b, f, 8 * len(c_sets)), l2=c_note, plan=plan_summary(hb, c_sets[0]))
            del c_sets, c_ws
            torch.cuda.empty_cache()
        extras["workloads"] = per_cfg
        extras["parallel_prompting"] = parallel_prompting_figure(hb, dev, stream, peaks, dist)

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
        # one thread, the tiny workload (whole steps) and this workload (a
        # sample of its rows, scaled to the full step)
        oracle.set_num_threads(1)
        one = {}
        tiny = make_config("tiny", seed=0)
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 1.0 or reps < 1:
            oracle.cascade(tiny)
            reps += 1
        one["tiny_us_per_step"] = (time.perf_counter() - t0) / reps * 1e6
        rows_all = [(b, h) for b in range(wl0.B) for h in range(wl0.Hq)]
        sample = rows_all[::16]
        t0 = time.perf_counter()
        oracle.cascade(wl0, sample)
        one[f"{wl0.name}_us_per_step"] = (time.perf_counter() - t0) * len(rows_all) / len(sample) * 1e6
        one["sample"] = f"tiny: whole steps; {wl0.name}: {len(sample)} of {len(rows_all)} rows, scaled"
        cpu["one_thread"] = one
        oracle.set_num_threads(cores)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": us_step / 1e3, "us_per_step": us_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(wl0, l2_note),
            "timing": timing,
            "roofline_step": roof,
            "roofline": roofline,
            "kernels_us": k_us,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": kernels_per_step * K,
            "clocks": clock_summary,
            "naive": naive,
            "decode_loop": loop,
            "extras": extras,
            "parity_spot": parity,
            "plan": plan_summary(hb, sets[0]),
            "device": props.name,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
