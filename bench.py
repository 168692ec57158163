#!/usr/bin/env python
"""Benchmark of the VerKV hot path on one GB300: PoissonComp + KVFetch on the Qwen3-4B-shaped
32K-token attention layer (batch 1, GQA 32/8, d = 128, bf16 K/V, 16 needles per KV head, 2-bit key
sketch of the paper's Appendix A.1, eta = 1/16, eps = delta = 0.05, 64 decode steps with half the
queries aimed at needles), with the library's default (bounded) staging cache.

One bench step = one pass of the whole hot path over one job: verkv_compress of the 32K context
(importance scores, water-filling, Poisson sample, compaction, sketch) followed by the 64
verkv_decode calls.  Inputs are resident in HBM (plus the pinned host copy the decode fetches from)
when the timed region starts; L2 is flushed (a 512 MB write) before every call and the flush is not
timed.  Prints one JSON line (rank 0).

Beside the headline the line carries: the staging cache off and unbounded, the fetch path's host-link
rate with staging off, binary shrinkage, the deployed shortlist, decode-time growth, the 36-layer
batch-8 stack (full K/V pinned on the host), the 128K long context, and the compress / decode sweep.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl verkv|reference] [--quick]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KVFetch decode µs/step & scored tokens/s at 32K ctx; % of HBM/host-link roofline"
UNIT = "scored tokens/s"
ROW_BYTES = 2 * 128 * 2          # one K + V row of one token and KV head, bf16


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="verkv", choices=["verkv", "reference"])
    p.add_argument("--n", type=int, default=32768)
    p.add_argument("--sketch", default="2bit", choices=["2bit", "int8", "exact"])
    p.add_argument("--decode-steps", type=int, default=64)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-flush", action="store_true", help="(profiling runs) skip the L2 flushes")
    p.add_argument("--no-secondary", action="store_true", help="only the headline workload")
    p.add_argument("--quick", action="store_true", help="fewer sweep points, 4 stack layers (a fast check)")
    p.add_argument("--only", default=None,
                   help="(profiling runs) one secondary measurement only: stack, long, sweep, staging")
    p.add_argument("--stack-layers", type=int, default=36)
    return p.parse_args()


def aggregate_ranks(step_ms, units_per_step, world, device):
    """Replicas: every rank ran its own job; the slowest rank's step time counts (MAX over ranks) and
    the value is the units of all ranks over that time.  Returns (value, step_ms)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(step_ms)], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    return world * units_per_step / (step_ms / 1e3), step_ms


def workload(args, rank=0):
    from verified_kv_cache_gb300 import workloads
    return workloads.qwen_layer_case(seed=1 + 1000 * rank, n=args.n, steps=args.decode_steps, sketch=args.sketch)


def config_string(w, S):
    return (f"qwen3-4b-shaped attention layer, n={w.n}, batch 1, GQA {w.n_q}/{w.n_kv}, d={w.d}, bf16 K/V, "
            f"{w.sketch} sketch, eta=1/{round(1 / w.eta)}, eps={w.eps}, delta={w.delta}, {S} decode steps per job "
            f"(compress + decodes), half the queries aimed at needles")


def read_peaks():
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = {}
    if os.path.exists(pk):
        try:
            with open(pk) as f:
                peaks = json.load(f)
        except ValueError:
            peaks = {}
    hbm = peaks.get("hbm_gbs")
    return (hbm, "measured") if hbm else (6800.0, "fallback")


def cpu_model():
    """The host CPU's model name (/proc/cpuinfo on x86, lscpu on Arm, where cpuinfo names no model)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name") and ":" in line:
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name") and ":" in line:
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


# ----------------------------------------------------------------------------- clocks
class Clocks:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 6]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
            except ValueError:
                continue
            for k, v in zip(names, r[3:7]):
                if "Active" in v and "Not" not in v:
                    reasons.add(k)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- roofline bookkeeping
def sketch_bytes_per_token(sketch, d=128, kv_dtype="bf16"):
    """Bytes of the key sketch per token and KV head: 2-bit codes of d/4 channels plus the fp16 zero and
    scale of each channel per 128-token group; int8 codes plus an fp32 scale; exact keys."""
    return {"2bit": (d // 4) * 2 / 8 + (d // 4) * 4 / 128, "int8": d + 4,
            "exact": d * (2 if kv_dtype == "bf16" else 4)}[sketch]


def algorithmic_bytes(kernel, stats, traces, w, row_bytes, batch=1):
    """Bytes each kernel must move by the method's definition (per launch), from the compressed sizes
    and the decode traces.  Intermediates a kernel writes for the next one are not counted.  `stats`
    holds the head statistics of every sequence of the batch."""
    Hkv, Hq, n, d = w.n_kv, w.n_q, w.n, w.d
    L = sum(s["n_l"] for s in stats)
    H = sum(s["n_h"] for s in stats)
    R = sum(s["n_resident"] for s in stats)
    s_sk = sketch_bytes_per_token(w.sketch, d, w.kv_dtype)
    if kernel == "score":             # sketch of every L token, the L/H position of every token,
        return L * s_sk + batch * Hkv * n * 4 + H * row_bytes / 2 + batch * Hq * d * 4   # exact keys of H, q
    if kernel == "attn":              # resident K/V rows from HBM once per KV head, the fetched rows found
        staged = traces.get("union_rows", 0) - traces.get("host_rows", 0)   # in the staging cache, the
        return (R + staged + traces.get("host_rows", 0)) * row_bytes + batch * Hq * d * 8   # rows staged, q/out
    if kernel == "attn_link":         # the fetched rows that crossed the host link, once per KV head
        return traces.get("host_rows", 0) * row_bytes
    return None


def measured_counters(w):
    """The committed ncu record of this workload's decode kernels (DRAM bytes and warp instructions per
    launch), if the kernel source is the one the counters were taken on (else {}: changed since)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"traffic_qwen3-4b-{w.n // 1024}k-{w.sketch}.txt")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        body = "".join(line for line in f if not line.startswith("#"))
    try:
        rec = json.loads(body)
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
    except (ValueError, KeyError, OSError):
        return {}
    return rec if sha == rec["source_sha256"] else {}


def measured_traffic(w):
    """DRAM bytes per launch of the decode kernels from the committed ncu summary (see measured_counters)."""
    return measured_counters(w).get("dram_bytes_per_launch", {})


def roof_entry(kernel, avg_ms, by, peak, unit, bound, peak_source, traffic=None, note=None):
    ach = by / (avg_ms / 1e3) / 1e9
    e = {"kernel": kernel, "bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
         "traffic": traffic, "peak_source": peak_source, "algorithmic_bytes": by, "avg_us": avg_ms * 1e3}
    if note:
        e["note"] = note
    return e


def kernel_agg(kt):
    agg = {}
    for name, ms in kt:
        a = agg.setdefault(name, [0.0, 0])
        a[0] += ms
        a[1] += 1
    return agg


def measure_link_peak(dev, st):
    """Host-link peak: a bulk pinned host -> device copy of 256 MiB (the link the fetch uses)."""
    import torch
    src = torch.empty(256 * 1024 * 1024, dtype=torch.uint8).pin_memory()
    dst = torch.empty_like(src, device=dev)
    best = None
    for _ in range(4):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(st)
        dst.copy_(src, non_blocking=True)
        b_.record(st)
        b_.synchronize()
        ms_ = a_.elapsed_time(b_)
        best = ms_ if best is None else min(best, ms_)
    del src, dst
    return 256 * 1024 * 1024 / (best / 1e3) / 1e9


def footprint(stats, w, stage_rows):
    """Device memory of one slot against its full K/V cache: the resident rows (H u S), the staging
    cache's capacity, and the sketch."""
    import math as _m
    res = sum(s["n_resident"] for s in stats)
    fetchable = [s["n_l"] - s["n_s"] for s in stats]
    eta_n = _m.ceil(w.eta * w.n)
    if stage_rows == -2:
        cap = sum(min(eta_n, f) for f in fetchable)
    elif stage_rows == -1:
        cap = sum(fetchable)
    else:
        cap = sum(min(stage_rows, f) for f in fetchable)
    full = len(stats) * w.n * ROW_BYTES
    sk = len(stats) * w.n * sketch_bytes_per_token(w.sketch, w.d, w.kv_dtype)
    return {"resident_rows": res, "staging_rows_capacity": cap, "sketch_bytes": sk,
            "kv_fraction_resident": res * ROW_BYTES / full,
            "kv_fraction_resident_plus_staging": (res + cap) * ROW_BYTES / full,
            "fraction_incl_sketch": ((res + cap) * ROW_BYTES + sk) / full}


# ----------------------------------------------------------------------------- the GPU arm
def run_verkv(args):
    import torch
    import torch.distributed as dist

    from verified_kv_cache_gb300 import binding, build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    build.build()
    hbm_peak, peak_src = read_peaks()
    w = workload(args, rank)
    ctx = binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=w.n, n_layers=1, n_seqs=1, max_batch=1,
                        n_sink=w.n_sink, n_local=w.n_local, eta=w.eta, seed=w.seed, sketch=w.sketch,
                        kv_dtype=w.kv_dtype)
    kv_np = w.kv_host_layout(0)
    kv_host = torch.from_numpy(kv_np).view(torch.bfloat16).pin_memory()
    kv_dev = kv_host.to(dev)
    obs_host = torch.from_numpy(w.obs_q[0]).pin_memory()
    obs = obs_host.to(dev)
    q_host = torch.from_numpy(w.queries[:, :1]).pin_memory()      # [S, 1, Hq, d]
    q_dev = q_host.to(dev)
    out = torch.empty_like(q_dev)
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    W = w.obs_q.shape[2]
    S = w.queries.shape[0]
    st = torch.cuda.current_stream()
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def flush():
        if not args.no_flush:
            flush_buf.fill_(1.0)

    def one_step(events, kv_src=None):
        n_launch = 0
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        stats = ctx.compress(0, 0, w.n, kv_host, kv_dev if kv_src is None else kv_src, obs, W, None, st)
        e1.record(st)
        n_launch += ctx.last_launch_count()
        events.append(("compress", e0, e1))
        for s in range(S):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
            b.record(st)
            n_launch += ctx.last_launch_count()
            events.append(("decode", a, b))
        return stats, n_launch

    # the clock sampler starts before the warm-up: its start-up (driver attach) must not fall in the
    # timed region, where it stalled one host-synchronous compress by several milliseconds
    clocks = Clocks(dev.index or 0) if rank == 0 else None
    time.sleep(0.5)
    for _ in range(max(args.warmup, 0)):
        one_step([])
    torch.cuda.synchronize()
    # fetch statistics of the workload (one untimed job with traces)
    ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
    fetch_frac, no_fetch, union_rows, host_rows, kstars, pf_copied, pf_used = [], 0, [], [], [], [], []
    tlines = {"needle": [], "random": []}   # device timeline of each call (even steps aim at needles)
    ctx.set_timeline(True)
    for s in range(S):
        flush()
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
        tlines["needle" if s % 2 == 0 else "random"].append(ctx.timeline(st))
        tr = ctx.decode_trace(w.n_q)
        for h in range(w.n_kv):
            u, hr = ctx.fetch_stats(0, h)
            pc, pu = ctx.prefetch_stats(0, h)
            union_rows.append(u)
            host_rows.append(hr)
            pf_copied.append(pc)
            pf_used.append(pu)
            fetch_frac.append(u / w.n)
        no_fetch += sum(t["no_fetch"] for t in tr)
        kstars += [t["kstar"] for t in tr]
    ctx.set_timeline(False)
    timeline = {kind: {k: round(statistics.median(t[k] for t in ts), 1) for k in ts[0]
                       if all(math.isfinite(t[k]) for t in ts)}
                for kind, ts in tlines.items() if ts}
    stats0 = ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)

    # timed region: per-call events only (events between the kernels of a call would stop the
    # programmatic launch overlap of the decode kernels)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    events = []
    launches = 0
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        _, nl = one_step(events)
        launches += nl
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    # the same K steps again with an event pair around every kernel: per-kernel durations for the
    # rooflines and the kernel shares, with the rows the attention itself read over the host link in
    # those calls (the events stop the overlap of the kernels, so the prefetch, which runs beside the
    # decision, finds it decided and copies next to nothing there)
    ctx.set_kernel_timing(True)
    kt = []
    kt_host = []
    for _ in range(args.steps):
        one_step([])
        kt += ctx.kernel_times(st)   # drains the per-kernel records (one sync between steps)
    ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
    for s in range(S):
        flush()
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
        kt_host.append(sum(ctx.fetch_stats(0, h)[1] for h in range(w.n_kv)))
    ctx.kernel_times(st)
    torch.cuda.synchronize()
    ctx.set_kernel_timing(False)
    comp_ms = [a.elapsed_time(b) for k, a, b in events if k == "compress"]
    dec_ms = [a.elapsed_time(b) for k, a, b in events if k == "decode"]
    step_ms = (sum(comp_ms) + sum(dec_ms)) / args.steps
    units_per_step = S * 1 * w.n_q * w.n        # scored tokens: every query head scores every token
    value, step_ms = aggregate_ranks(step_ms, units_per_step, world, dev)

    agg = kernel_agg(kt)
    total_ms = sum(v[0] for v in agg.values())
    # the attention's rows in the per-kernel timing pass (what its timed launches moved) for its rooflines
    traces = {"union_rows": statistics.mean(union_rows) * w.n_kv if union_rows else 0,
              "host_rows": statistics.mean(kt_host) if kt_host else 0}
    # the whole decode job as it runs: every byte over the host link (the prefetch's copies and the
    # attention's own reads) against the decode time
    link_bytes = (statistics.mean(host_rows) + statistics.mean(pf_copied)) * w.n_kv * ROW_BYTES if host_rows else 0
    job_link = {"bytes_per_call": link_bytes, "decode_us_per_call": statistics.mean(dec_ms) * 1e3,
                "achieved_gbs": link_bytes / (statistics.mean(dec_ms) / 1e3) / 1e9}
    traffic = measured_traffic(w)
    link_peak = measure_link_peak(dev, st) if rank == 0 else None
    if link_peak:
        job_link["frac_of_link_peak"] = job_link["achieved_gbs"] / link_peak

    def roof_hbm(kname, note=None):
        if kname not in agg:
            return None
        by = algorithmic_bytes(kname, stats0, traces, w, ROW_BYTES)
        return roof_entry(kname, agg[kname][0] / agg[kname][1], by, hbm_peak, "GB/s", "hbm",
                          f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)", traffic.get(kname), note)

    def roof_link(kname):
        if kname not in agg or not link_peak:
            return None
        by = algorithmic_bytes(kname + "_link", stats0, traces, w, ROW_BYTES)
        return roof_entry(kname, agg[kname][0] / agg[kname][1], by, link_peak, "GB/s", "host_link",
                          "measured in this run: pinned host -> device copy of 256 MiB", None,
                          "rows that crossed the host link over the whole attention kernel's time")

    # headline roofline: the attention kernel, the dominant kernel among those with a byte bound (the
    # decision is latency-bound and reported as time only); its bound is the resource whose bytes take
    # longer at peak (HBM for the resident and staged rows, the host link for the rows that cross it)
    roofline = roof_hbm("attn", "resident + staged + newly staged rows and q/out over the attention's time")
    if link_peak and "attn" in agg:
        t_link = algorithmic_bytes("attn_link", stats0, traces, w, ROW_BYTES) / link_peak
        t_hbm = algorithmic_bytes("attn", stats0, traces, w, ROW_BYTES) / hbm_peak
        if t_link > t_hbm:
            roofline = roof_link("attn")
    roof_score = roof_hbm("score")
    # the 2-bit scan is bound by instruction issue (exact float-float sketch logits on the CUDA cores):
    # its issue roofline is the warp instructions of a launch (committed ncu counter) over its time,
    # against 4 instructions per cycle on each of the SMs at the sampled SM clock
    roof_issue = None
    inst = measured_counters(w).get("warp_instructions_per_launch", {}).get("score")
    if inst and "score" in agg and clk and clk.get("sm_mhz"):
        import torch as _t
        sms = _t.cuda.get_device_properties(dev).multi_processor_count
        avg_s = agg["score"][0] / agg["score"][1] / 1e3
        peak = sms * 4 * clk["sm_mhz"] * 1e6
        roof_issue = {"kernel": "score", "bound": "issue", "achieved": inst / avg_s, "peak": peak,
                      "unit": "warp instructions/s", "frac": inst / avg_s / peak, "warp_instructions": inst,
                      "avg_us": avg_s * 1e6, "peak_source": f"{sms} SMs x 4 issue slots x sampled {clk['sm_mhz']} MHz"}
    roof_decide = ({"kernel": "decide", "bound": "latency", "avg_us": agg["decide"][0] / agg["decide"][1] * 1e3,
                    "achieved": None, "peak": None, "frac": None,
                    "note": "cluster barriers and block reductions over on-chip rows; reported as time only"}
                   if "decide" in agg else None)

    # ---------------------------------------------------------------- end to end through the public API
    e2e = None
    if not args.no_e2e:
        kv_scratch = torch.empty_like(kv_dev)
        obs_scratch = torch.empty_like(obs)
        q_scratch = torch.empty_like(q_dev)
        h2d = kv_host.numel() * 2 + obs_host.numel() * 4 + q_host.numel() * 4
        d2h = out.numel() * 4
        e_ms = []
        for it in range(args.warmup + args.steps):
            # the same L2 policy as the device-timed steps: flushed (untimed) before every call, each
            # segment timed by its own event pair; the copies sit inside the first and last segments
            segs = []
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            kv_scratch.copy_(kv_host, non_blocking=True)
            obs_scratch.copy_(obs_host, non_blocking=True)
            q_scratch.copy_(q_host, non_blocking=True)
            ctx.compress(0, 0, w.n, kv_host, kv_scratch, obs_scratch, W, None, st)
            b.record(st)
            segs.append((a, b))
            for s in range(S):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                ctx.decode(0, [0], q_scratch[s], w.eps, w.delta, out[s], st)
                if s == S - 1:
                    out_host.copy_(out, non_blocking=True)
                b.record(st)
                segs.append((a, b))
            torch.cuda.synchronize()
            if it >= args.warmup:
                e_ms.append(sum(x.elapsed_time(y) for x, y in segs))
        e2e = {"value": world * units_per_step / (statistics.mean(e_ms) / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": statistics.mean(e_ms)}
        del kv_scratch

    secondary = {}
    only = args.only
    if rank == 0 and not args.no_secondary:
        if only in (None, "staging"):
            secondary["staging_off"] = staging_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush, 0, link_peak)
            secondary["staging_all_rows"] = staging_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush, -1,
                                                        link_peak)
        if only is None:
            secondary["binary_shrinkage"] = binary_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush)
            secondary["deployed_binary_shortlist128"] = binary_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush,
                                                                   shortlist=128)
            secondary["growth_append1"] = growth_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush)
    ctx.close()
    if rank == 0 and not args.no_secondary:
        del kv_dev, flush_buf
        torch.cuda.empty_cache()
        if only in (None, "stack"):
            secondary["stack36_b8_int8"] = stack36_run(args, dev, st, hbm_peak, peak_src, link_peak)
            torch.cuda.empty_cache()
        if only in (None, "long"):
            secondary["long_context_128k_int8"] = long_context_run(args, dev, st, hbm_peak, peak_src, link_peak)
            torch.cuda.empty_cache()
        if only in (None, "sweep"):
            secondary["sweep"] = sweep_run(args, dev, st, hbm_peak, peak_src, link_peak,
                                           clk.get("sm_mhz") if clk else None)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and only is None:
        cpu = cpu_baseline(args, w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": config_string(w, S),
                       "step": f"verkv_compress + {S} x verkv_decode", "l2": "flushed (512 MB write) before every "
                       "call; flush not timed", "staging": "library default: ceil(eta n) rows per KV head",
                       "kernel_times": "a second pass of the same steps with an event pair around every kernel",
                       "parallelism": f"replicas x{world}"},
            "decode_us_per_step": statistics.mean(dec_ms) * 1e3,
            "decode_us_p50": statistics.median(dec_ms) * 1e3,
            "compress_us": statistics.mean(comp_ms) * 1e3,
            "compress_us_steps": [round(x * 1e3, 1) for x in comp_ms],
            "wall_ms_per_step": t_wall / args.steps * 1e3,
            "fetch_fraction_per_token": statistics.mean(fetch_frac) if fetch_frac else None,
            "host_rows_per_call": statistics.mean(host_rows) * w.n_kv,
            "union_rows_per_call": traces["union_rows"],
            "prefetch": {"rows_copied_per_call": statistics.mean(pf_copied) * w.n_kv,
                         "rows_used_per_call": statistics.mean(pf_used) * w.n_kv,
                         "precision": sum(pf_used) / max(1, sum(pf_copied))},
            "link_over_decode_job": job_link,
            "timeline_us": dict(timeline, note="median device times of the untimed statistics job's calls, us after "
                                               "the scoring kernel started (L2 flushed before each call; the "
                                               "decision starts once the scoring completes)"),
            "device_footprint": footprint(stats0, w, -2),
            "no_fetch_rate": no_fetch / max(1, len(kstars)),
            "mean_kstar": statistics.mean(kstars) if kstars else None,
            "kernel_share": {k: round(v[0] / total_ms, 4) for k, v in sorted(agg.items(), key=lambda kv: -kv[1][0])},
            "kernel_avg_us": {k: round(v[0] / v[1] * 1e3, 2) for k, v in agg.items()},
            "roofline": roofline, "roofline_score": roof_score, "roofline_score_issue": roof_issue,
            "roofline_attn": roof_hbm("attn"),
            "roofline_attn_link": roof_link("attn"), "roofline_decide": roof_decide,
            "host_link_peak_gbs": link_peak,
            "e2e": e2e, "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu,
        }
        line.update(secondary)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- secondary measurements
def timed_calls(calls, flush, st):
    """Run each call between its own event pair (L2 flushed, untimed, before each); returns ms."""
    import torch
    ev = []
    for c in calls:
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        c()
        b.record(st)
        ev.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def staging_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush, cap, link_peak):
    """The headline job with another staging capacity (0 = off: every fetched row crosses the host link
    at every step; -1 = every row of L minus S).  Decode time per call, rows per call, the footprint,
    and per fetching call the attention kernel's time (the fetch is fused into it): with staging off
    the rows that cross the link over that time is the fetch path's host-link rate."""
    import torch

    from verified_kv_cache_gb300 import binding
    ctx = binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=w.n, n_layers=1, n_seqs=1, max_batch=1,
                        n_sink=w.n_sink, n_local=w.n_local, eta=w.eta, seed=w.seed, sketch=w.sketch,
                        kv_dtype=w.kv_dtype)
    ctx.set_stage_capacity(cap)
    W, S = w.obs_q.shape[2], w.queries.shape[0]
    out = torch.empty_like(q_dev)
    stats = ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
    for s in range(S):   # warm-up job
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
    ms = []
    for _ in range(max(1, args.steps)):
        ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
        ms += timed_calls([lambda s=s: ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st) for s in range(S)],
                          flush, st)
    # one more job with per-kernel times and the rows of every call
    ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
    ctx.set_kernel_timing(True)
    union, host, attn_fetch_ms, host_fetch_rows = [], [], [], []
    for s in range(S):
        flush()
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
        kt = ctx.kernel_times(st)
        u = h = 0
        for kv in range(w.n_kv):
            a, b = ctx.fetch_stats(0, kv)
            u += a
            h += b
        union.append(u)
        host.append(h)
        if h > 0:
            attn_fetch_ms.append(sum(t for k, t in kt if k == "attn"))
            host_fetch_rows.append(h)
    ctx.set_kernel_timing(False)
    ctx.close()
    res = {"stage_rows_per_kv_head": {0: "off", -1: "all of L minus S"}.get(cap, cap),
           "decode_us_per_step": statistics.mean(ms) * 1e3, "decode_us_p50": statistics.median(ms) * 1e3,
           "union_rows_per_call": statistics.mean(union), "host_rows_per_call": statistics.mean(host),
           "fetch_fraction_per_token": statistics.mean(union) / (w.n_kv * w.n),
           "device_footprint": footprint(stats, w, cap)}
    if attn_fetch_ms:
        by = statistics.mean(host_fetch_rows) * ROW_BYTES
        t = statistics.mean(attn_fetch_ms)
        res["fetching_calls"] = len(attn_fetch_ms)
        res["attn_us_on_fetching_calls"] = t * 1e3
        res["host_bytes_per_fetching_call"] = by
        if link_peak:
            res["fetch_link"] = roof_entry("attn", t, by, link_peak, "GB/s", "host_link",
                                           "measured in this run: pinned host -> device copy of 256 MiB", None,
                                           "rows read over the host link by a fetching call / that call's "
                                           "attention kernel time (the fetch is fused into the attention)")
    return res


def binary_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush, shortlist=0):
    """The same workload with the binary shrinkage coefficients of Appendix A.2 (and, with shortlist >
    0, the Appendix A.1 shortlist and exact weights for sampled and shortlisted tokens): decode time
    (per-call events, L2 flushed before every call), fetch statistics and the kernel times."""
    import torch

    from verified_kv_cache_gb300 import binding
    ctx = binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=w.n, n_layers=1, n_seqs=1, max_batch=1,
                        n_sink=w.n_sink, n_local=w.n_local, eta=w.eta, seed=w.seed, sketch=w.sketch,
                        kv_dtype=w.kv_dtype, shrinkage="binary")
    if shortlist:
        ctx.set_shortlist(shortlist)
    W, S = w.obs_q.shape[2], w.queries.shape[0]
    out = torch.empty_like(q_dev)
    ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
    for s in range(S):   # warm-up
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
    ms = []
    for _ in range(max(1, args.steps)):
        ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
        ms += timed_calls([lambda s=s: ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st) for s in range(S)],
                          flush, st)
    fetch, nof, shr, ks = [], 0, [], []
    ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
    ctx.set_kernel_timing(True)
    for s in range(S):
        flush()
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
        tr = ctx.decode_trace(w.n_q)
        fetch += [ctx.fetch_stats(0, h)[0] / w.n for h in range(w.n_kv)]
        nof += sum(t["no_fetch"] for t in tr)
        shr += [t["n_shrunk"] for t in tr]
        ks += [t["kstar"] for t in tr]
    agg = kernel_agg(ctx.kernel_times(st))
    ctx.set_kernel_timing(False)
    ctx.close()
    return {"decode_us_per_step": statistics.mean(ms) * 1e3, "decode_us_p50": statistics.median(ms) * 1e3,
            "fetch_fraction_per_token": statistics.mean(fetch), "no_fetch_rate": nof / len(ks),
            "mean_kstar": statistics.mean(ks), "mean_n_shrunk": statistics.mean(shr),
            "kernel_avg_us": {k: round(v[0] / v[1] * 1e3, 2) for k, v in agg.items()}}


def growth_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush):
    """A serving loop on the same workload (decode-time growth, App. A.3.1): before each of the 64
    decode calls one generated token (random bf16 K/V rows, one per KV head, already on the device)
    is appended to H with verkv_append.  Time per step = append + decode (per-step events, L2 flushed
    before every step); the context grows from n to n + 64 over the job."""
    import torch

    from verified_kv_cache_gb300 import binding
    W, S = w.obs_q.shape[2], w.queries.shape[0]
    ctx = binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=w.n + S, n_layers=1, n_seqs=1, max_batch=1,
                        n_sink=w.n_sink, n_local=w.n_local, eta=w.eta, seed=w.seed, sketch=w.sketch,
                        kv_dtype=w.kv_dtype)
    ctx.set_append_capacity(S)
    g = torch.Generator(device=q_dev.device).manual_seed(31)
    new_kv = torch.randn((S, w.n_kv, 1, 2, w.d), generator=g, device=q_dev.device).to(torch.bfloat16)
    out = torch.empty_like(q_dev)
    ms = []
    for rep in range(1 + max(1, args.steps)):   # the first job is a warm-up
        ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)

        def step(s):
            ctx.append(0, 0, 1, new_kv[s], st)
            ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
        t = timed_calls([lambda s=s: step(s) for s in range(S)], flush, st)
        if rep > 0:
            ms += t
    assert ctx.appended(0, 0) == S
    ctx.close()
    return {"workload": "the bench layer with one token appended to H before every decode call",
            "us_per_step": statistics.mean(ms) * 1e3, "us_p50": statistics.median(ms) * 1e3,
            "tokens_appended_per_job": S}


# ----------------------------------------------------------------------------- seeded inputs on the GPU
def gpu_layer_inputs(seed, B, n, dev, Hkv=8, Hq=32, d=128, n_needles=16, W=32, steps=8, query_mode="needle_half",
                     qscale=1.0):
    """The Qwen3-4B-shaped layer's recipe (the same distributions as workloads.qwen_layer_case), drawn
    on the device from a seeded generator because the large configurations hold billions of values:
    K, V ~ N(0,1) in bf16, `n_needles` keys per KV head at distinct positions in [4, n - 128) scaled by
    4, observation queries N(0,1) [B, Hq, W, d], decode queries qscale N(0,1) [steps, B, Hq, d], of
    which the even steps aim at a needle of the head's KV group (q = 3 k_needle + N(0,1), needles
    round-robin) under "needle_half".  Returns (kv [B, Hkv, n, 2, d] bf16, obs, q) on the device."""
    import torch
    g = torch.Generator(device=dev).manual_seed(int(seed))
    K = torch.randn((B, Hkv, n, d), generator=g, device=dev)
    V = torch.randn((B, Hkv, n, d), generator=g, device=dev)
    nd = None
    if n_needles:
        keys = torch.rand((B, Hkv, n - 132), generator=g, device=dev)
        nd = keys.topk(n_needles, dim=-1).indices + 4          # distinct positions in [4, n - 128)
        K.scatter_(2, nd[..., None].expand(-1, -1, -1, d), 4.0 * K.gather(2, nd[..., None].expand(-1, -1, -1, d)))
    K = K.to(torch.bfloat16)
    kv = torch.stack([K, V.to(torch.bfloat16)], dim=3)
    del V
    obs = torch.randn((B, Hq, W, d), generator=g, device=dev) if W else None
    q = qscale * torch.randn((steps, B, Hq, d), generator=g, device=dev)
    if query_mode == "needle_half" and nd is not None:
        G = Hq // Hkv
        for s in range(0, steps, 2):
            for h in range(Hq):
                pos = nd[:, h // G, (s // 2 + h) % n_needles]                       # [B]
                q[s, :, h] += 3.0 * K[torch.arange(B, device=dev), h // G, pos].float()
    return kv, obs, q


def pinned_copy(t):
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def host_memory_bytes():
    """Memory this process may still pin: MemAvailable, capped by a cgroup limit if one is set."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    for p in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(p) as f:
                v = f.read().strip()
            if v.isdigit():
                lim = int(v)
                used = 0
                for q in ("/sys/fs/cgroup/memory.current", "/sys/fs/cgroup/memory/memory.usage_in_bytes"):
                    if os.path.exists(q):
                        with open(q) as g:
                            used = int(g.read().strip())
                        break
                avail = min(avail or lim, lim - used)
        except (OSError, ValueError):
            pass
    return avail


def layer_rooflines(agg, stats, w_like, traces, hbm_peak, peak_src, link_peak, batch):
    out = {}
    for k in ("score", "attn"):
        if k in agg:
            by = algorithmic_bytes(k, stats, traces, w_like, ROW_BYTES, batch=batch)
            out["roofline_" + k] = roof_entry(k, agg[k][0] / agg[k][1], by, hbm_peak, "GB/s", "hbm",
                                              f"{peak_src} hbm_gbs")
    if "attn" in agg and link_peak and traces.get("host_rows"):
        by = algorithmic_bytes("attn_link", stats, traces, w_like, ROW_BYTES, batch=batch)
        out["roofline_attn_link"] = roof_entry("attn", agg["attn"][0] / agg["attn"][1], by, link_peak, "GB/s",
                                               "host_link", "measured pinned host -> device copy")
    return out


class _W:
    """Shape record for algorithmic_bytes (the large configurations have no numpy workload)."""

    def __init__(self, n, eta, sketch, n_kv=8, n_q=32, d=128):
        self.n, self.eta, self.sketch, self.n_kv, self.n_q, self.d, self.kv_dtype = n, eta, sketch, n_kv, n_q, d, "bf16"


def stack36_run(args, dev, st, hbm_peak, peak_src, link_peak):
    """The 36-layer decode stack (attention only): batch 8 sequences of 32K tokens per layer, GQA 32/8,
    int8 sketch, eta = 1/32, eps = delta = 0.1, random per-layer queries, the full K/V of every layer and
    sequence in pinned host memory (36 GiB).  One job = every layer of the stack called in order for each
    of 128 decode steps (36 x 128 verkv_decode calls of batch 8); the working set of a layer call is
    larger than L2 and consecutive calls touch different layers, so L2 is not flushed.  When the host
    cannot pin the whole stack, the largest layer count that fits is run and reported."""
    import torch

    from verified_kv_cache_gb300 import binding
    B, n, Hkv, Hq, d, steps = 8, args.n, 8, 32, 128, 128
    eta, eps, delta = 1 / 32, 0.1, 0.1
    per_layer = B * Hkv * n * ROW_BYTES
    avail = host_memory_bytes()
    want = 4 if args.quick else args.stack_layers
    layers = want if avail is None else max(1, min(want, int(0.6 * avail // per_layer)))
    ctx = binding.VerKV(n_kv_heads=Hkv, n_q_heads=Hq, max_tokens=n, n_layers=layers, n_seqs=B, max_batch=B,
                        n_sink=4, n_local=128, eta=eta, seed=0, sketch="int8", kv_dtype="bf16")
    hosts, stats, qs = [], [], []
    t0 = time.perf_counter()
    for l in range(layers):
        kv, obs, q = gpu_layer_inputs(2000 + l, B, n, dev, n_needles=16, W=32, steps=steps, query_mode="random")
        for b in range(B):
            h = pinned_copy(kv[b])
            hosts.append(h)
            stats += ctx.compress(l, b, n, h, kv[b], obs[b], 32, None, st)
        qs.append(q)
        del kv, obs
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t0
    out = torch.empty((B, Hq, d), device=dev)
    ids = list(range(B))
    for s in range(2):   # warm-up: two steps through the stack
        for l in range(layers):
            ctx.decode(l, ids, qs[l][s], eps, delta, out, st)
    torch.cuda.synchronize()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for s in range(steps):
        for l in range(layers):
            ctx.decode(l, ids, qs[l][s], eps, delta, out, st)
    b_.record(st)
    torch.cuda.synchronize()
    job_ms = a.elapsed_time(b_)
    # per-kernel times and fetch fractions over the first 4 steps of the stack
    ctx.set_kernel_timing(True)
    fetch, host = [], []
    kt = []
    for s in range(4):
        for l in range(layers):
            ctx.decode(l, ids, qs[l][s], eps, delta, out, st)
            kt += ctx.kernel_times(st)
            for bb in range(B):
                for h in range(Hkv):
                    u, hr = ctx.fetch_stats(bb, h)
                    fetch.append(u / n)
                    host.append(hr)
    ctx.set_kernel_timing(False)
    # the prefetch's rows (copied beside the decision, read by the attention) over two more steps,
    # without per-kernel events (they would serialise the prefetch behind the decision)
    pf_c, pf_u = [], []
    for s in range(4, 6):
        for l in range(layers):
            ctx.decode(l, ids, qs[l][s], eps, delta, out, st)
            c_, u_ = 0, 0
            for bb in range(B):
                for h in range(Hkv):
                    pc, pu = ctx.prefetch_stats(bb, h)
                    c_ += pc
                    u_ += pu
            pf_c.append(c_)
            pf_u.append(u_)
    agg = kernel_agg(kt)
    calls = steps * layers
    traces = {"union_rows": statistics.mean(fetch) * n * B * Hkv, "host_rows": statistics.mean(host) * B * Hkv}
    wl = _W(n, eta, "int8")
    layer_stats = stats[:B * Hkv]
    res = {"workload": f"36-layer stack (attention only), batch {B} x n={n}, GQA {Hq}/{Hkv}, d={d}, bf16 K/V, int8 "
                       f"sketch, eta=1/32, eps=delta=0.1, random per-layer queries, {steps} decode steps",
           "layers_run": layers, "layers_wanted": want, "host_bytes_pinned": layers * per_layer,
           "host_memory_available": avail, "setup_s": setup_s,
           "job_ms": job_ms, "decode_us_per_layer_call": job_ms / calls * 1e3,
           "us_per_token_step_all_layers": job_ms / steps * 1e3,
           "scored_tokens_per_s": B * Hq * n * calls / (job_ms / 1e3),
           "fetch_fraction_per_token": statistics.mean(fetch), "host_rows_per_call": traces["host_rows"],
           "prefetch": {"rows_copied_per_call": statistics.mean(pf_c), "rows_used_per_call": statistics.mean(pf_u),
                        "precision": statistics.mean(pf_u) / max(1e-9, statistics.mean(pf_c))},
           "kernel_avg_us": {k: round(v[0] / v[1] * 1e3, 2) for k, v in agg.items()},
           "l2": "not flushed: per-layer working set above L2, layers called in turn"}
    res.update(layer_rooflines(agg, layer_stats, wl, traces, hbm_peak, peak_src, link_peak, B))
    ctx.close()
    del hosts, qs
    return res


def long_context_run(args, dev, st, hbm_peak, peak_src, link_peak):
    """The 128K long context: batch 1, GQA 32/8, 64 needles per KV head, int8 sketch, eta = 1/16,
    eps = 0.02, delta = 0.05, seeded synthetic importance scores (caller-supplied), queries scale x
    N(0,1) with the scale calibrated so that about 20% of L is fetched.  Staging default."""
    import numpy as np
    import torch

    from verified_kv_cache_gb300 import binding, workloads
    steps = 8
    w = workloads.long_context_case(n=131072, steps=steps)
    scores = torch.from_numpy(workloads.synthetic_scores(w.n_kv, w.n, seed=300)).to(dev)
    ctx = binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=w.n, n_layers=1, n_seqs=1, max_batch=1,
                        n_sink=w.n_sink, n_local=w.n_local, eta=w.eta, seed=w.seed, sketch=w.sketch,
                        kv_dtype=w.kv_dtype)
    kv_h = torch.from_numpy(w.kv_host_layout(0)).view(torch.bfloat16).pin_memory()
    kv_d = kv_h.to(dev)
    q = torch.from_numpy(np.ascontiguousarray(w.queries[:, :1])).to(dev)
    out = torch.empty_like(q)
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)
    comp = timed_calls([lambda: ctx.compress(0, 0, w.n, kv_h, kv_d, None, 0, scores, st)] * 3, flush, st)
    stats = ctx.compress(0, 0, w.n, kv_h, kv_d, None, 0, scores, st)
    dec = []
    for rep in range(3):
        ctx.compress(0, 0, w.n, kv_h, kv_d, None, 0, scores, st)
        t = timed_calls([lambda s=s: ctx.decode(0, [0], q[s], w.eps, w.delta, out[s], st) for s in range(steps)],
                        flush, st)
        if rep > 0:
            dec += t
    ctx.compress(0, 0, w.n, kv_h, kv_d, None, 0, scores, st)
    ctx.set_kernel_timing(True)
    fetch, host, ks, nl = [], [], [], []
    kt = []
    for s in range(steps):
        flush()
        ctx.decode(0, [0], q[s], w.eps, w.delta, out[s], st)
        kt += ctx.kernel_times(st)
        tr = ctx.decode_trace(w.n_q)
        ks += [t["kstar"] for t in tr]
        nl += [t["n_l"] for t in tr]
        for h in range(w.n_kv):
            u, hr = ctx.fetch_stats(0, h)
            fetch.append(u / w.n)
            host.append(hr)
    ctx.set_kernel_timing(False)
    agg = kernel_agg(kt)
    traces = {"union_rows": statistics.mean(fetch) * w.n * w.n_kv, "host_rows": statistics.mean(host) * w.n_kv}
    res = {"workload": f"long context n={w.n}, batch 1, GQA {w.n_q}/{w.n_kv}, 64 needles, int8 sketch, eta=1/16, "
                       f"eps={w.eps}, delta={w.delta}, query scale 1.3 (about 20% of L fetched), {steps} decode calls",
           "compress_us": statistics.mean(comp) * 1e3,
           "decode_us_per_call": statistics.mean(dec) * 1e3, "decode_us_p50": statistics.median(dec) * 1e3,
           "scored_tokens_per_s": w.n_q * w.n / (statistics.mean(dec) / 1e3),
           "fetch_fraction_per_token": statistics.mean(fetch),
           "kstar_over_L": statistics.mean(k / max(1, m) for k, m in zip(ks, nl)),
           "host_rows_per_call": traces["host_rows"],
           "kernel_avg_us": {k: round(v[0] / v[1] * 1e3, 2) for k, v in agg.items()}}
    res.update(layer_rooflines(agg, stats, w, traces, hbm_peak, peak_src, link_peak, 1))
    ctx.close()
    return res


def sweep_run(args, dev, st, hbm_peak, peak_src, link_peak, sm_mhz=None):
    """The sweep over 8 KV heads, d = 128, bf16: verkv_compress at n in {32K, 64K, 128K, 256K} (the
    whole compress: importance scores from 32 observation queries per query head, water-filling,
    Philox sample, compaction, int8 sketch; and with caller-supplied scores), and verkv_decode at
    n = 32K over eta in {1/8, 1/16, 1/32} x eps in {0.02, 0.05, 0.1}, delta = 0.05, batch in
    {1, 8, 32}, int8 sketch, the Qwen3-4B-shaped query mix (half aimed at needles): per point the
    decode time, scored tokens/s, fetch fraction and the score / attention rooflines; and one batch-8
    point (eta = 1/16, eps = 0.05) with the paper's 2-bit sketch."""
    import torch

    from verified_kv_cache_gb300 import binding
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)
    res = {"compress": [], "decode": [], "decode_2bit": []}
    ns = [32768, 65536] if args.quick else [32768, 65536, 131072, 262144]
    for n in ns:
        kv, obs, _ = gpu_layer_inputs(700 + n // 1024, 1, n, dev, n_needles=16, W=32, steps=1)
        h = pinned_copy(kv[0])
        ctx = binding.VerKV(n_kv_heads=8, n_q_heads=32, max_tokens=n, n_layers=1, n_seqs=1, max_batch=1, n_sink=4,
                            n_local=128, eta=1 / 16, seed=0, sketch="int8", kv_dtype="bf16")
        scores = torch.rand((8, n), device=dev) ** 4
        ctx.compress(0, 0, n, h, kv[0], obs[0], 32, None, st)
        t_obs = timed_calls([lambda: ctx.compress(0, 0, n, h, kv[0], obs[0], 32, None, st)] * 3, flush, st)
        t_tau = timed_calls([lambda: ctx.compress(0, 0, n, h, kv[0], None, 0, scores, st)] * 3, flush, st)
        res["compress"].append({"n": n, "eta": "1/16", "us_with_scores_from_observation_queries":
                                statistics.mean(t_obs) * 1e3, "us_with_caller_scores": statistics.mean(t_tau) * 1e3,
                                "tokens_per_s_caller_scores": 8 * n / (statistics.mean(t_tau) / 1e3)})
        ctx.close()
        del kv, obs, h
        torch.cuda.empty_cache()
    n = 32768
    batches = [1, 8] if args.quick else [1, 8, 32]
    etas = [1 / 16] if args.quick else [1 / 8, 1 / 16, 1 / 32]
    epss = [0.05] if args.quick else [0.02, 0.05, 0.1]
    steps = 8

    def point(ctx, B, eta, eps, sketch, q, ids, out, stats):
        """One decode point: event-timed calls, then per-kernel times, fetch statistics, rooflines."""
        for s in range(2):
            ctx.decode(0, ids, q[s], eps, 0.05, out, st)
        ms = timed_calls([lambda s=s: ctx.decode(0, ids, q[s], eps, 0.05, out, st) for s in range(steps)], flush, st)
        ctx.set_kernel_timing(True)
        fetch, host, kt = [], [], []
        for s in range(steps):
            flush()
            ctx.decode(0, ids, q[s], eps, 0.05, out, st)
            kt += ctx.kernel_times(st)
            for b in range(B):
                for hh in range(8):
                    u, hr = ctx.fetch_stats(b, hh)
                    fetch.append(u / n)
                    host.append(hr)
        ctx.set_kernel_timing(False)
        agg = kernel_agg(kt)
        traces = {"union_rows": statistics.mean(fetch) * n * B * 8, "host_rows": statistics.mean(host) * B * 8}
        pt = {"batch": B, "eta": f"1/{round(1 / eta)}", "eps": eps, "delta": 0.05, "sketch": sketch,
              "decode_us_per_call": statistics.mean(ms) * 1e3,
              "scored_tokens_per_s": B * 32 * n / (statistics.mean(ms) / 1e3),
              "fetch_fraction_per_token": statistics.mean(fetch),
              "kernel_avg_us": {k: round(v[0] / v[1] * 1e3, 2) for k, v in agg.items()}}
        rl = layer_rooflines(agg, stats, _W(n, eta, sketch), traces, hbm_peak, peak_src, link_peak, B)
        pt.update({k: round(v["frac"], 4) for k, v in rl.items()})
        # the 2-bit scan is bound by instruction issue: the committed ncu count of the batch-1 launch of
        # the bench layer, times the batch (the same work per KV head), over the launch's time, against
        # SMs x 4 issue slots x the SM clock sampled during the headline's timed region
        inst1 = measured_counters(_W(n, 1 / 16, "2bit")).get("warp_instructions_per_launch", {}).get("score")
        if sketch == "2bit" and inst1 and sm_mhz and "score" in agg:
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            avg_s = agg["score"][0] / agg["score"][1] / 1e3
            pt["roofline_score_issue"] = round(inst1 * B / avg_s / (sms * 4 * sm_mhz * 1e6), 4)
        return pt

    for B in batches:
        kv, obs, q = gpu_layer_inputs(800 + B, B, n, dev, n_needles=16, W=32, steps=steps)
        hosts = [pinned_copy(kv[b]) for b in range(B)]
        out = torch.empty((B, 32, 128), device=dev)
        ids = list(range(B))
        sketches = ["int8", "2bit"] if B == 8 else ["int8"]
        for sketch in sketches:
            for eta in (etas if sketch == "int8" else [1 / 16]):
                ctx = binding.VerKV(n_kv_heads=8, n_q_heads=32, max_tokens=n, n_layers=1, n_seqs=B, max_batch=B,
                                    n_sink=4, n_local=128, eta=eta, seed=0, sketch=sketch, kv_dtype="bf16")
                stats = []
                for b in range(B):
                    stats += ctx.compress(0, b, n, hosts[b], kv[b], obs[b], 32, None, st)
                for eps in (epss if sketch == "int8" else [0.05]):
                    pt = point(ctx, B, eta, eps, sketch, q, ids, out, stats)
                    res["decode" if sketch == "int8" else "decode_2bit"].append(pt)
                ctx.close()
        del kv, obs, q, hosts
        torch.cuda.empty_cache()
    res["note"] = ("roofline_* per point are fractions: score and attn of the measured HBM copy peak, attn_link of "
                   "the measured host-link peak; int8 sketch (the configs' sketch) in `decode`, one batch-8 point "
                   "with the paper's 2-bit sketch in `decode_2bit`")
    return res


# ----------------------------------------------------------------------------- the oracle (CPU)
def oracle_sample(w, steps, threads):
    """One bounded oracle pass over the workload: compress of every KV head (importance scores,
    water-filling, Poisson sample, sketch) and the given decode steps (every query row: logits, the
    decision with the oracle's O(|L| log |L|) closed forms, the attention), spread over `threads`
    host threads (the oracle's C calls release the interpreter lock).  Returns (compress_s, decode_s)."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    G, Wn = w.group, w.obs_q.shape[2]

    def comp(h):
        tau = oracle.tau(w.K[0, h], w.obs_q[0, h * G:(h + 1) * G].reshape(G * Wn, w.d), w.n_sink, w.n_local)
        _, _, _, r = oracle.waterfill(tau, w.n_sink, w.n_local, w.eta * w.n)
        f = oracle.poisson_sample(r, w.seed, h, 0, 0)
        sk = oracle.sketch_2bit(w.K[0, h]) if w.sketch == "2bit" else oracle.sketch_int8(w.K[0, h])
        return f, r, sk

    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        state = list(ex.map(comp, range(w.n_kv)))
        t1 = time.perf_counter()

        def row(args_):
            s, hq = args_
            h = hq // G
            f, r, sk = state[h]
            q = w.queries[s, 0, hq].astype(np.float64)
            te = oracle.logits_exact(q, w.K[0, h])
            ts = oracle.logits_2bit(q, *sk) if w.sketch == "2bit" else oracle.logits_int8(q, *sk)
            res = oracle.kvfetch_row(f, r, te, ts, w.eps, w.delta, mode=1)
            oracle.attention_row(f, r, te, w.V[0, h], res["lam"], res["exact_mask"])

        list(ex.map(row, [(s, hq) for s in steps for hq in range(w.n_q)]))
        t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def cpu_baseline(args, w):
    """The oracle on the host cores over one whole job of the headline workload (compress + every
    decode step), measured, not extrapolated."""
    threads = os.cpu_count() or 1
    S = w.queries.shape[0]
    comp_s, dec_s = oracle_sample(w, range(S), threads)
    return {"value": S * w.n_q * w.n / (comp_s + dec_s), "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"one whole job: oracle compress of all {w.n_kv} KV heads + all {S} decode steps (all {w.n_q} "
                      f"query rows each) on {threads} host threads (a thread per KV head, then per query row)",
            "compress_s": comp_s, "decode_s_per_step": dec_s / S}


REF_DECODE_STEPS = 16   # decode steps per reference-arm step: a quarter of the job, 8 needle and 8 random queries


def run_reference(args):
    """The reference arm: the oracle on the host cores.  Each step is a measured quarter of the headline
    job: the compress and the first 16 of its 64 decode steps (8 aimed at needles, 8 random); value =
    the scored tokens of those 16 steps / the step's time, so the compress weighs four times as much as
    in a whole job (it is about a sixth of a step).  The warm-up steps run the compress and one decode
    step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args, 0)
    S = w.queries.shape[0]
    k = min(REF_DECODE_STEPS, S)
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_sample(w, range(1), threads)
    times, comps, decs = [], [], []
    for _ in range(args.steps):
        c, d = oracle_sample(w, range(k), threads)
        times.append(c + d)
        comps.append(c)
        decs.append(d)
    step_s = statistics.mean(times)
    value = k * w.n_q * w.n / step_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": config_string(w, S), "step": f"oracle compress + decode steps 0..{k - 1} of the job",
                       "parallelism": f"{threads} host threads"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "cpu_model": cpu_model(),
                             "sample": f"each step: oracle compress of all KV heads + decode steps 0..{k - 1} of the "
                                       f"{S}-step job ({k // 2} needle, {k - k // 2} random queries) on {threads} host "
                                       f"threads, measured; value = scored tokens of those {k} steps / step time; "
                                       f"warm-up steps: compress + 1 decode step"},
            "compress_s": statistics.mean(comps), "decode_s_per_step": statistics.mean(decs) / k,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_verkv(args)


if __name__ == "__main__":
    main()
