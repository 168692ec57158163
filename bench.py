#!/usr/bin/env python
"""Benchmark of the VerKV hot path on one GB300: PoissonComp + KVFetch on the Qwen3-4B-shaped
32K-token attention layer (batch 1, GQA 32/8, d = 128, bf16 K/V, 16 needles per KV head, 2-bit key
sketch of the paper's Appendix A.1, eta = 1/16, eps = delta = 0.05, 64 decode steps with half the
queries aimed at needles).

One bench step = one pass of the whole hot path over one job: verkv_compress of the 32K context
(importance scores, water-filling, Poisson sample, compaction, sketch) followed by the 64
verkv_decode calls.  Inputs are resident in HBM (plus the pinned host copy the decode fetches from)
when the timed region starts; L2 is flushed (a 512 MB write) before every call and the flush is not
timed.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl verkv|reference]
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
    p.add_argument("--no-secondary", action="store_true",
                   help="skip the binary-shrinkage and batch-8 stack-layer measurements")
    p.add_argument("--only-stack", action="store_true",
                   help="(profiling runs) only the batch-8 stack-layer measurement, printed as one JSON line")
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
def algorithmic_bytes(kernel, stats, traces, w, row_bytes, batch=1):
    """Bytes each kernel must move by the method's definition (per launch), from the compressed sizes
    and the decode traces.  Intermediates a kernel writes for the next one are not counted.  `stats`
    holds the head statistics of every sequence of the batch."""
    Hkv, Hq, n, d = w.n_kv, w.n_q, w.n, w.d
    L = sum(s["n_l"] for s in stats)
    H = sum(s["n_h"] for s in stats)
    R = sum(s["n_resident"] for s in stats)
    sk = {"2bit": (d // 4) * 2 / 8 + (d // 4) * 4 / 128, "int8": d + 4, "exact": d * (2 if w.kv_dtype == "bf16" else 4)}
    s_sk = sk[w.sketch]
    if kernel == "score":             # sketch of every L token, the L/H position of every token,
        return L * s_sk + batch * Hkv * n * 4 + H * row_bytes / 2 + batch * Hq * d * 4   # exact keys of H, q
    if kernel == "weights":           # r of L
        return L * 4 * (Hq // Hkv)
    if kernel == "decide":            # per query row and L entry: its float-float logit, r, the two ratios
        return L * (Hq // Hkv) * (8 + 4 + 8 + 4 + 4)   # of r, the resident slot; w^ written back
    if kernel == "attn":              # resident K/V rows from HBM once per KV head, the fetched rows found
        staged = traces.get("union_rows", 0) - traces.get("host_rows", 0)   # in the staging cache, the
        return (R + staged + traces.get("host_rows", 0)) * row_bytes + batch * Hq * d * 8   # rows staged, q/out
    if kernel == "attn_link":         # the fetched rows that crossed the host link, once per KV head
        return traces.get("host_rows", 0) * row_bytes
    return None


def measured_traffic(w):
    """DRAM bytes per launch of the decode kernels from the committed ncu summary of this workload, if
    the kernel source is the one the counters were taken on (else {}: the kernels changed since)."""
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
    return rec["dram_bytes_per_launch"] if sha == rec["source_sha256"] else {}


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
    # warm-up
    for _ in range(max(args.warmup, 0)):
        one_step([])
    torch.cuda.synchronize()
    # fetch statistics of the workload (one untimed decode sweep with traces)
    ctx.compress(0, 0, w.n, kv_host, kv_dev, obs, W, None, st)
    fetch_frac, no_fetch, union_rows, host_rows, kstars = [], 0, [], [], []
    for s in range(S):
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
        tr = ctx.decode_trace(w.n_q)
        for h in range(w.n_kv):
            u, hr = ctx.fetch_stats(0, h)
            union_rows.append(u)
            host_rows.append(hr)
            fetch_frac.append(u / w.n)
        no_fetch += sum(t["no_fetch"] for t in tr)
        kstars += [t["kstar"] for t in tr]
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
    # rooflines and the kernel shares
    ctx.set_kernel_timing(True)
    kt = []
    for _ in range(args.steps):
        one_step([])
        kt += ctx.kernel_times(st)   # drains the per-kernel records (one sync between steps)
    torch.cuda.synchronize()
    ctx.set_kernel_timing(False)
    comp_ms = [a.elapsed_time(b) for k, a, b in events if k == "compress"]
    dec_ms = [a.elapsed_time(b) for k, a, b in events if k == "decode"]
    step_ms = (sum(comp_ms) + sum(dec_ms)) / args.steps
    units_per_step = S * 1 * w.n_q * w.n        # scored tokens: every query head scores every token
    value, step_ms = aggregate_ranks(step_ms, units_per_step, world, dev)

    # per-kernel shares and the dominant kernel
    agg = {}
    for name, ms in kt:
        a = agg.setdefault(name, [0.0, 0])
        a[0] += ms
        a[1] += 1
    total_ms = sum(v[0] for v in agg.values())
    dec_kernels = {k: v for k, v in agg.items() if k not in ("tau_tile", "tau_rowstat", "tau_finish", "waterfill",
                                                             "sample", "compact", "gather_resident", "pair_energy",
                                                             "select_pairs", "sketch_2bit", "sketch_int8",
                                                             "copy_keys")}
    dom = max(agg.items(), key=lambda kv: kv[1][0])[0] if agg else None
    row_bytes = 2 * w.d * 2
    traces = {"union_rows": statistics.mean(union_rows) * w.n_kv if union_rows else 0,
              "host_rows": statistics.mean(host_rows) * w.n_kv if host_rows else 0}

    import json as _json
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) \
            else open(os.devnull) as f:
        try:
            peaks = _json.load(f)
        except Exception:
            peaks = {}
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0

    traffic = measured_traffic(w)
    traffic_note = ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch (profiles/traffic_*.txt); rows "
                    "fetched from pinned host memory cross NVLink-C2C and are not DRAM traffic") if traffic else \
        "null: no ncu capture of the current kernel source"

    def roof(kname):
        if kname not in agg:
            return None
        avg_ms = agg[kname][0] / agg[kname][1]
        by = algorithmic_bytes(kname, stats0, traces, w, row_bytes)
        if by is None:
            return {"kernel": kname, "bound": "latency", "avg_us": avg_ms * 1e3, "achieved": None, "peak": None,
                    "unit": None, "frac": None, "traffic": None}
        ach = by / (avg_ms / 1e3) / 1e9
        return {"kernel": kname, "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                "frac": ach / hbm_peak, "traffic": traffic.get(kname), "traffic_note": traffic_note,
                "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes": by, "avg_us": avg_ms * 1e3}

    # host-link peak: a bulk pinned host -> device copy (the same link the fetch uses)
    link_peak = None
    if rank == 0:
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
        link_peak = src.numel() / (best / 1e3) / 1e9
        del src, dst

    def roof_link(kname):
        if kname not in agg or not link_peak:
            return None
        avg_ms = agg[kname][0] / agg[kname][1]
        by = algorithmic_bytes(kname + "_link", stats0, traces, w, row_bytes)
        ach = by / (avg_ms / 1e3) / 1e9
        return {"kernel": kname, "bound": "host_link", "achieved": ach, "peak": link_peak, "unit": "GB/s",
                "frac": ach / link_peak, "traffic": traffic.get(kname), "traffic_note": traffic_note,
                "peak_source": "measured in this run: pinned host -> device copy of 256 MiB",
                "algorithmic_bytes": by, "avg_us": avg_ms * 1e3}

    # the attention kernel also carries the fetch: its bound is the resource whose bytes take longer
    # at peak (the host link for the rows that cross it, HBM for the resident and staged rows)
    roofline = roof(dom)
    if dom == "attn" and link_peak:
        t_link = algorithmic_bytes("attn_link", stats0, traces, w, row_bytes) / link_peak
        t_hbm = algorithmic_bytes("attn", stats0, traces, w, row_bytes) / hbm_peak
        if t_link >= t_hbm:
            roofline = roof_link(dom)
    roof_score = roof("score")
    roof_attn = roof("attn")
    roof_link_attn = roof_link("attn")

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

    secondary = {}
    if rank == 0 and not args.no_secondary:
        secondary["binary_shrinkage"] = binary_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush)
        secondary["deployed_binary_shortlist128"] = binary_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush,
                                                               shortlist=128)
        secondary["growth_append1"] = growth_run(args, w, kv_host, kv_dev, obs, q_dev, st, flush)
    ctx.close()
    if rank == 0 and not args.no_secondary:
        del kv_dev, flush_buf
        torch.cuda.empty_cache()
        secondary["stack_layer_b8_int8"] = stack_run(args, dev, st, hbm_peak, peak_src)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"qwen3-4b-shaped attention layer, n={w.n}, batch 1, GQA {w.n_q}/{w.n_kv}, "
                                   f"d={w.d}, bf16 K/V, {w.sketch} sketch, eta=1/{round(1 / w.eta)}, "
                                   f"eps={w.eps}, delta={w.delta}, {S} decode steps per job (compress + decodes)",
                       "step": "verkv_compress + 64 x verkv_decode", "l2": "flushed (512 MB write) before every "
                       "call; flush not timed", "kernel_times": "a second pass of the same steps with an "
                       "event pair around every kernel", "parallelism": f"replicas x{world}"},
            "decode_us_per_step": statistics.mean(dec_ms) * 1e3,
            "decode_us_p50": statistics.median(dec_ms) * 1e3,
            "compress_us": statistics.mean(comp_ms) * 1e3,
            "compress_us_steps": [round(x * 1e3, 1) for x in comp_ms],
            "wall_ms_per_step": t_wall / args.steps * 1e3,
            "fetch_fraction_per_token": statistics.mean(fetch_frac) if fetch_frac else None,
            "host_rows_per_call": traces["host_rows"], "union_rows_per_call": traces["union_rows"],
            "staging": "rows fetched over the host link are kept in device memory and re-used by later calls of "
                       "the job (cleared by each compress)",
            "no_fetch_rate": no_fetch / max(1, len(kstars)),
            "mean_kstar": statistics.mean(kstars) if kstars else None,
            "kernel_share": {k: round(v[0] / total_ms, 4) for k, v in sorted(agg.items(), key=lambda kv: -kv[1][0])},
            "kernel_avg_us": {k: round(v[0] / v[1] * 1e3, 2) for k, v in agg.items()},
            "roofline": roofline, "roofline_score": roof_score, "roofline_attn": roof_attn,
            "roofline_attn_link": roof_link_attn, "host_link_peak_gbs": link_peak,
            "e2e": e2e, "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu,
        }
        line.update(secondary)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- secondary measurements
def _kernel_agg(kt):
    agg = {}
    for name, ms in kt:
        a = agg.setdefault(name, [0.0, 0])
        a[0] += ms
        a[1] += 1
    return agg


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
        for s in range(S):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
            b.record(st)
            ms.append((a, b))
    torch.cuda.synchronize()
    dec_ms = [a.elapsed_time(b) for a, b in ms]
    fetch, nof, shr, ks = [], 0, [], []
    ctx.set_kernel_timing(True)
    for s in range(S):
        flush()
        ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
        tr = ctx.decode_trace(w.n_q)
        fetch += [len(ctx.fetch_set(0, h, w.n)) / w.n for h in range(w.n_kv)]
        nof += sum(t["no_fetch"] for t in tr)
        shr += [t["n_shrunk"] for t in tr]
        ks += [t["kstar"] for t in tr]
    agg = _kernel_agg(ctx.kernel_times(st))
    ctx.set_kernel_timing(False)
    ctx.close()
    return {"decode_us_per_step": statistics.mean(dec_ms) * 1e3, "decode_us_p50": statistics.median(dec_ms) * 1e3,
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
        for s in range(S):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            ctx.append(0, 0, 1, new_kv[s], st)
            ctx.decode(0, [0], q_dev[s], w.eps, w.delta, out[s], st)
            b.record(st)
            if rep > 0:
                ms.append((a, b))
    torch.cuda.synchronize()
    assert ctx.appended(0, 0) == S
    step_ms = [a.elapsed_time(b) for a, b in ms]
    ctx.close()
    return {"workload": "the bench layer with one token appended to H before every decode call",
            "us_per_step": statistics.mean(step_ms) * 1e3, "us_p50": statistics.median(step_ms) * 1e3,
            "tokens_appended_per_job": S}


def stack_run(args, dev, st, hbm_peak, peak_src):
    """One layer of the 36-layer stack workload: batch 8 sequences of 32K tokens, GQA 32/8, int8
    sketch, eta = 1/32, eps = delta = 0.1, random queries.  Per-call events (L2 flushed before every
    call) and per-kernel events; the HBM roofline of the sketch scan and of the attention at batch 8."""
    import torch

    from verified_kv_cache_gb300 import binding, workloads
    B, steps = 8, 16
    w = workloads.stack_layer_case(layer=0, n=args.n, batch=B, steps=steps)
    ctx = binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=w.n, n_layers=1, n_seqs=B, max_batch=B,
                        n_sink=w.n_sink, n_local=w.n_local, eta=w.eta, seed=w.seed, sketch=w.sketch,
                        kv_dtype=w.kv_dtype)
    W = w.obs_q.shape[2]
    stats, hosts = [], []
    for b in range(B):
        kv_h = torch.from_numpy(w.kv_host_layout(b)).view(torch.bfloat16).pin_memory()
        hosts.append(kv_h)
        kv_d = kv_h.to(dev)
        obs = torch.from_numpy(w.obs_q[b]).to(dev)
        stats += ctx.compress(0, b, w.n, kv_h, kv_d, obs, W, None, st)
        del kv_d
    q = torch.from_numpy(w.queries).to(dev)             # [steps, B, Hq, d]
    out = torch.empty_like(q)
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    ids = list(range(B))
    for s in range(3):
        ctx.decode(0, ids, q[s], w.eps, w.delta, out[s], st)
    ev = []
    for s in range(steps):
        flush_buf.fill_(1.0)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        ctx.decode(0, ids, q[s], w.eps, w.delta, out[s], st)
        b_.record(st)
        ev.append((a, b_))
    torch.cuda.synchronize()
    dec_ms = [a.elapsed_time(b_) for a, b_ in ev]
    ctx.set_kernel_timing(True)
    fetch = []
    for s in range(steps):
        flush_buf.fill_(1.0)
        ctx.decode(0, ids, q[s], w.eps, w.delta, out[s], st)
        for b in range(B):
            fetch += [len(ctx.fetch_set(b, h, w.n)) / w.n for h in range(w.n_kv)]
    agg = _kernel_agg(ctx.kernel_times(st))
    ctx.set_kernel_timing(False)
    row_bytes = 2 * w.d * 2

    def roof(k):
        if k not in agg:
            return None
        avg_ms = agg[k][0] / agg[k][1]
        by = algorithmic_bytes(k, stats, {}, w, row_bytes, batch=B)
        ach = by / (avg_ms / 1e3) / 1e9
        return {"kernel": k, "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                "traffic": None, "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes": by,
                "avg_us": avg_ms * 1e3}

    res = {"workload": f"stack layer: batch {B} x n={w.n}, GQA {w.n_q}/{w.n_kv}, int8 sketch, eta=1/32, "
                       f"eps=delta=0.1, {steps} decode calls, random queries",
           "decode_us_per_call": statistics.mean(dec_ms) * 1e3,
           "scored_tokens_per_s": B * w.n_q * w.n / (statistics.mean(dec_ms) / 1e3),
           "fetch_fraction_per_token": statistics.mean(fetch) if fetch else None,
           "kernel_avg_us": {k: round(v[0] / v[1] * 1e3, 2) for k, v in agg.items()},
           "roofline_score": roof("score"), "roofline_attn": roof("attn")}
    ctx.close()
    del hosts, flush_buf
    return res


# ----------------------------------------------------------------------------- the oracle (CPU)
def oracle_sample(w, decode_steps):
    """One bounded oracle pass: compress of all KV heads and `decode_steps` decode steps (all query
    rows, the oracle's O(|L| log |L|) closed forms).  Returns (compress_s, decode_s)."""
    import numpy as np

    import oracle
    G, Wn = w.group, w.obs_q.shape[2]
    t0 = time.perf_counter()
    flags, r32, sk = [], [], []
    for h in range(w.n_kv):
        tau = oracle.tau(w.K[0, h], w.obs_q[0, h * G:(h + 1) * G].reshape(G * Wn, w.d), w.n_sink, w.n_local)
        c, _, _, r = oracle.waterfill(tau, w.n_sink, w.n_local, w.eta * w.n)
        flags.append(oracle.poisson_sample(r, w.seed, h, 0, 0))
        r32.append(r)
        sk.append(oracle.sketch_2bit(w.K[0, h]) if w.sketch == "2bit" else oracle.sketch_int8(w.K[0, h]))
    t1 = time.perf_counter()
    for s in range(decode_steps):
        for hq in range(w.n_q):
            h = hq // G
            q = w.queries[s, 0, hq].astype(np.float64)
            te = oracle.logits_exact(q, w.K[0, h])
            ts = oracle.logits_2bit(q, *sk[h]) if w.sketch == "2bit" else oracle.logits_int8(q, *sk[h])
            res = oracle.kvfetch_row(flags[h], r32[h], te, ts, w.eps, w.delta, mode=1)
            oracle.attention_row(flags[h], r32[h], te, w.V[0, h], res["lam"], res["exact_mask"])
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def cpu_baseline(args, w, decode_steps=2):
    comp_s, dec_s = oracle_sample(w, decode_steps)
    S = args.decode_steps
    # one job = compress + S decodes; the sample runs compress once and `decode_steps` decodes
    job_s = comp_s + dec_s * S / decode_steps
    value = S * w.n_q * w.n / job_s
    return {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"oracle compress of all {w.n_kv} KV heads + {decode_steps} of {S} decode steps (all "
                      f"{w.n_q} query rows), single thread; job time = compress + decode time x {S}/{decode_steps}",
            "compress_s": comp_s, "decode_s_per_step": dec_s / decode_steps}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args, 0)
    S = args.decode_steps
    dec_steps = 1
    for _ in range(args.warmup):
        oracle_sample(w, dec_steps)
    times = []
    for _ in range(args.steps):
        c, d = oracle_sample(w, dec_steps)
        times.append(c + d * S / dec_steps)
    job_s = statistics.mean(times)
    value = S * w.n_q * w.n / job_s
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": job_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"qwen3-4b-shaped attention layer, n={w.n}, batch 1, GQA {w.n_q}/{w.n_kv}, "
                                   f"{w.sketch} sketch, {S} decode steps per job"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"each step: oracle compress + {dec_steps} decode step, job time = compress "
                                       f"+ decode x {S}/{dec_steps}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse()
    if args.only_stack:
        import torch

        from verified_kv_cache_gb300 import build
        build.build()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        peaks = {}
        pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
        if os.path.exists(pk):
            with open(pk) as f:
                peaks = json.load(f)
        hbm = peaks.get("hbm_gbs")
        print(json.dumps({"stack_layer_b8_int8": stack_run(args, dev, torch.cuda.current_stream(), hbm or 6800.0,
                                                           "measured" if hbm else "fallback")}))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_verkv(args)


if __name__ == "__main__":
    main()
