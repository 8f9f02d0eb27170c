"""Benchmark: effective HBM GB/s and busBW of the chunk-schedule executor.

One *step* executes every collective of the suite once, each on its own
synthetic inputs resident in HBM:

  hier_ar   hierarchical AllReduce, R=16 (2 groups x 8), fp32, 64 MiB/rank, 16 micro-batches
  a2a       two-phase AllToAll, R=32 (4 x 8), fp16, 1 MiB block per (src, dst)
  ring_bf16 ring AllReduce, R=8, bf16, 256 MiB/rank, 24 channels
  ring_f32  ring AllReduce, R=8, fp32, 256 MiB/rank, 24 channels
  a2n       AllToNext, R=24 (3 x 8), fp32, 128 MiB/rank, relayed cross-group pairs
  ag_3m     ring AllGather, R=8, bf16, 3 MiB/rank output, 4 channels
  rs_3m     ring ReduceScatter, R=8, bf16, 3 MiB/rank input, 4 channels
  ar_1m     ring AllReduce, R=8, fp32, 1 MiB/rank, 1 channel

value = schedule bytes of the step (bytes every fused instruction reads and
writes, FIFO staging included) / device time of the step.  A schedule that
moves fewer bytes (direct transport, unchained copy hops) lowers the step
time and the byte count together; collective_min_bytes_gbs (each input read
once, each output written once, per second) does not depend on that choice.  The step's working
set (~19 GiB) is far larger than L2, so consecutive collectives evict each
other; no separate flush.

``--impl reference`` times the CPU oracle (single thread) on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MiB = 1 << 20

# name, kind, R, G, dtype, bytes per chunk, dist, seed, plan options
SUITE = [
    # parameters the workload fixes are kept (24 channels, 16 micro-batches,
    # 1 channel, <= 4 channels); the others are the best measured settings.
    # fuse="nochain": reductions fused, copy-only receives left unchained so
    # that direct transport makes each all-gather hop one plain copy
    ("hier_ar", 3, 16, 8, 0, 4 * MiB, "normal", 2,
     # (every fold: the in-group reduce-scatter runs two ranks per step, the
     # inter-group send joins the step it feeds, the in-group all-gather's
     # copies run two ranks per step)
     dict(fuse="nochain", link_mode=1, channels=8, microbatches=16, tb_alloc=1, slot_bytes=65536, fifo_slots=8,
          mb_window=4, fold=7)),
    ("a2a", 4, 32, 8, 2, 1 * MiB, "uniform", 3,
     dict(channels=8, link_mode=1, channel_scaling=0, tb_alloc=2, tb_budget=256)),
    # reduce-scatter steps two ranks at a time (reduction chains folded),
    # all-gather copies two ranks at a time (copy chains folded)
    ("ring_bf16", 0, 8, 0, 1, 32 * MiB, "normal", 4,
     dict(fuse="nochain", link_mode=1, channels=24, slot_bytes=131072, microbatches=16, fifo_slots=4, tb_alloc=2,
          tb_budget=192, fold=7)),
    ("ring_f32", 0, 8, 0, 0, 32 * MiB, "normal", 4,
     dict(fuse="nochain", link_mode=1, channels=24, slot_bytes=131072, microbatches=16, fifo_slots=4, tb_alloc=2,
          tb_budget=192, fold=7)),
    # relay hops as plain direct copies (no fusion into FIFO forwards); the
    # link-free copies binned into 144 threadblocks, one per SM (the
    # 512-thread build)
    ("a2n", 5, 24, 8, 0, 16 * MiB, "normal", 4,
     dict(fuse=False, channels=16, link_mode=1, microbatches=16, tb_alloc=2, tb_budget=152, channel_scaling=0,
          fold=15)),
    ("ag_3m", 1, 8, 0, 1, 3 * MiB // 8, "normal", 1,
     # every hop a direct copy into the next rank's output (no FIFO), the
     # first one in the same pass as the rank's own block (a copy-send with
     # its receive folded in); the small collectives run on the sequential
     # engine (fewer hand-offs per step), each program on a cluster of CTAs
     # that share its slots' data
     # (copy chains three hops per step: 3 steps per program)
     dict(fuse="nochain", channels=4, link_mode=1, engine=1, cluster=4, nthreads=256, fold=15)),
    # FIFOs at least one execution deep (8 slots): no slot is reused within
    # an execution, so nothing is posted or waited for its consumption
    ("rs_3m", 2, 8, 0, 1, 3 * MiB // 8, "normal", 1, dict(channels=4, engine=1, cluster=4, nthreads=256,
                                                          fifo_slots=8, fold=7)),
    ("ar_1m", 0, 8, 0, 0, 1 * MiB // 8, "uniform", 0, dict(fuse="nochain", link_mode=1, channels=1, tb_alloc=2,
                                                            tb_budget=16, engine=1, cluster=8, nthreads=128,
                                                            fifo_slots=8, fold=15)),
]
ESIZE = {0: 4, 1: 2, 2: 2, 3: 4}
NAMES = {0: "f32", 1: "bf16", 2: "f16", 3: "i32"}
METRIC = "effective HBM GB/s & busBW per collective vs GB300 HBM roofline, 1 GPU"


def sources_hash():
    """Key of the DRAM traffic recorded in profiles/: the executor and planner
    sources, the suite rows that run on the pipelined kernel (the launches
    the traffic covers) and the instruction lists the compiler makes of
    them.  The compiler's source stands in only through its output, so a
    compiler change that leaves these schedules alone keeps the record."""
    import glob
    import hashlib
    import collective_communication_schedule_gb300 as ccl
    csrc = os.path.join(ROOT, "collective_communication_schedule_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                   glob.glob(os.path.join(csrc, "*.cpp")) + glob.glob(os.path.join(csrc, "*.h")),
                   key=os.path.basename)
    h = hashlib.sha256()
    for f in files:
        if os.path.basename(f) == "ccl_compiler.cpp":
            continue
        with open(f, "rb") as fh:
            h.update(fh.read())
    rows = [r for r in SUITE if r[8].get("engine", 0) != 1]
    h.update(repr(rows).encode())
    for name, kind, R, G, dt, cb, dist, seed, opts in rows:
        sched, _ = schedule_and_opts(ccl, kind, R, G, opts)
        h.update(repr([tuple(sorted(d.items())) for d in sched.instrs()]).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when it records another kernel or when the sources or the suite
    changed since it was captured."""
    try:
        kv = {}
        with open(os.path.join(ROOT, "profiles", "roofline_traffic.txt")) as f:
            for line in f:
                if line.strip() and not line.startswith("#"):
                    k, v = line.split(None, 1)
                    kv[k] = v.strip()
        if kv.get("sources_sha256_16") != sources_hash() or kv.get("kernel") != kernel:
            return None
        return int(kv["traffic_bytes_per_launch"])
    except Exception:
        return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_name(stats):
    """The executor kernel a plan launches: engine, protocol and the thread
    limit it was built for (512: eight vectors in flight per thread, 1024:
    four)."""
    maxt = stats.kernel_build or (512 if stats.nthreads <= 512 else 1024)
    if stats.engine == 1:
        return f"ccl_exec_seq_kernel<{maxt}>"
    return "ccl_exec_kernel<LL, 512>" if stats.protocol == 1 else f"ccl_exec_kernel<simple, {maxt}>"


def schedule_and_opts(ccl, kind, R, G, opts):
    """The built-in schedule of a suite row (the row's `fuse` key chooses
    the compiler's fusion: True, False or "nochain") and the remaining plan
    options."""
    opts = dict(opts)
    fuse = opts.pop("fuse", True)
    flags = ccl.FLAG_NOCHAIN_COPIES if fuse == "nochain" else (0 if fuse else ccl.FLAG_NOFUSE)
    return ccl.Schedule.builtin(kind, R, G, flags), opts


def combine_replicas(res, world, device=None):
    """Whole-job line of N replicas: step times are the maximum over ranks
    (device and end-to-end), values count the bytes of every replica."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([res["ms_per_step"], res["e2e"]["ms_per_step"]], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms, e2e_ms = float(t[0].item()), float(t[1].item())
    out = dict(res)
    sb = res["config"]["schedule_bytes_per_step"]
    out["ms_per_step"] = round(ms, 4)
    out["value"] = round(sb * world / (ms * 1e6), 1)
    out["n_gpus"] = world
    out["e2e"] = dict(res["e2e"], ms_per_step=round(e2e_ms, 3), value=round(sb * world / (e2e_ms * 1e6), 1),
                      h2d_bytes_per_step=res["e2e"]["h2d_bytes_per_step"] * world,
                      d2h_bytes_per_step=res["e2e"]["d2h_bytes_per_step"] * world)
    out["gpu_launches"] = res["gpu_launches"] * world
    return out


def barrier():
    """Barrier across replicas (no-op on one GPU)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def selected_suite(args):
    """The suite, or a subset (--only) at reduced chunk size (--scale) for
    profiling captures."""
    out = []
    only = set(args.only.split(",")) if getattr(args, "only", None) else None
    for row in SUITE:
        if only and row[0] not in only:
            continue
        name, kind, R, G, dt, chunk_bytes, dist, seed, opts = row
        scale = getattr(args, "scale", 1.0) or 1.0
        cb = max(16, int(chunk_bytes * scale) // 16 * 16)
        out.append((name, kind, R, G, dt, cb, dist, seed, opts))
    return out


def build_suite(ccl, torch, datagen, args, with_host=False):
    import numpy as np
    items = []
    for name, kind, R, G, dt, chunk_bytes, dist, seed, opts in selected_suite(args):
        ce = chunk_bytes // ESIZE[dt]
        sched, popts = schedule_and_opts(ccl, kind, R, G, opts)
        plan = ccl.Plan(sched, ce, dt, **popts)
        st = plan.stats()
        nin, nout = plan.in_elems, plan.out_elems
        tdt = {0: torch.float32, 1: torch.int16, 2: torch.int16, 3: torch.int32}[dt]
        # draw on the host per rank (datagen recipe), copy once to HBM
        rng = np.random.default_rng(seed)
        d_in, d_out, h_in, h_out = [], [], [], []
        for r in range(R):
            a = datagen.draw(rng, dist, nin, dt)
            t = torch.from_numpy(a.view(np.int16) if dt in (1, 2) else a)
            d_in.append(t.cuda())
            d_out.append(torch.empty(nout, dtype=tdt, device="cuda"))
            if with_host:
                h_in.append(t.pin_memory())
                h_out.append(torch.empty(nout, dtype=tdt).pin_memory())
        items.append(dict(name=name, kind=kind, R=R, G=G, dt=dt, ce=ce, plan=plan, stats=st, d_in=d_in,
                          d_out=d_out, h_in=h_in, h_out=h_out, dist=dist, seed=seed, opts=opts))
    return items


def run_gpu(args):
    import torch
    import collective_communication_schedule_gb300 as ccl
    import datagen

    peak, peak_kind = peaks()
    items = build_suite(ccl, torch, datagen, args, with_host=True)
    stream = torch.cuda.current_stream()
    # warm-up
    for _ in range(args.warmup):
        for it in items:
            it["plan"].execute(it["d_in"], it["d_out"], stream)
    torch.cuda.synchronize()
    for it in items:
        it["plan"].status()

    # timed device region: events around every launch on the launching stream
    K = args.steps
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in items]
          for _ in range(K)]
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_all0.record(stream)
    for k in range(K):
        for j, it in enumerate(items):
            ev[k][j][0].record(stream)
            it["plan"].execute(it["d_in"], it["d_out"], stream)
            ev[k][j][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    for it in items:
        it["plan"].status()
    total_ms = t_all0.elapsed_time(t_all1)
    per = []
    sched_bytes = sum(it["stats"].schedule_bytes for it in items)
    by_kernel = {}   # kernel name -> [launches, ms, schedule bytes]
    for j, it in enumerate(items):
        ts = [ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(K)]
        mean_ms = sum(ts) / len(ts)
        kk = by_kernel.setdefault(kernel_name(it["stats"]), [0, 0.0, 0])
        kk[0] += K
        kk[1] += sum(ts)
        kk[2] += K * it["stats"].schedule_bytes
        st = it["stats"]
        gbs = st.schedule_bytes / (mean_ms * 1e6)
        algbw = st.data_bytes_per_rank / (mean_ms * 1e6)
        per.append({
            "name": it["name"], "ranks": it["R"], "dtype": NAMES[it["dt"]],
            "bytes_per_rank": st.data_bytes_per_rank, "mean_us": round(mean_ms * 1e3, 2),
            "median_us": round(statistics.median(ts) * 1e3, 2),
            "schedule_gbs": round(gbs, 1), "min_bytes_gbs": round(st.min_bytes / (mean_ms * 1e6), 1),
            "frac_of_peak": round(gbs / peak, 3), "min_bytes_frac": round(st.min_bytes / (mean_ms * 1e6) / peak, 3),
            "algbw_gbs": round(algbw, 1), "busbw_gbs": round(algbw * st.busbw_factor, 1),
            "frac_of_nominal_8tbs": round(gbs / 8000.0, 3),
            "threadblocks": st.nthreadblocks, "threadblocks_connection": st.nthreadblocks_connection,
            "channels": st.channels, "microbatches": st.microbatches,
            "slot_bytes": st.slot_bytes, "nthreads": st.nthreads,
        })
    # outside the timed region: threadblock idle fractions (instrumented
    # plan) and, for collectives whose buffers fit in L2, the time with L2
    # flushed before every execution (flush outside the events)
    if not args.no_extras:
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
        flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device="cuda")
        for rec, it in zip(per, items):
            sched, popts = schedule_and_opts(ccl, it["kind"], it["R"], it["G"], it["opts"])
            inst = ccl.Plan(sched, it["ce"], it["dt"], instrument=1, **popts)
            inst.execute(it["d_in"], it["d_out"], stream)
            torch.cuda.synchronize()
            inst.status()
            tl = inst.timeline()
            rec["mean_idle"], rec["max_idle"] = round(tl["mean_idle"], 3), round(tl["max_idle"], 3)
            del inst
            footprint = it["R"] * (it["plan"].in_elems + it["plan"].out_elems) * ESIZE[it["dt"]]
            if footprint < l2:
                ts = []
                for _ in range(10):
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    it["plan"].execute(it["d_in"], it["d_out"], stream)
                    b.record(stream)
                    torch.cuda.synchronize()
                    ts.append(a.elapsed_time(b))
                it["plan"].status()
                rec["l2_flushed_median_us"] = round(statistics.median(ts) * 1e3, 2)
        del flush
    step_ms = total_ms / K
    value = sched_bytes / (step_ms * 1e6)
    min_bytes = sum(it["stats"].min_bytes for it in items)
    # roofline of the dominant kernel (most device time): its algorithmic
    # bytes per launch over its mean launch duration
    dom = max(by_kernel, key=lambda n: by_kernel[n][1])
    n_dom, ms_dom, bytes_dom = by_kernel[dom]
    achieved = (bytes_dom / n_dom) / ((ms_dom / n_dom) * 1e6)
    kern_total = sum(v[1] for v in by_kernel.values())
    kernels = [{"kernel": n, "launches_per_step": v[0] // K, "share": round(v[1] / kern_total, 3),
                "achieved_gbs": round(v[2] / (v[1] * 1e6), 1)} for n, v in by_kernel.items()]

    # end to end through the C ABI with host buffers (H2D + execute + D2H per
    # collective).  The collectives of a step are independent, so they
    # rotate over a few streams (each plan always on the same one): input
    # copies of the next collectives overlap the output copies of earlier
    # ones (host<->device copies run in both directions at once).
    Ke = max(1, min(K, args.e2e_steps))
    h2d = sum(it["plan"].in_elems * ESIZE[it["dt"]] * it["R"] for it in items)
    d2h = sum(it["plan"].out_elems * ESIZE[it["dt"]] * it["R"] for it in items)
    if args.e2e_mode == "pipeline":
        # ccl_execute_host_async: every input copy on one stream, every
        # kernel on the launching stream, every output copy on a third, so
        # the copy engines of both directions stay busy across collectives
        e2e_streams = [stream, torch.cuda.Stream(), torch.cuda.Stream()]

        def e2e_pass():
            for it in items:
                it["plan"].execute_host_async(it["h_in"], it["h_out"], it["d_in"], it["d_out"], e2e_streams[1],
                                              stream, e2e_streams[2])
    else:
        e2e_streams = [stream] + [torch.cuda.Stream() for _ in range(max(1, args.e2e_streams) - 1)]

        def e2e_pass():
            for j, it in enumerate(items):
                s = e2e_streams[j % len(e2e_streams)]
                it["plan"].execute_host(it["h_in"], it["h_out"], it["d_in"], it["d_out"], s)

    e2e_pass()   # warm
    torch.cuda.synchronize()
    # the host link just before and just after the end-to-end steps (the
    # host side of a shared machine changes from minute to minute)
    link_before = host_link(torch, items, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in e2e_streams[1:]:
        s.wait_event(e0)
    for _ in range(Ke):
        e2e_pass()
    for s in e2e_streams[1:]:
        joined = torch.cuda.Event()
        joined.record(s)
        stream.wait_event(joined)
    e1.record(stream)
    torch.cuda.synchronize()
    for it in items:
        it["plan"].status()
    e2e_ms = e0.elapsed_time(e1) / Ke
    link = host_link(torch, items, stream)

    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": 1,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32/bf16/f16 (per collective)",
        "data": "synthetic (numpy PCG64 seeds 0-4)",
        "config": {"workload": "collective suite: hier AR 16x64MiB f32 + two-phase A2A 32x32MiB f16 + ring AR "
                               "8x256MiB bf16 & f32 (24 ch) + AllToNext 24x128MiB f32 + AG/RS 8x3MiB bf16 + "
                               "ring AR 8x1MiB f32",
                   "parallelism": "replicas only (R virtual ranks per GPU, no cross-GPU exchange)", "l2": "step working set ~19 GiB > L2 (no flush)",
                   "schedule_bytes_per_step": sched_bytes,
                   "collective_min_bytes_per_step": min_bytes,
                   **({"subset": args.only, "scale": args.scale} if (args.only or args.scale != 1.0) else {})},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "kernels": kernels,
                     "traffic": recorded_traffic(dom) if not (args.only or args.scale != 1.0) else None,
                     "traffic_unit": "bytes per launch (ncu dram read+write, profiles/roofline_traffic.txt)",
                     "traffic_basis": "full-size capture of the kernel's launches in one step, one pass each "
                                      "(pass count checked on half-size captures first; scaled half-size captures "
                                      "understate the AllReduce rows, whose FIFOs keep their size)",
                     "algorithmic_bytes_per_launch": bytes_dom // n_dom,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": {"value": round(sched_bytes / (e2e_ms * 1e6), 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3), "steps": Ke,
                "mode": args.e2e_mode, "streams": len(e2e_streams),
                # the same host buffers copied alone (no kernels, best of two
                # each), just after and just before the end-to-end steps: a
                # probe's floor_ms is the slowest of one way in, one way out and
                # both at once; the floor reported is the lower of the two (the
                # link at its best), a bound ms_per_step cannot beat
                "host_link_gbs": link,
                "host_link_before_gbs": link_before,
                "floor_ms_from_link": min(link.get("floor_ms", 0), link_before.get("floor_ms", 0))
                if link.get("both_each_way") else None},
        # bytes every collective must move at least (each input read once,
        # each output written once) per second of the step: unlike `value`,
        # independent of the schedule's transport and fusion choices
        "collective_min_bytes_gbs": round(min_bytes / (step_ms * 1e6), 1),
        "gpu_launches": K * len(items),
        "clocks": clk,
        "per_collective": per,
    }
    if not args.no_sweep:
        out["sweep"] = run_sweep(ccl, torch, datagen, args, peak)
    if not args.no_codegen_rows and not (args.only or args.scale != 1.0):
        # the latency-bound rows, whose steps the interpreter's record and
        # table reads lengthen the most, run both ways (outside the timed
        # region); `python bench.py --codegen` adds the large rows
        out["codegen"] = run_codegen(args, rows=["ar_1m", "ag_3m", "rs_3m"], stream=stream)
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(items, args.cpu_seconds)
    return out


def host_link(torch, items, stream):
    """Pinned host <-> device copy rates of the step's own buffers, with no
    kernel: every input to the device alone, every output to the host alone,
    and both directions at once on two streams (GB/s each way)."""
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    h2d = sum(t.numel() * t.element_size() for it in items for t in it["h_in"])
    d2h = sum(t.numel() * t.element_size() for it in items for t in it["d_out"])
    if not h2d or not d2h:
        return {}

    def timed(fn):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_event(a)
        down.wait_event(a)
        fn()
        for s in (up, down):
            e = torch.cuda.Event()
            e.record(s)
            stream.wait_event(e)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def copy_in():
        with torch.cuda.stream(up):
            for it in items:
                for d, h in zip(it["d_in"], it["h_in"]):
                    d.copy_(h, non_blocking=True)

    def copy_out():
        with torch.cuda.stream(down):
            for it in items:
                for h, d in zip(it["h_out"], it["d_out"]):
                    h.copy_(d, non_blocking=True)

    def both():
        copy_in()
        copy_out()
    timed(both)   # first touch of the copy paths, not counted
    # best of two of each (a busy host slows single copies at random)
    t_in = min(timed(copy_in), timed(copy_in))
    t_out = min(timed(copy_out), timed(copy_out))
    t_both = min(timed(both), timed(both))
    # the end-to-end step cannot be shorter than either direction alone or
    # than both at once
    return {"h2d": round(h2d / (t_in * 1e6), 1), "d2h": round(d2h / (t_out * 1e6), 1),
            "both_each_way": round(max(h2d, d2h) / (t_both * 1e6), 1),
            "floor_ms": round(max(t_in, t_out, t_both), 3)}


# The message-size sweep: ring AllGather and ReduceScatter, 8 ranks, bf16,
# per-rank buffer (AllGather output, ReduceScatter input) 32 KiB .. 2 MiB and
# 3 MiB, channels 1..4, normal(0,1) seed 1, each size planned from the
# collective's tuned table.  The small ring AllReduce's int32
# copy: 8 x 1 MiB, integers in [-1000, 1000], seed 0.
SWEEP_KIB = [32, 64, 128, 256, 512, 1024, 2048, 3072]
TABLE_DIR = os.path.join(ROOT, "collective_communication_schedule_gb300", "tables")
# the AllGather runs with its copy receives unchained (each hop a direct
# copy, chains folded two hops per step, as the suite's 3 MiB row); the
# ReduceScatter has no copy hops and runs fully fused
SWEEP_NOCHAIN = {1: True, 2: False}


def sweep_schedule(ccl, kind, R):
    return ccl.Schedule.builtin(kind, R, 0, ccl.FLAG_NOCHAIN_COPIES if SWEEP_NOCHAIN[kind] else 0)


def tuned_table(ccl, torch, datagen, kind, args):
    """The per-size tuning table of a sweep collective: the committed file
    when there is one (and --retune is not given), else tuned now (outside
    any timed region) and, with --table-out DIR, written there."""
    name = {1: "ring_allgather", 2: "ring_reducescatter"}[kind]
    path = os.path.join(TABLE_DIR, f"{name}_r8_bf16.json")
    if os.path.exists(path) and not args.retune:
        rows, _ = ccl.read_tune_table(path)
        return rows, os.path.relpath(path, ROOT)
    R = 8
    sizes = [kib * 1024 // 2 // R for kib in SWEEP_KIB]
    s = sweep_schedule(ccl, kind, R)
    nin = max(sizes) * (1 if kind == 1 else R)
    ins = [torch.from_numpy(a.view("int16")).cuda() for a in datagen.rank_inputs(1, "normal", R, nin, 1)]
    outs = [torch.empty(max(sizes) * (R if kind == 1 else 1), dtype=torch.int16, device="cuda") for _ in range(R)]
    rows = ccl.tune_table(s, 1, sizes, ins, outs, max_rounds=2, reps=5, max_channels=4)
    out_dir = args.table_out
    if out_dir:
        os.makedirs(out_dir, exist_ok=True)
        unchained = ", copy receives unchained" if SWEEP_NOCHAIN[kind] else ""
        ccl.write_tune_table(rows, 1, os.path.join(out_dir, os.path.basename(path)),
                             note=f"{name} R=8 bf16{unchained}, channels <= 4, tuned on {torch.cuda.get_device_name()}")
    return rows, "tuned in this run"


def run_sweep(ccl, torch, datagen, args, peak):
    """The message-size sweep (every size x channels 1-4, AllGather and
    ReduceScatter, 8 ranks bf16) and the 1 MiB ring AllReduce's int32 copy,
    each with its tuned
    configuration; median of 20 executions with warm L2 and of 10 with L2
    flushed before each (flush outside the events), threadblock idle
    fractions from one instrumented execution.  Measured after the timed
    region of the step."""
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device="cuda")
    R = 8

    def measure(sched, ce, dt, opts, d_in, d_out):
        plan = ccl.Plan(sched, ce, dt, opts=opts)
        st = plan.stats()
        warm = _time_plan(torch, plan, d_in, d_out, stream, reps=20, warm=3)
        ts = []
        for _ in range(10):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.execute(d_in, d_out, stream)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        plan.status()
        cold = statistics.median(ts)
        del plan
        o2 = ccl.PlanOpts.from_buffer_copy(opts)
        o2.instrument = 1
        inst = ccl.Plan(sched, ce, dt, opts=o2)
        inst.execute(d_in, d_out, stream)
        torch.cuda.synchronize()
        inst.status()
        tl = inst.timeline()
        del inst
        algbw = st.data_bytes_per_rank / (cold * 1e6)
        return {"us": round(cold * 1e3, 2), "us_warm_l2": round(warm * 1e3, 2),
                "schedule_gbs": round(st.schedule_bytes / (cold * 1e6), 1),
                "frac_of_peak": round(st.schedule_bytes / (cold * 1e6) / peak, 4),
                "algbw_gbs": round(algbw, 2), "busbw_gbs": round(algbw * st.busbw_factor, 2),
                "threadblocks": st.nthreadblocks, "threadblocks_connection": st.nthreadblocks_connection,
                "mean_idle": round(tl["mean_idle"], 3), "max_idle": round(tl["max_idle"], 3),
                "engine": st.engine, "nthreads": st.nthreads, "slot_bytes": st.slot_bytes,
                "link_mode": opts.link_mode, "tb_alloc": opts.tb_alloc}

    out = {"note": "per-rank buffer S: AllGather output, ReduceScatter input; us = median with L2 flushed", "rows": []}
    for kind, kname in ((1, "allgather"), (2, "reducescatter")):
        rows, src = tuned_table(ccl, torch, datagen, kind, args)
        out[f"{kname}_table"] = src
        sched = sweep_schedule(ccl, kind, R)
        for kib in SWEEP_KIB:
            ce = kib * 1024 // 2 // R
            nin = ce * (1 if kind == 1 else R)
            nout = ce * (R if kind == 1 else 1)
            d_in = [torch.from_numpy(a.view("int16")).cuda() for a in datagen.rank_inputs(1, "normal", R, nin, 1)]
            d_out = [torch.empty(nout, dtype=torch.int16, device="cuda") for _ in range(R)]
            base = ccl.lookup_tune_table(rows, ce)
            for ch in (1, 2, 3, 4):
                o = ccl.PlanOpts.from_buffer_copy(base)
                o.channels = ch
                rec = {"collective": kname, "dtype": "bf16", "per_rank_kib": kib, "channels": ch}
                try:
                    rec.update(measure(sched, ce, 1, o, d_in, d_out))
                except ccl.CclError as e:
                    rec["error"] = str(e)[:100]
                out["rows"].append(rec)
    # the small ring AllReduce's int32 copy: the f32 row's options
    row = [r for r in SUITE if r[0] == "ar_1m"][0]
    sched, popts = schedule_and_opts(ccl, 0, R, 0, row[8])
    ce = 1 * MiB // 4 // R
    d_in = [torch.from_numpy(a).cuda() for a in datagen.rank_inputs(0, "int", R, R * ce, 3)]
    d_out = [torch.empty(R * ce, dtype=torch.int32, device="cuda") for _ in range(R)]
    o = ccl.default_opts()
    for k, v in popts.items():
        setattr(o, k, v)
    rec = {"collective": "allreduce", "dtype": "i32", "per_rank_kib": 1024, "channels": o.channels}
    rec.update(measure(sched, ce, 3, o, d_in, d_out))
    out["rows"].append(rec)
    del flush
    return out


ORACLE_PROGRAMS = {0: ("ring_allreduce", lambda R, G: (R,)), 1: ("ring_allgather", lambda R, G: (R,)),
                   2: ("ring_reducescatter", lambda R, G: (R,)), 3: ("hier_allreduce", lambda R, G: (G, R // G)),
                   4: ("alltoall_two_phase", lambda R, G: (G, R // G)), 5: ("alltonext", lambda R, G: (G, R // G))}
# the plan option defaults the suite rows rely on (ccl_plan_opts_default):
# direct transport unless a row asks for FIFOs, receives and copy chains
# folded unless a row says otherwise (the rows with reduction chains fold
# them too: fold 7)
DEFAULT_LINK_MODE = 1
DEFAULT_FOLD = 3


def oracle_program(kind, R, G):
    """The oracle's own program of a built-in collective: (ops, nchunks)."""
    from oracle import schedules as OS
    nm, a = ORACLE_PROGRAMS[kind]
    return OS.BUILTINS[nm](*a(R, G))


def oracle_bytes(kind, R, G, dt, ce, opts):
    """Schedule bytes and collective-minimum bytes of one execution of a
    suite row, counted by the oracle from its own program (fused-instruction
    semantics, the row's fusion mode and transport)."""
    from oracle import bytes as OB
    ops, nch = oracle_program(kind, R, G)
    fuse = opts.get("fuse", True)
    mode = "nochain" if fuse == "nochain" else ("full" if fuse else "none")
    direct = opts.get("link_mode", DEFAULT_LINK_MODE) == 1
    fold = int(opts.get("fold", DEFAULT_FOLD))
    return (OB.schedule_bytes(ops, R, nch, ce, dt, mode, direct, fold), OB.min_bytes(ops, R, nch, ce, dt))


def _oracle_inputs(it):
    """Host copies of the inputs: the GPU arm's pinned buffers, or a fresh
    draw with the same recipe (reference arm)."""
    import numpy as np
    import datagen
    if it.get("h_in"):
        return [t.numpy().view(np.uint16) if it["dt"] in (1, 2) else t.numpy() for t in it["h_in"]]
    rng = np.random.default_rng(it["seed"])
    nin = it["nin"]
    return [datagen.draw(rng, it["dist"], nin, it["dt"]) for _ in range(it["R"])]


def oracle_prepare(items):
    """The oracle's programs and host inputs of every collective (drawn once)."""
    import oracle
    oracle.build()
    prepared = []
    for it in items:
        ops, nch = oracle_program(it["kind"], it["R"], it["G"])
        prepared.append((it, ops, nch, _oracle_inputs(it)))
    return prepared


def cpu_baseline(items, budget_s, divisor=None, prepared=None):
    """The oracle (C, one thread) on a bounded sample: every collective of the
    suite on the same inputs restricted to 1/divisor of the in-chunk offsets
    (the oracle maps chunk to chunk offset by offset, so a column sample is
    an exact part of the full result).  divisor=None calibrates it so that the
    three timed repetitions take about ``budget_s`` seconds.  ``prepared``:
    the result of oracle_prepare(items), when the caller keeps it."""
    import numpy as np
    import oracle
    if prepared is None:
        prepared = oracle_prepare(items)

    def one_pass(div, reps):
        t_total, bytes_total, sampled = 0.0, 0.0, []
        for it, ops, nch, ins in prepared:
            ce = it["ce"]
            cols = max(1, ce // div)
            offs = (np.arange(cols, dtype=np.int64) * (ce // cols)).astype(np.int64)
            cols_in = [np.ascontiguousarray(x.reshape(nch[0], ce)[:, offs]).reshape(-1) for x in ins]
            ts = []
            for _ in range(reps):
                t0 = time.perf_counter()
                oracle.run(ops, it["R"], nch, cols, it["dt"], cols_in)
                ts.append(time.perf_counter() - t0)
            t_total += statistics.median(ts)
            # the oracle's own count of the row's schedule bytes on the sample
            bytes_total += oracle_bytes(it["kind"], it["R"], it["G"], it["dt"], cols, it["opts"])[0]
            sampled.append(f"{it['name']}:{cols}/{ce}")
        return t_total, bytes_total, sampled

    if divisor is None:
        t, _, _ = one_pass(4096, 1)
        want = 4096.0 * 3.0 * t / budget_s      # divisor whose 3 repetitions take ~budget_s
        divisor = 1
        while divisor < want and divisor < 4096:
            divisor *= 2
    t_total, bytes_total, sampled = one_pass(divisor, 3)
    return {"value": round(bytes_total / t_total / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "host_cpus": os.cpu_count(),
            "sample": f"every collective of the step on 1/{divisor} of the in-chunk offsets, median of 3 ("
                      + ", ".join(sampled) + ")",
            "seconds": round(t_total, 3)}


def run_reference(args):
    """The oracle as the reference arm: same metric on bounded samples."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    # nothing of the product runs here: programs, inputs and byte counts
    # all come from the oracle and datagen
    items = []
    for name, kind, R, G, dt, chunk_bytes, dist, seed, opts in selected_suite(args):
        ce = chunk_bytes // ESIZE[dt]
        _, nch = oracle_program(kind, R, G)
        items.append(dict(name=name, kind=kind, R=R, G=G, dt=dt, ce=ce, dist=dist, seed=seed, nin=nch[0] * ce,
                          opts=opts))
    # inputs drawn once; every warm-up and timed step runs the oracle on the
    # same bounded sample
    prepared = oracle_prepare(items)
    cb = None
    for _ in range(args.warmup + args.steps):
        cb = cpu_baseline(items, args.cpu_seconds, divisor=1024, prepared=prepared)
    return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32/bf16/f16 (per collective)", "data": "synthetic (numpy PCG64 seeds 0-4)",
            "config": {"workload": "collective suite (same as the GPU arm), each step a 1/1024 sample of in-chunk offsets"},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _time_plan(torch, plan, d_in, d_out, stream, reps=5, warm=2, side=None):
    """Median device time (ms) of `reps` executions after `warm`; `side`, when
    given, is called before each execution to queue concurrent work."""
    ts = []
    for k in range(warm + reps):
        if side is not None:
            side()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plan.execute(d_in, d_out, stream)
        b.record(stream)
        torch.cuda.synchronize()
        if k >= warm:
            ts.append(a.elapsed_time(b))
    plan.status()
    return statistics.median(ts)


def run_ablation(args):
    """Scheduler (RR / HPDS) x threadblock allocation (connection / packed)
    on the large collectives: device time, threadblocks, sub-pipelines and
    threadblock idle fractions (one JSON line per configuration)."""
    import torch
    import collective_communication_schedule_gb300 as ccl
    import datagen
    names = args.only.split(",") if args.only else ["hier_ar", "a2a", "a2n", "ring_f32"]
    args.only = ",".join(names)
    items = build_suite(ccl, torch, datagen, args)
    stream = torch.cuda.current_stream()
    for it, row in zip(items, selected_suite(args)):
        base = dict(row[8])
        del it["plan"]
        for sched in (ccl.SCHED_RR, ccl.SCHED_HPDS):
            for alloc in (ccl.TB_CONNECTION, ccl.TB_PACKED):
                opts = dict(base, scheduler=sched, tb_alloc=alloc)
                sch, popts = schedule_and_opts(ccl, it["kind"], it["R"], it["G"], opts)
                rec = {"ablation": it["name"], "scheduler": ["rr", "hpds"][sched],
                       "tb_alloc": ["connection", "packed"][alloc]}
                try:
                    plan = ccl.Plan(sch, it["ce"], it["dt"], **popts)
                    ms = _time_plan(torch, plan, it["d_in"], it["d_out"], stream)
                    st = plan.stats()
                    del plan
                    inst = ccl.Plan(sch, it["ce"], it["dt"], instrument=1, **popts)
                    _time_plan(torch, inst, it["d_in"], it["d_out"], stream, reps=1, warm=1)
                    tl = inst.timeline()
                    del inst
                    rec.update(us=round(ms * 1e3, 1), schedule_gbs=round(st.schedule_bytes / (ms * 1e6), 1),
                               threadblocks=st.nthreadblocks, threadblocks_connection=st.nthreadblocks_connection,
                               subpipelines=st.nsubpipelines, mean_idle=round(tl["mean_idle"], 3),
                               max_idle=round(tl["max_idle"], 3))
                except ccl.CclError as e:
                    rec["error"] = str(e)[:120]
                torch.cuda.empty_cache()
                print(json.dumps(rec), flush=True)


def run_interference(args):
    """Interference-aware tuning: tune one collective in isolation and again
    while a bf16 GEMM runs on a concurrent stream; time both choices under
    the GEMM (AutoCCL report: interference of concurrent computation).
    Also times an exhaustive grid in isolation to place the isolated tuner's
    choice.  One JSON line."""
    import torch
    import collective_communication_schedule_gb300 as ccl
    import datagen
    name = args.only or "ring_f32"
    args.only = name
    it = build_suite(ccl, torch, datagen, args)[0]
    row = selected_suite(args)[0]
    del it["plan"]
    stream = torch.cuda.current_stream()
    side_stream = torch.cuda.Stream()
    n = 8192
    ga = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    gb = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    gc = torch.empty(n, n, device="cuda", dtype=torch.bfloat16)

    def gemm():
        with torch.cuda.stream(side_stream):
            for _ in range(4):
                torch.matmul(ga, gb, out=gc)

    base = dict(row[8])
    sch, popts = schedule_and_opts(ccl, it["kind"], it["R"], it["G"], base)
    start = ccl.default_opts()
    for k, v in popts.items():
        setattr(start, k, v)

    def make_probe(with_gemm):
        def probe(o):
            try:
                plan = ccl.Plan(sch, it["ce"], it["dt"], opts=o)
            except ccl.CclError:
                return 0.0
            try:
                ms = _time_plan(torch, plan, it["d_in"], it["d_out"], stream, reps=3, warm=1,
                                side=gemm if with_gemm else None)
                return plan.stats().schedule_bytes / (ms * 1e6)
            except ccl.CclError:
                return 0.0
            finally:
                del plan
                torch.cuda.synchronize()
        return probe

    iso_best, iso_bw, iso_n = ccl.tune_search(make_probe(False), start=start)
    int_best, int_bw, int_n = ccl.tune_search(make_probe(True), start=start)

    def t_us(o, with_gemm):
        plan = ccl.Plan(sch, it["ce"], it["dt"], opts=o)
        ms = _time_plan(torch, plan, it["d_in"], it["d_out"], stream, reps=7, warm=2,
                        side=gemm if with_gemm else None)
        del plan
        return round(ms * 1e3, 1)

    def cfg(o):
        return {"channels": o.channels, "nthreads": o.nthreads, "slot_bytes": o.slot_bytes,
                "tb_alloc": o.tb_alloc, "protocol": o.protocol}

    # exhaustive grid in isolation (the tuner's resource grid, both policies,
    # flag protocol), best point
    grid_best, grid_us, grid_n = None, None, 0
    for alloc in (ccl.TB_CONNECTION, ccl.TB_PACKED):
        for ch in (1, 2, 4, 8, 12, 16, 24, 32, 48):
            for nt in (128, 256, 512, 1024):
                for sl in (16384, 32768, 65536, 131072, 262144, 524288, 1048576):
                    o = ccl.default_opts()
                    for k, v in popts.items():
                        setattr(o, k, v)
                    o.tb_alloc, o.channels, o.nthreads, o.slot_bytes = alloc, ch, nt, sl
                    bw = make_probe(False)(o)
                    grid_n += 1
                    if bw > 0 and (grid_us is None or it["stats"].schedule_bytes / (bw * 1e3) < grid_us):
                        grid_us = it["stats"].schedule_bytes / (bw * 1e3)
                        grid_best = cfg(o)
    out = {"interference": name, "gemm": f"bf16 {n}x{n}x{n}, 4 per execution on a concurrent stream",
           "isolated_tuned": cfg(iso_best), "interference_tuned": cfg(int_best),
           "probes": {"isolated": iso_n, "interference": int_n, "grid": grid_n},
           "us": {"isolated_cfg_alone": t_us(iso_best, False), "isolated_cfg_with_gemm": t_us(iso_best, True),
                  "interference_cfg_with_gemm": t_us(int_best, True), "default_cfg_alone": t_us(start, False),
                  "grid_best_alone": round(grid_us, 1) if grid_us else None},
           "grid_best": grid_best}
    out["gain_under_interference"] = round(out["us"]["isolated_cfg_with_gemm"] / out["us"]["interference_cfg_with_gemm"], 3)
    print(json.dumps(out))


def run_alltoallv(args):
    """Second workload: uneven AllToAll of a mixture-of-experts layer.  32
    ranks (one expert each), 4096 tokens per rank of 4096 bf16 values (one
    8 KiB chunk per token), Zipf(1.2) expert popularity (datagen recipe,
    seed 3).  One JSON line per plan configuration."""
    import numpy as np
    import torch
    import collective_communication_schedule_gb300 as ccl
    import datagen
    R, tokens, hidden = 32, int(4096 * args.scale), 4096
    counts = datagen.alltoallv_counts(3, R, tokens)
    sch = ccl.Schedule.alltoallv(counts)
    nin, nout = sch.info().nchunks[0] * hidden, sch.info().nchunks[1] * hidden
    rng = np.random.default_rng(3)
    d_in = [torch.from_numpy(datagen.draw(rng, "normal", nin, ccl.BF16).view(np.int16)).cuda() for _ in range(R)]
    d_out = [torch.empty(nout, dtype=torch.int16, device="cuda") for _ in range(R)]
    stream = torch.cuda.current_stream()
    peak, _ = peaks()
    # channels in proportion to a pair's size (channel_scaling): the hot
    # expert's pairs get many threadblocks, the small pairs one
    # balanced allocation: a rank's direct copies binned into a few large
    # threadblocks instead of one small threadblock per pair
    configs = [dict(link_mode=1, tb_alloc=1, channels=4, bulk=1)] + \
              [dict(link_mode=1, tb_alloc=2, channels=c, channel_scaling=0, tb_budget=b)
               for c in (2, 4, 8) for b in (256, 512)]
    for o in configs:
        rec = {"workload": "alltoallv", "ranks": R, "tokens_per_rank": tokens, "chunk_bytes": hidden * 2,
               "max_in_chunks": int(counts.sum(1).max()), "max_out_chunks": int(counts.sum(0).max()), "opts": o}
        try:
            plan = ccl.Plan(sch, hidden, ccl.BF16, **o)
            ms = _time_plan(torch, plan, d_in, d_out, stream, reps=args.steps, warm=args.warmup)
            st = plan.stats()
            rec.update(us=round(ms * 1e3, 1), schedule_gbs=round(st.schedule_bytes / (ms * 1e6), 1),
                       frac_of_peak=round(st.schedule_bytes / (ms * 1e6) / peak, 3),
                       min_bytes_gbs=round(st.min_bytes / (ms * 1e6), 1), threadblocks=st.nthreadblocks,
                       nthreads=st.nthreads)
            del plan
        except ccl.CclError as e:
            rec["error"] = str(e)[:120]
        print(json.dumps(rec), flush=True)


def run_codegen(args, rows=None, stream=None):
    """Generated against interpreted kernels (ReSCCL report, §II.2: a kernel
    per schedule instead of an interpreter): each suite row's plan run both
    ways on the same inputs, median of --steps executions after --warmup,
    with the generated kernel's generation + compile time.  Returns one
    record per row."""
    import torch
    import collective_communication_schedule_gb300 as ccl
    import datagen
    names = rows or (args.only.split(",") if args.only else ["ar_1m", "ag_3m", "rs_3m", "hier_ar"])
    saved = args.only
    args.only = ",".join(names)
    items = build_suite(ccl, torch, datagen, args)
    args.only = saved
    stream = stream or torch.cuda.current_stream()
    out = []
    for it in items:
        rec = {"row": it["name"], "engine": it["stats"].engine}
        ms_i = _time_plan(torch, it["plan"], it["d_in"], it["d_out"], stream, reps=max(5, args.steps),
                          warm=max(3, args.warmup))
        rec["interpreted_us"] = round(ms_i * 1e3, 2)
        sched, popts = schedule_and_opts(ccl, it["kind"], it["R"], it["G"], it["opts"])
        try:
            gen = ccl.Plan(sched, it["ce"], it["dt"], codegen=1, **popts)
            st = gen.stats()
            ms_g = _time_plan(torch, gen, it["d_in"], it["d_out"], stream, reps=max(5, args.steps),
                              warm=max(3, args.warmup))
            rec.update(generated_us=round(ms_g * 1e3, 2), speedup=round(ms_i / ms_g, 3),
                       codegen_ms=round(st.codegen_ms, 1), threadblocks=st.nthreadblocks, steps=st.nsteps)
            del gen
        except ccl.CclError as e:
            rec["error"] = str(e)[:160]
        out.append(rec)
        del it["plan"]
        torch.cuda.empty_cache()
    return out


def hier_allgather_program(G, ng):
    """A user chunk program for the hierarchical AllGather of the HetCCL
    summary ("hierarchical algorithm design and pipelined execution"): an
    in-group step, a cross-group step and a final in-group step, the
    cross-group transfers overlapping the in-group work.  Groups of G ranks
    stand for the clusters.  Every rank places its block and copies it, from
    its input, to the rank with its local index in every other group; then
    ring rounds inside every group carry each block on from the rank it
    entered the group at.  One chunk in per rank, R = G * ng chunks out.
    Rows: (op, src_rank, src_buf, src_off, dst_rank, dst_buf, dst_off, count)."""
    R = G * ng
    ops = []
    for r in range(R):
        ops.append((0, r, 0, 0, r, 1, r, 1))
        for h in range(ng):
            if h != r // G:
                ops.append((0, r, 0, 0, h * G + r % G, 1, r, 1))
    for k in range(G - 1):           # ring round k inside every group
        for h in range(ng):
            for blk in range(R):     # entered group h at local index blk % G
                a = h * G + (blk % G + k) % G
                b = h * G + (blk % G + k + 1) % G
                ops.append((0, a, 1, blk, b, 1, blk, 1))
    return ops, (1, R, 0)


def run_hier_allgather(args):
    """NEXT workload: hierarchical AllGather, 16 ranks as 2 groups x 8, bf16,
    4 MiB in and 64 MiB out per rank (normal(0,1), seed 5), against the flat
    ring AllGather on the same ranks and bytes.  One JSON line per plan."""
    import numpy as np
    import torch
    import collective_communication_schedule_gb300 as ccl
    import datagen
    G, ng = 8, 2
    R = G * ng
    ce = int(2 * MiB * args.scale)            # bf16 elements per chunk (4 MiB)
    rng = np.random.default_rng(5)
    d_in = [torch.from_numpy(datagen.draw(rng, "normal", ce, ccl.BF16).view(np.int16)).cuda() for _ in range(R)]
    d_out = [torch.empty(R * ce, dtype=torch.int16, device="cuda") for _ in range(R)]
    stream = torch.cuda.current_stream()
    peak, _ = peaks()
    ops, nch = hier_allgather_program(G, ng)
    hier = ccl.Schedule.compile(ops, R, nch, fuse=False)
    flat = ccl.Schedule.builtin(ccl.RING_ALLGATHER, R, 0, ccl.FLAG_NOFUSE)
    flat_fused = ccl.Schedule.builtin(ccl.RING_ALLGATHER, R)
    direct = dict(channels=8, link_mode=1)
    balanced = dict(channels=8, link_mode=1, tb_alloc=2, tb_budget=304)
    # unfused with direct copies: every hop one copy into the next rank's
    # output (the hierarchical program fused through FIFOs needs more slots
    # and threadblocks than fit); the flat ring also fused through FIFOs
    runs = [("hierarchical", False, hier, direct), ("hierarchical", False, hier, balanced),
            ("flat ring", False, flat, direct), ("flat ring", False, flat, balanced),
            ("flat ring", True, flat_fused, dict(channels=8))]
    for name, fuse, sched, o in runs:
        rec = {"workload": "allgather", "algorithm": name, "ranks": R, "groups": ng,
               "out_bytes_per_rank": R * ce * 2, "fuse": fuse, "opts": o}
        try:
            plan = ccl.Plan(sched, ce, ccl.BF16, **o)
            ms = _time_plan(torch, plan, d_in, d_out, stream, reps=args.steps, warm=args.warmup)
            st = plan.stats()
            rec.update(us=round(ms * 1e3, 1), schedule_gbs=round(st.schedule_bytes / (ms * 1e6), 1),
                       frac_of_peak=round(st.schedule_bytes / (ms * 1e6) / peak, 3),
                       algbw_gbs=round(R * ce * 2 / (ms * 1e6), 1),   # output bytes per rank
                       min_bytes_gbs=round(st.min_bytes / (ms * 1e6), 1), threadblocks=st.nthreadblocks)
            del plan
        except ccl.CclError as e:
            rec["error"] = str(e)[:120]
        print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--e2e-mode", default="pipeline", choices=["pipeline", "streams"],
                    help="pipeline: ccl_execute_host_async over copy-in / compute / copy-out streams; "
                         "streams: ccl_execute_host rotating over --e2e-streams")
    ap.add_argument("--e2e-streams", type=int, default=2,
                    help="streams the end-to-end leg rotates over (2 measured best: 477 GB/s vs 389 with 4)")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip idle fractions and L2-flushed timings")
    ap.add_argument("--no-sweep", action="store_true", help="skip the AllGather / ReduceScatter size sweep")
    ap.add_argument("--retune", action="store_true", help="tune the sweep's tables now instead of reading them")
    ap.add_argument("--table-out", default="", help="directory to write tables tuned by --retune to")
    ap.add_argument("--only", default="", help="comma-separated subset of the suite (profiling)")
    ap.add_argument("--scale", type=float, default=1.0, help="chunk size factor (profiling)")
    ap.add_argument("--ablation", action="store_true", help="scheduler x threadblock allocation table")
    ap.add_argument("--interference", action="store_true",
                    help="tune one collective (--only, default ring_f32) alone and beside a bf16 GEMM")
    ap.add_argument("--alltoallv", action="store_true", help="second workload: uneven (MoE) AllToAll")
    ap.add_argument("--hier-allgather", action="store_true",
                    help="hierarchical AllGather (in-group, cross-group, in-group) against the flat ring")
    ap.add_argument("--codegen", action="store_true",
                    help="generated against interpreted kernels for suite rows (--only, default ar_1m, ag_3m, "
                         "rs_3m, hier_ar)")
    ap.add_argument("--no-codegen-rows", action="store_true",
                    help="leave the generated-kernel comparison of the small rows out of the main line")
    args = ap.parse_args()
    if args.ablation or args.interference or args.alltoallv or args.hier_allgather or args.codegen:
        import torch
        torch.cuda.set_device(0)
        if args.codegen:
            for rec in run_codegen(args):
                print(json.dumps(rec), flush=True)
        elif args.ablation:
            run_ablation(args)
        elif args.interference:
            run_interference(args)
        elif args.hier_allgather:
            run_hier_allgather(args)
        else:
            run_alltoallv(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args)
        if out is not None:
            print(json.dumps(out))
        return
    if world > 1:
        # replicas only: every rank runs the same single-GPU suite on its own GPU
        import torch
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        res = combine_replicas(run_gpu(args), world, device="cuda")
        if rank == 0:
            print(json.dumps(res))
        dist.destroy_process_group()
        return
    import torch
    torch.cuda.set_device(0)
    print(json.dumps(run_gpu(args)))


if __name__ == "__main__":
    main()
