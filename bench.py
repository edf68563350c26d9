#!/usr/bin/env python3
"""Benchmark of the ONNX broadcast binary elementwise engine on GB300.

Metric: effective HBM GB/s = algorithmic bytes (A, B and out, each counted
once) / time.  The headline workload is the contiguous fp32 pair: Mul and Div
of two [2^28] tensors (A, B ~ N(0,1); Div's B = |N(0,1)| + 0.5); one step is
one plan lookup (cache hit) plus one Mul launch plus one Div launch, 6 GiB of
algorithmic traffic.  Inputs (3 GiB) are larger than L2, so no flush is
needed between steps.

Also reported: the dominant kernel's roofline (per-launch CUDA events on the
launching stream), an end-to-end number through ebin_execute_mapped (pinned
host buffers read and written in place by the kernel inside the timed region;
the copy pipeline of ebin_execute_host beside it), the oracle timed on a bounded
sample on the host, SM clocks sampled during the timed region, and a table of
every workload (one line per operator/family) timed with rotating buffers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica ("replicas
only": the engine has no exchange step); value sums all ranks' bytes over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s per op/family and % of GB300 8 TB/s roofline"
UNIT = "GB/s"
HBM_NOMINAL_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
HEADLINE = ("mul_f32_contiguous", "div_f32_contiguous")
WORKLOAD = "Mul and Div fp32 contiguous, A and B [268435456] (2^28), out [2^28]"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-families", action="store_true", help="skip the per-workload table")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--only", default=None,
                    help="time one workload case alone (for profiling), e.g. mul_f32_contiguous")
    ap.add_argument("--scale-log2", type=int, default=0,
                    help="with --only: shrink the 1-D workloads by 2^S")
    ap.add_argument("--cases", default=None,
                    help="time these workloads (comma-separated names) with the per-workload "
                         "table's method (rotating buffers, back-to-back launches) and exit")
    return ap.parse_args()


# ----------------------------------------------------------------- distributed plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(bytes_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_per_rank * world / max_seconds / 1e9


# ----------------------------------------------------------------- measurement helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel_tag: str):
    """dram read+write bytes per launch recorded in profiles/ for this kernel, if any."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                if line.startswith("traffic_bytes_per_launch[%s]:" % kernel_tag):
                    try:
                        return int(line.split(":", 1)[1].strip())
                    except ValueError:
                        return None
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in a thread."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.window = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        t0, t1 = self.window or (0, time.time())
        inside = [s for t, s in self.samples if t0 - 0.25 <= t <= t1 + 0.25 and len(s) >= 8]
        if not inside:
            inside = [s for _, s in self.samples if len(s) >= 8][-3:]
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in inside:
            try:
                sm.append(float(s[0]))
                smax.append(float(s[1]))
            except ValueError:
                continue
            for name, v in zip(names, s[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- our engine

def upload(arr):
    import numpy as np
    import torch
    flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
    return torch.from_numpy(flat).to("cuda", non_blocking=False)


def _case_plan(eb, c):
    """(descriptor, plan, host inputs) of a workload case of two or three inputs."""
    desc = eb.descriptor(c.op, c.dtype, **c.attrs)
    if c.make_c is not None:
        plan = eb.Plan3(desc, c.shape_a, c.shape_b, c.shape_c)
        return desc, plan, [c.make_a(), c.make_b(), c.make_c()]
    return desc, eb.Plan(desc, c.shape_a, c.shape_b, strides_b=c.strides_b), \
        [c.make_a(), c.make_b()]


def _case_run(eb, plan, bufs, stream):
    """One launch of a case's plan on device buffers [inputs..., out]."""
    if len(bufs) == 4:
        eb.execute3(plan, *bufs, stream=stream)
    else:
        eb.execute(plan, *bufs, stream=stream)


def time_family_table(eb, torch, cases, l2_bytes, peak):
    """Per-workload GB/s with enough rotating buffer sets to defeat L2."""
    rows = {}
    stream = torch.cuda.current_stream()
    for c in cases:
        desc, plan, host = _case_plan(eb, c)
        osz = eb.ITEMSIZE[desc.out_dtype]
        isz = eb.ITEMSIZE[c.dtype]
        nbytes = sum(x.size for x in host) * isz + plan.numel * osz
        nrot = max(1, math.ceil(4 * l2_bytes / max(nbytes, 1)))
        nrot = min(nrot, 64)
        sets = []
        dev = [upload(x) for x in host]
        for i in range(nrot):
            sets.append([d.clone() if i else d for d in dev] +
                        [torch.empty(plan.numel * osz, dtype=torch.uint8, device="cuda")])
        for i in range(3):
            _case_run(eb, plan, sets[i % nrot], stream)
        # back-to-back launches between two events (the per-launch cost of a
        # pipeline), rotating buffer sets so that each launch reads from HBM
        reps = max(32, 2 * nrot)
        times = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for i in range(reps):
                _case_run(eb, plan, sets[i % nrot], stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e-3 / reps)
        if eb.get_device_status(stream) != 0:
            raise RuntimeError("device status set by " + c.name)
        med = statistics.median(times)
        gbs = nbytes / med / 1e9
        rows[c.name] = {"op": c.op, "dtype": c.dtype, "family": plan.family,
                        "bytes": nbytes, "us_median": round(med * 1e6, 2),
                        "us_best": round(min(times) * 1e6, 2), "gbs": round(gbs, 1),
                        "frac_of_measured": round(gbs / peak, 4),
                        "frac_of_8tbs": round(gbs / HBM_NOMINAL_GBS, 4),
                        "rotating_sets": nrot, "timing": "%d back-to-back launches" % reps}
        del sets, dev
        torch.cuda.empty_cache()
    return rows


def run_ours(args, dist: Dist):
    import numpy as np
    import torch

    import broadcast_elementwise_gb300 as eb
    from datagen import workloads

    torch.cuda.set_device(dist.local_rank)
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = getattr(props, "L2_cache_size", 128 << 20)
    peak, peak_kind = measured_peak()
    stream = torch.cuda.current_stream()

    cm, cd = workloads.by_name(HEADLINE[0]), workloads.by_name(HEADLINE[1])
    a = cm.make_a()
    b_mul = cm.make_b()
    b_div = cd.make_b()
    n = a.size
    dA, dBm, dBd = upload(a), upload(b_mul), upload(b_div)
    dOm = torch.empty(n * 4, dtype=torch.uint8, device="cuda")
    dOd = torch.empty(n * 4, dtype=torch.uint8, device="cuda")
    d_mul = eb.descriptor("Mul", "float32")
    d_div = eb.descriptor("Div", "float32")
    bytes_per_launch = 3 * n * 4
    bytes_per_step = 2 * bytes_per_launch
    h = stream.cuda_stream

    def step(ev=None):
        pm = eb.ebin_plan_create(d_mul.handle, (n,), (n,))       # plan cache hit
        pd = eb.ebin_plan_create(d_div.handle, (n,), (n,))
        if ev:
            ev[0].record(stream)
        eb.ebin_execute(pm, dA.data_ptr(), dBm.data_ptr(), dOm.data_ptr(), h)
        if ev:
            ev[1].record(stream)
        eb.ebin_execute(pd, dA.data_ptr(), dBd.data_ptr(), dOd.data_ptr(), h)
        if ev:
            ev[2].record(stream)
        eb.ebin_plan_release(pm)
        eb.ebin_plan_release(pd)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # timed region: exactly K steps, device-timed
    K = args.steps
    clocks = ClockSampler(dev)
    time.sleep(0.5)
    dist.barrier()
    torch.cuda.synchronize()
    launches0 = eb.ebin_launch_count()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record(stream)
    for _ in range(K):
        step()
    t_stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    dist.barrier()
    launches = eb.ebin_launch_count() - launches0
    total_s = t_start.elapsed_time(t_stop) * 1e-3
    max_s = dist.max(total_s)
    clocks.mark(wall0, wall1)

    # per-launch durations of the two kernels (same stream, events around each)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
    for i in range(K):
        step(evs[i])
    torch.cuda.synchronize()
    mul_s = [e[0].elapsed_time(e[1]) * 1e-3 for e in evs]
    div_s = [e[1].elapsed_time(e[2]) * 1e-3 for e in evs]
    clock_info = clocks.stop()
    if eb.get_device_status(stream) != 0:
        raise RuntimeError("device status set during the benchmark")

    mean_mul, mean_div = statistics.mean(mul_s), statistics.mean(div_s)
    dom_name, dom_s = ("div_f32_contiguous", mean_div) if mean_div >= mean_mul else \
        ("mul_f32_contiguous", mean_mul)
    achieved = bytes_per_launch / dom_s / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profile_traffic(dom_name),
                "kernel": "k_contiguous<%s fp32>" % ("Div" if dom_name.startswith("div") else "Mul"),
                "peak_kind": peak_kind,
                "frac_of_8tbs": round(achieved / HBM_NOMINAL_GBS, 4),
                "mul_us_mean": round(mean_mul * 1e6, 2), "div_us_mean": round(mean_div * 1e6, 2),
                "algorithmic_bytes_per_launch": bytes_per_launch}

    # end to end through the host-buffer entry point
    e2e = None
    if args.e2e_steps > 0:
        hA = torch.from_numpy(a.view(np.uint8)).pin_memory()
        hBm = torch.from_numpy(b_mul.view(np.uint8)).pin_memory()
        hBd = torch.from_numpy(b_div.view(np.uint8)).pin_memory()
        hOm = torch.empty(n * 4, dtype=torch.uint8).pin_memory()
        hOd = torch.empty(n * 4, dtype=torch.uint8).pin_memory()

        def copy_step():
            pm = eb.ebin_plan_create(d_mul.handle, (n,), (n,))
            pd = eb.ebin_plan_create(d_div.handle, (n,), (n,))
            eb.ebin_execute_host(pm, hA.data_ptr(), hBm.data_ptr(), hOm.data_ptr(),
                                 dA.data_ptr(), dBm.data_ptr(), dOm.data_ptr(), h)
            eb.ebin_execute_host(pd, hA.data_ptr(), hBd.data_ptr(), hOd.data_ptr(),
                                 dA.data_ptr(), dBd.data_ptr(), dOd.data_ptr(), h)
            eb.ebin_plan_release(pm)
            eb.ebin_plan_release(pd)

        def mapped_step():
            pm = eb.ebin_plan_create(d_mul.handle, (n,), (n,))
            pd = eb.ebin_plan_create(d_div.handle, (n,), (n,))
            eb.ebin_execute_mapped(pm, hA.data_ptr(), hBm.data_ptr(), hOm.data_ptr(), h)
            eb.ebin_execute_mapped(pd, hA.data_ptr(), hBd.data_ptr(), hOd.data_ptr(), h)
            eb.ebin_plan_release(pm)
            eb.ebin_plan_release(pd)

        def timed_e2e(step):
            step()
            torch.cuda.synchronize()
            dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.e2e_steps):
                step()
            e1.record(stream)
            torch.cuda.synchronize()
            return dist.max(e0.elapsed_time(e1) * 1e-3)

        copy_s = timed_e2e(copy_step)
        e2e_s = timed_e2e(mapped_step)
        # the mapped path wrote the outputs last: check a sample of them
        check = np.random.default_rng(7).integers(0, n, 4096)
        for ho, bb, opname in ((hOm, b_mul, "Mul"), (hOd, b_div, "Div")):
            got = ho.numpy().view(np.float32)[check]
            want = a[check] * bb[check] if opname == "Mul" else a[check] / bb[check]
            if not np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32)):
                raise RuntimeError("mapped end-to-end output differs from float32 %s" % opname)
        e2e = {"value": round(aggregate(bytes_per_step * args.e2e_steps, dist.world, e2e_s), 1),
               "unit": UNIT, "h2d_bytes_per_step": 4 * n * 4, "d2h_bytes_per_step": 2 * n * 4,
               "steps": args.e2e_steps,
               "api": "ebin_execute_mapped (pinned host buffers read and written in place by the "
                      "kernel over NVLink-C2C; inputs and outputs cross the host link every step)",
               "copy_pipeline_value": round(aggregate(bytes_per_step * args.e2e_steps,
                                                      dist.world, copy_s), 1),
               "copy_pipeline_api": "ebin_execute_host (copy engines, chunked over two streams)"}
        del hA, hBm, hBd, hOm, hOd

    # the oracle on a bounded sample, host cores, rank 0 only
    cpu = None
    if dist.rank == 0 and dist.world == 1:
        cpu = cpu_baseline_sample(a, b_mul, b_div)

    families = None
    if not args.no_families and dist.rank == 0:
        del dOm, dOd
        torch.cuda.empty_cache()
        others = [c for c in workloads.cases() if c.name not in HEADLINE]
        families = {}
        for name, ts in ((HEADLINE[0], mul_s), (HEADLINE[1], div_s)):
            med = statistics.median(ts)
            gbs = bytes_per_launch / med / 1e9
            families[name] = {"op": "Mul" if name == HEADLINE[0] else "Div", "dtype": "float32",
                              "family": "contiguous", "bytes": bytes_per_launch,
                              "us_median": round(med * 1e6, 2), "us_best": round(min(ts) * 1e6, 2),
                              "gbs": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
                              "frac_of_8tbs": round(gbs / HBM_NOMINAL_GBS, 4),
                              "rotating_sets": 1}
        families.update(time_family_table(eb, torch, others, l2_bytes, peak))

    value = aggregate(bytes_per_step * K, dist.world, max_s)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dist.world,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(max_s / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64, N(0,1) inputs; Div divisor |N(0,1)|+0.5)",
        "config": {"workload": WORKLOAD, "ops_per_step": ["Mul", "Div"],
                   "family": "contiguous", "bytes_per_step": bytes_per_step,
                   "l2": "inputs larger than L2 (3 GiB per step vs %d MiB L2); no flush"
                         % (l2_bytes >> 20),
                   "parallelism": "replicas" if dist.world > 1 else "single GPU",
                   "gpu": props.name},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clock_info, "families": families,
    }
    if dist.rank == 0:
        print(json.dumps(out), flush=True)


def host_cpu():
    """(CPU model, logical cores) of the host the baseline runs on."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return model or platform.processor() or platform.machine(), os.cpu_count()


def cpu_baseline_sample(a, b_mul, b_div, min_seconds=10.0, max_passes=16):
    """The oracle on the host: whole Mul+Div passes over the workload until
    about `min_seconds` of single-threaded CPU work has been done."""
    import oracle
    passes = 0
    t0 = time.perf_counter()
    while passes < max_passes:
        oracle.run("Mul", a, b_mul, "float32")
        oracle.run("Div", a, b_div, "float32")
        passes += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    model, nproc = host_cpu()
    return {"value": round(passes * 2 * 3 * a.size * 4 / dt / 1e9, 4), "unit": UNIT, "cores": 1,
            "kind": "oracle", "cpu_model": model, "nproc": nproc,
            "sample": "%d full Mul+Div pass(es) over the %d-element workload (single-threaded C "
                      "oracle, full multi-index per element), %.1f s" % (passes, a.size, dt)}


# ----------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    from datagen import workloads
    import oracle
    n_sample = 1 << 22
    cm, cd = workloads.by_name(HEADLINE[0], scale_log2=28 - 22), \
        workloads.by_name(HEADLINE[1], scale_log2=28 - 22)
    a, bm, bd = cm.make_a(), cm.make_b(), cd.make_b()
    assert a.size == n_sample

    def step():
        oracle.run("Mul", a, bm, "float32")
        oracle.run("Div", a, bd, "float32")

    for _ in range(max(args.warmup, 3)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = 2 * 3 * n_sample * 4 * args.steps / dt / 1e9
    sample = ("Mul and Div on the first %d of the 2^28 elements per step (single-threaded C "
              "oracle, full multi-index per element)" % n_sample)
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
           "n_gpus": dist.world, "steps": args.steps, "warmup": max(args.warmup, 3),
           "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": WORKLOAD, "ops_per_step": ["Mul", "Div"], "sample": sample},
           "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                            "cpu_model": host_cpu()[0], "nproc": host_cpu()[1],
                            "sample": sample},
           "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_one_case(args):
    """One workload alone: warmup, then --steps launches timed one by one."""
    import torch

    import broadcast_elementwise_gb300 as eb
    from datagen import workloads

    c = workloads.by_name(args.only, scale_log2=args.scale_log2)
    desc, plan, host = _case_plan(eb, c)
    osz = eb.ITEMSIZE[desc.out_dtype]
    bufs = [upload(x) for x in host] + \
        [torch.empty(plan.numel * osz, dtype=torch.uint8, device="cuda")]
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        _case_run(eb, plan, bufs, stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s0, s1 in evs:
        s0.record(stream)
        _case_run(eb, plan, bufs, stream)
        s1.record(stream)
    torch.cuda.synchronize()
    if eb.get_device_status(stream) != 0:
        raise RuntimeError("device status set")
    ts = [x.elapsed_time(y) * 1e-3 for x, y in evs]
    nbytes = sum(x.size for x in host) * eb.ITEMSIZE[c.dtype] + plan.numel * osz
    med = statistics.median(ts)
    print(json.dumps({"case": c.name, "family": plan.family, "numel": plan.numel,
                      "bytes": nbytes, "us_median": round(med * 1e6, 2),
                      "gbs": round(nbytes / med / 1e9, 1)}), flush=True)


def run_cases(args):
    """The per-workload table for the named workloads only, one JSON line each."""
    import torch

    import broadcast_elementwise_gb300 as eb
    from datagen import workloads

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2_bytes = getattr(props, "L2_cache_size", 128 << 20)
    peak, _ = measured_peak()
    names = [n.strip() for n in args.cases.split(",") if n.strip()]
    rows = time_family_table(eb, torch, [workloads.by_name(n) for n in names], l2_bytes, peak)
    for name in names:
        print(json.dumps(dict(case=name, **rows[name])), flush=True)


def main():
    args = parse_args()
    if args.only:
        run_one_case(args)
        return
    if args.cases:
        run_cases(args)
        return
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
