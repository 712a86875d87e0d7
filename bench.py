"""Benchmark of the fused DW->PW convolution module on GB300.

One step = one fused evaluation (fcm_run, mode FUSED) of the whole batch of the MobileNet-style
layer: N=64, 56x56, C=128, DW 3x3 s1 p1 + ReLU6, PW 128->128 + ReLU6, fp16 storage with fp32
accumulation.  Inputs are seeded synthetic tensors already resident in HBM; to keep L2 (129 MB)
from serving them, each step uses the next of R input/output buffer sets whose total is more
than twice the L2 size.

Prints ONE JSON line (rank 0).  `value` is the achieved algorithmic HBM bandwidth (input +
weights + scale/bias + output, each once) of the whole job over K steps launched back to back
between two CUDA events (no event between launches, which would serialise them); images/s is
reported beside it, and the spread of single launches from a separate untimed pass.  `e2e`
measures the same bytes end to end from pinned host memory through fcm_run_host_async, every
step's copies in and out inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--mode fused|unfused]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host cores
  python bench.py --report FILE          # also time every workload, fused and unfused
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

METRIC = ("fused DW→PW conv: achieved HBM GB/s (% of roofline) and images/s per layer")
L2_BYTES = 129 * 1024 * 1024
DEFAULT_WORKLOAD = "mobilenet_dwpw_f16"
DATA = ("synthetic: seeded splitmix64 streams; activations N(0,1), weights N(0,1/fan_in), "
        "scale U[0.5,1.5], bias U[-0.1,0.1] (uniform[-1,1] for the fp32 layer)")
DATA_I8 = ("synthetic: seeded splitmix64 streams; int8 activations and weights uniform on "
           "[-128,127], fp32 requantization scales U[0.5,1.5] x 32/(spread of the accumulator), "
           "biases U[-4,4]")


def data_of(wl) -> str:
    return DATA_I8 if wl.dtype == "i8" else DATA


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--mode", default="fused", choices=["fused", "unfused"])
    p.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc", "tc_roles", "tc_workers"])
    p.add_argument("--report", default=None, help="write a per-workload JSON report here")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    return p.parse_args()


# --------------------------------------------------------------------------- environment
def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_digest() -> str:
    """Digest of the files that define the tensor-core kernels and their launch plans (the
    DRAM traffic of a launch depends on nothing else)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "pointwise_conv_cnn_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("tc_") or f == "fcm_device.cuh":
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, mode: str) -> dict:
    """DRAM bytes (read + written) of one step and the bytes the step's kernels wrote (L2
    write sectors), from the committed ncu summary, only if it was taken on the current kernel
    sources; nulls otherwise."""
    none = {"dram": None, "l2_write": None}
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return none
    try:
        d = json.load(open(path))
        ent = d.get(f"{workload}:{mode}")
        if ent and ent.get("source_digest") == kernel_source_digest():
            dram = ent.get("dram_bytes_per_launch", ent.get("dram_bytes_per_step"))
            return {"dram": dram, "l2_write": ent.get("l2_write_bytes")}
    except (OSError, ValueError, AttributeError):
        pass
    return none


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:9]))
            except Exception:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows[-3:]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------------------------ our path
def torch_dtype(torch, dtype):
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
            "i8": torch.int8}[dtype]


def oracle_step(oracle, wk, wl, case, nthreads: int):
    """One evaluation of the oracle's single-pass module on `case` (fp64, or the INT8 one) with
    `nthreads` OpenMP threads (the oracle's thread count is sticky, so every call sets it)."""
    if wl.dtype == "i8":
        fn = {"dense": oracle.fused_dense_i8, "pwdw": oracle.pwdw_i8}.get(wl.conv1, oracle.fused_i8)
        return lambda: fn(case.x, case.w1, case.s1, case.b1, case.wp, case.s2, case.b2, wl.act1,
                          wl.act2, wl.stride, wl.pad, nthreads=nthreads)
    f = case.f64()
    return lambda: oracle.fused(f["x"], f["w1"], f["s1"], f["b1"], f["wp"], f["s2"], f["b2"],
                                wl.act1, wl.act2, wl.stride, wl.pad, conv1=wl.conv1,
                                nthreads=nthreads)


def storage_tensor(torch, arr, dtype):
    import numpy as np
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr))


def time_ours(torch, fcm, wk, wl, mode, kernel, steps, warmup, device, dist=None,
              sample_clocks=False):
    case = wk.make_case(wl)
    mod = fcm.FusedConvModule(fcm.desc_from_workload(wl, kernel=kernel), case.w1, case.wp,
                              case.s1, case.b1, case.s2, case.b2)
    sh = wl.shapes()
    mb = wl.min_bytes()
    set_bytes = mb["x"] + mb["y"]
    nsets = max(2, math.ceil(2 * L2_BYTES / set_bytes) + 1)
    x0 = storage_tensor(torch, case.x, wl.dtype).to(device)
    xs = [x0] + [x0.clone() for _ in range(nsets - 1)]
    ys = [torch.empty(sh["y"], dtype=torch_dtype(torch, wl.dtype), device=device)
          for _ in range(nsets)]
    stream = torch.cuda.Stream(device=device)
    launches_per_step = 2 if mode == "unfused" else 1
    with torch.cuda.stream(stream):
        for i in range(warmup):
            mod.run(xs[i % nsets], ys[i % nsets], mode, stream=stream)
        stream.synchronize()
        mod.check(stream)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(device)
        sampler = ClockSampler(device.index or 0) if sample_clocks else None
        if sampler:
            sampler.start()
            time.sleep(0.3)
        t0 = time.time()
        # The timed region holds the launches alone: an event recorded between two launches
        # would make the second wait for the first to finish, where programmatic dependent
        # launch lets its prologue overlap the first one's tail.
        start.record(stream)
        for i in range(steps):
            mod.run(xs[i % nsets], ys[i % nsets], mode, stream=stream)
        end.record(stream)
        end.synchronize()
        t1 = time.time()
        torch.cuda.synchronize(device)
        if dist is not None:
            dist.barrier()
        clocks = sampler.stop(t0, t1) if sampler else None
        mod.check(stream)
        # Untimed pass: each launch between its own pair of events (launches serialised), for
        # the spread of single-launch durations.
        n_iso = min(steps, 200)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_iso)]
        for i in range(n_iso):
            ev[i][0].record(stream)
            mod.run(xs[i % nsets], ys[i % nsets], mode, stream=stream)
            ev[i][1].record(stream)
        stream.synchronize()
        mod.check(stream)
    region_ms = start.elapsed_time(end)
    iso_ms = [a.elapsed_time(b) for a, b in ev]
    res = {"region_ms": region_ms, "ms_per_step": region_ms / steps,
           "iso_ms_mean": statistics.fmean(iso_ms), "iso_ms_median": statistics.median(iso_ms),
           "iso_ms_p10": percentile(iso_ms, 10), "iso_ms_p90": percentile(iso_ms, 90),
           "nsets": nsets, "set_bytes": set_bytes, "plan": mod.plan, "clocks": clocks,
           "launches": steps * launches_per_step, "case": case, "module": mod}
    return res


def percentile(values, q: float) -> float:
    """q-th percentile, linear between the closest ranks."""
    v = sorted(values)
    if not v:
        return float("nan")
    pos = (len(v) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (pos - lo)


def time_e2e(torch, mod, case, wl, mode, steps, device):
    """End to end through the public API: every step copies its input from pinned host memory,
    runs the module and copies the result back to pinned host memory (fcm_run_host_async, so
    that one step's output copies overlap the next step's input copies, as a serving loop
    would run them); the region ends when the stream has completed the last step's copy out."""
    sh = wl.shapes()
    x_h = storage_tensor(torch, case.x, wl.dtype).pin_memory()
    y_h = torch.empty(sh["y"], dtype=torch_dtype(torch, wl.dtype)).pin_memory()
    stream = torch.cuda.Stream(device=device)
    for _ in range(2):
        mod.run_host(x_h, y_h, mode, stream=stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    start.record(stream)
    for _ in range(steps):
        mod.run_host_async(x_h, y_h, mode, stream=stream)
    end.record(stream)
    end.synchronize()
    mb = wl.min_bytes()
    return start.elapsed_time(end) / steps, mb["x"], mb["y"]


def cpu_baseline(wk, wl, seconds: float) -> dict:
    """The fp64 oracle as it stands, on a bounded sample of the same workload (whole images,
    the batch repeated if one pass is shorter than `seconds`), all host cores (OpenMP)."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    mb = wl.min_bytes()
    per_image_bytes = mb["fused"] / wl.n

    def timed(n_img, reps):
        sub = wl.with_(n=n_img)
        run = oracle_step(oracle, wk, sub, wk.make_case(sub), threads)
        t = time.perf_counter()
        for _ in range(reps):
            run()
        return time.perf_counter() - t

    t1 = timed(1, 1)
    # one image on one core, for the single-threaded figure
    sub1 = wl.with_(n=1)
    run1 = oracle_step(oracle, wk, sub1, wk.make_case(sub1), 1)
    ts = time.perf_counter()
    run1()
    t_single = time.perf_counter() - ts
    n_img = int(max(1, min(wl.n, seconds / max(t1, 1e-6))))
    reps = max(1, int(seconds / max(t1 * n_img, 1e-6)))
    t = timed(n_img, reps)
    ips = n_img * reps / t
    return {"value": round(ips * per_image_bytes / 1e9, 6), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "images_per_s": round(ips, 4),
            "single_thread_images_per_s": round(1.0 / t_single, 4),
            "sample": f"{n_img} of {wl.n} images of {wl.name} x {reps} passes, "
                      f"{'INT8 oracle' if wl.dtype == 'i8' else 'fp64 oracle_fused'}, "
                      f"{threads} OpenMP threads, {t:.2f} s"}


# ------------------------------------------------------------------ multi-rank aggregation
def max_over_ranks(value: float, dist, device) -> float:
    """The largest `value` over all ranks (the slowest rank's time), or `value` alone when
    there is no process group.  `device` is where the reduction tensor lives (cuda for NCCL,
    cpu for gloo)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: int, images_per_rank: int, world: int, region_ms: float,
                   steps: int) -> tuple[float, float]:
    """Whole-job GB/s and images/s: every rank runs its own replica of the step (weak
    scaling), so the job moves world x the per-rank bytes in the slowest rank's time."""
    step_s = region_ms / 1e3 / steps
    return bytes_per_rank * world / step_s / 1e9, images_per_rank * world / step_s


def run_ours(args):
    import torch
    import pointwise_conv_cnn_gb300 as fcm
    from pointwise_conv_cnn_gb300 import build as nvbuild
    from pointwise_conv_cnn_gb300 import workloads as wk

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    if rank == 0:
        nvbuild.build()
    if dist is not None:
        dist.barrier()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wl = wk.BY_NAME[args.workload]
    res = time_ours(torch, fcm, wk, wl, args.mode, args.kernel, args.steps, args.warmup, device,
                    dist, sample_clocks=(local == 0))
    region_ms = max_over_ranks(res["region_ms"], dist, device)
    steps = args.steps
    mb = wl.min_bytes()
    value, images_per_s = job_throughput(mb["fused"], wl.n, world, region_ms, steps)
    peaks = load_peaks()
    # the step's launches back to back inside the timed region (max over ranks): one launch of
    # the fused kernel per step in the default mode
    step_s = region_ms / steps / 1e3
    traffic = ncu_traffic(wl.name, args.mode)
    achieved = mb["fused"] / step_s / 1e9
    e2e_ms, hb, db = time_e2e(torch, res["module"], res["case"], wl, args.mode,
                              max(5, min(100, steps // 10)), device)
    e2e_value = mb["fused"] * world / (e2e_ms / 1e3) / 1e9
    plan = res["plan"]
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(region_ms / steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"i8": "int8"}.get(wl.dtype, wl.dtype),
        "data": data_of(wl),
        "config": {"workload": wl.name, "n": wl.n, "h": wl.h, "w": wl.w, "c": wl.c,
                   "k_out": wl.k_out, "conv1": wl.conv1, "ksize": wl.ksize, "stride": wl.stride,
                   "pad": wl.pad, "act1": wl.act1, "act2": wl.act2, "mode": args.mode,
                   "kernel": {1: "simt", 2: "tcgen05"}[plan["kernel"]],
                   "tile": [plan["tile_h"], plan["tile_w"]], "ctas": plan["ctas"],
                   "global_batch": wl.n * world, "parallelism": f"replicas{world}",
                   "l2": f"rotating {res['nsets']} input/output sets "
                         f"({res['nsets'] * res['set_bytes'] / 2**20:.0f} MiB > 2 x 129 MB L2)"},
        "images_per_s": round(images_per_s, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 3),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic["dram"],
                     "traffic_l2_write": traffic["l2_write"],
                     "bytes_per_launch": mb["fused"],
                     "step_us": round(step_s * 1e6, 3),
                     "launches_per_step": res["launches"] // steps,
                     "isolated_us_mean": round(res["iso_ms_mean"] * 1e3, 3),
                     "isolated_us_median": round(res["iso_ms_median"] * 1e3, 3),
                     "isolated_us_p10": round(res["iso_ms_p10"] * 1e3, 3),
                     "isolated_us_p90": round(res["iso_ms_p90"] * 1e3, 3),
                     "peak_source": peaks["source"]},
        "e2e": {"value": round(e2e_value, 3), "unit": "GB/s", "h2d_bytes_per_step": hb,
                "d2h_bytes_per_step": db, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wk, wl, args.cpu_seconds)
    if args.report and rank == 0:
        out_report = {"headline": out, "workloads": report_all(torch, fcm, wk, device)}
        with open(args.report, "w") as f:
            json.dump(out_report, f, indent=1, default=str)
    if rank == 0:
        print(json.dumps(out, default=str), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def report_all(torch, fcm, wk, device):
    rows = []
    peaks = load_peaks()
    for wl in wk.WORKLOADS:
        for mode in ("fused", "unfused"):
            for kernel in ("auto", "simt"):
                if kernel == "simt" and wl.dtype in ("f32", "i8"):   # f32: SIMT only; i8: TC only
                    continue
                steps = 200 if wl.n > 1 else 2000
                try:
                    r = time_ours(torch, fcm, wk, wl, mode, kernel, steps, 10, device)
                except Exception as e:  # an unsupported request is recorded, not fatal
                    rows.append({"workload": wl.name, "mode": mode, "kernel": kernel,
                                 "error": str(e)})
                    continue
                mb = wl.min_bytes()
                ks = r["ms_per_step"] / 1e3
                rows.append({"workload": wl.name, "mode": mode, "kernel": kernel,
                             "chosen": {1: "simt", 2: "tcgen05"}[r["plan"]["kernel"]],
                             "us_per_step": round(ks * 1e6, 3),
                             "isolated_us": round(r["iso_ms_mean"] * 1e3, 3),
                             "isolated_us_median": round(r["iso_ms_median"] * 1e3, 3),
                             "isolated_us_p10_p90": [round(r["iso_ms_p10"] * 1e3, 3),
                                                     round(r["iso_ms_p90"] * 1e3, 3)],
                             "images_per_s": round(wl.n / ks, 1),
                             "algo_gbs": round(mb["fused"] / ks / 1e9, 1),
                             "frac_hbm": round(mb["fused"] / ks / 1e9 / peaks["hbm_gbs"], 4),
                             "plan": r["plan"]})
                r["module"].close()
    return rows


# ------------------------------------------------------------------------ reference arm
def run_reference(args):
    """The fp64 CPU oracle, as it stands, on the host cores: each step evaluates a bounded
    sample (whole images) of the same workload; rank 0 alone runs it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from pointwise_conv_cnn_gb300 import workloads as wk
    oracle.build()
    wl = wk.BY_NAME[args.workload]
    threads = oracle.max_threads()
    n_img = 1 if wl.n > 1 else wl.n
    sub = wl.with_(n=n_img)
    step = oracle_step(oracle, wk, sub, wk.make_case(sub), threads)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t) / args.steps
    per_image = wl.min_bytes()["fused"] / wl.n
    value = n_img * per_image / dt / 1e9
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
           "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None,
           "dtype": "int8" if wl.dtype == "i8" else "f64", "data": data_of(wl),
           "config": {"workload": wl.name, "n": wl.n, "h": wl.h, "w": wl.w, "c": wl.c,
                      "k_out": wl.k_out, "images_per_step": n_img},
           "images_per_s": round(n_img / dt, 4),
           "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": threads,
                            "kind": "oracle",
                            "sample": f"{n_img} image(s) of {wl.n} per step of {wl.name}, "
                                      f"{'INT8' if wl.dtype == 'i8' else 'fp64'} oracle, "
                                      f"{threads} OpenMP threads"},
           "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
