#!/usr/bin/env python3
"""DBSCAN benchmark: pair evaluations per second (N^2 / t) and end-to-end ms.

Default workload: blobs_1m_d3 (N = 1,000,000 integer points in [0, 2047]^3,
500 Gaussian blobs sigma = 12, 3 filaments, 20% uniform noise; eps = 10,
minPts = 8), seeded and synthetic.  One step = one full DBSCAN (prep, count,
compact, union, flatten, border, finalize) on device-resident points; the L2
is flushed (a 256 MiB write) between timed steps, outside the timed events.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the CPU oracle
instead (bounded samples of the same workload, on the host cores).
Under torchrun (N > 1) each rank runs an independent replica of the workload
(no data-path collective); timing is the max over ranks.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DBSCAN pair evals/s (N²/t) and end-to-end ms at N=1M, d=3, one GB300"
UNIT = "pair evals/s"
FP32_LANES_PER_SM = 128          # FP32 FMA lanes per Blackwell SM
SM_COUNT_FALLBACK = 152
SM_MAX_MHZ_FALLBACK = 2070.0
BF16_FALLBACK_TFLOPS = 1900.0    # recipe fallback when no measured peak exists
TF32_PER_BF16 = 1.1 / 2.25       # nominal dense tf32 / bf16 ratio


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="blobs_1m_d3")
    ap.add_argument("--n", type=int, default=None,
                    help="run a smaller set drawn like the workload (profiling cases only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-culled", action="store_true")
    ap.add_argument("--no-f16acc", action="store_true",
                    help="skip timing the opt-in f16-accumulator variant")
    ap.add_argument("--no-ffma", action="store_true",
                    help="skip timing the same call on CUDA cores only (fp32 FFMA)")
    ap.add_argument("--no-fused", action="store_true",
                    help="small problems too take the multi-kernel path")
    ap.add_argument("--force-path", default=None,
                    choices=["fp32", "tf32", "bf16", "f16", "f16acc16"],
                    help="allow only this arithmetic path (fp32 = CUDA cores)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (timing only)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.idx = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return None


def count_flops(n: int, d: int) -> float:
    """Algorithmic FLOP of the count sweep: each unordered pair once, d FMAs."""
    return 2.0 * d * n * (n - 1) / 2.0


KERNEL_FILES = ("sweep_tc.cu", "tc_schedule.h", "dbscan_internal.cuh")


def kernel_code_hash(texts=None) -> str:
    """sha256 of the tensor-core sweep's code: its source and the headers it
    includes (or the given texts), with comments and blank lines removed (a
    comment edit does not change the kernel)."""
    if texts is None:
        texts = [open(os.path.join(ROOT, "all_pairs_distance_gb300", "csrc", name)).read()
                 for name in KERNEL_FILES]
    h = hashlib.sha256()
    for text in texts:
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.strip() for ln in text.splitlines() if ln.strip()]
        h.update(("\n".join(lines) + "\n").encode())
    return h.hexdigest()


def recorded_profile(workload: str, path: str, key: str):
    """A figure of the count sweep's committed ncu capture
    (``profiles/count_sweep_<workload>.json``), or None when the record is
    missing, the kernel's code changed since it was taken, or this run took
    another path."""
    rec_path = os.path.join(ROOT, "profiles", f"count_sweep_{workload}.json")
    if not os.path.exists(rec_path):
        return None
    with open(rec_path) as f:
        rec = json.load(f)
    if rec.get("sweep_path") != path or rec.get("sweep_code_sha256") != kernel_code_hash():
        return None
    v = rec.get(key)
    return float(v) if v is not None else None


def recorded_traffic(workload: str, path: str):
    """Per-launch DRAM bytes of the count sweep from the committed ncu record,
    or None when the record is missing, the kernel's code changed since, or
    this run took another path."""
    return recorded_profile(workload, path, "traffic_bytes_per_launch")


def executed_count_flops(n: int, kpad: int) -> float:
    """FLOP the tensor-core count sweep executes per launch: every 128 x 128
    tile pair of the upper triangle (diagonal included) as a K = kpad MMA."""
    t = (n + 127) // 128
    return t * (t + 1) / 2.0 * 128.0 * 128.0 * 2.0 * kpad


def cpu_baseline(P, eps, min_pts, target_s=12.0):
    """The oracle as it stands on a leading sample of the workload, sized for
    about target_s seconds of single-threaded work.  -> dict."""
    import oracle
    m0 = min(len(P), 6000)
    t = time.perf_counter()
    oracle.dbscan(P[:m0], eps, min_pts)
    t0 = time.perf_counter() - t
    per_pair = t0 / (m0 * m0)
    m = int(min(len(P), max(m0, (target_s / per_pair) ** 0.5)))
    t = time.perf_counter()
    oracle.dbscan(P[:m], eps, min_pts)
    dt = time.perf_counter() - t
    return {"value": m * m / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {m} of {len(P)} points of the workload, full oracle DBSCAN "
                      f"(count + BFS), single-threaded, {dt:.1f} s"}


def cpu_baseline_parallel(P, eps, min_pts, m=40000):
    """The same oracle source built with OpenMP (its count loop on all host
    cores; the cluster expansion stays serial, and dominates) on the first m
    points.  -> dict, or None without an OpenMP compiler."""
    import oracle
    threads = oracle.parallel_threads()
    if threads == 0:
        return None
    m = min(len(P), m)
    t = time.perf_counter()
    oracle.dbscan_parallel(P[:m], eps, min_pts)
    dt = time.perf_counter() - t
    t = time.perf_counter()
    oracle.dbscan(P[:m], eps, min_pts)       # the single-threaded build on the same sample
    ds = time.perf_counter() - t
    return {"value": m * m / dt, "unit": UNIT, "cores": threads,
            "kind": "oracle, OpenMP build of the same source",
            "single_thread_same_sample": m * m / ds,
            "sample": f"first {m} of {len(P)} points of the workload, full oracle DBSCAN "
                      f"(count on {threads} threads, cluster expansion serial), {dt:.1f} s"}


# arithmetic of each path: operand type and accumulator
DTYPE_NAMES = {"fp32": "f32", "tf32": "tf32-f32acc", "bf16": "bf16-f32acc", "f16": "f16-f32acc",
               "f16acc16": "f16-f16acc"}


def roofline_fields(info, n, d, count_ms, peaks, sms, max_mhz) -> dict:
    """Roofline of the count sweep against the peak of the unit that runs it:
    the FP32 CUDA-core peak (derived) for the fp32 path, else the dense tensor
    peak of the MMA kind (f16 and bf16 at the measured bf16 rate, tf32 at the
    nominal tf32/bf16 ratio).  ``achieved`` counts algorithmic FLOP (2d per
    unordered pair); ``executed_frac`` counts what the MMAs execute (the
    operand rows padded to K), and ``encoding_ceiling`` is their ratio, the
    most ``frac`` can reach with the tensor pipe saturated."""
    path = info["path"]
    achieved = count_flops(n, d) / (count_ms * 1e-3) / 1e12
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * max_mhz * 1e6 / 1e12
    fp32_source = (f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x "
                   f"{max_mhz:.0f} MHz (max SM clock" +
                   (", MEASURED_PEAKS.json)" if peaks else ", recipe fallback)"))
    if path == "fp32":
        kernel = ("fused single-launch pipeline (every stage in one cooperative kernel, fp32 FFMA "
                  "on CUDA cores; its whole time is charged to the count's FLOP)"
                  if info.get("fused") else "count sweep on CUDA cores (fp32 FFMA, upper triangle)")
        return {"bound": "alu", "achieved": achieved, "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": achieved / fp32_peak, "kernel": kernel,
                "peak_source": fp32_source + " -- of derived FP32 FMA peak"}
    bf16 = (peaks or {}).get("bf16_tflops", BF16_FALLBACK_TFLOPS)
    sust = (peaks or {}).get("bf16_tflops_sustained")
    ratio = TF32_PER_BF16 if path == "tf32" else 1.0
    tc_peak = bf16 * ratio
    src = ("measured bf16 burst (MEASURED_PEAKS.json) -- of measured" if peaks else
           "recipe fallback bf16 -- of fallback")
    if path == "tf32":
        src += f"; x {TF32_PER_BF16:.3f} (nominal dense tf32/bf16 ratio 1.1/2.25)"
    elif path != "bf16":
        src += "; f16 shares the dense bf16 rate"
    executed = executed_count_flops(n, info["kpad"]) / (count_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
            "frac": achieved / tc_peak,
            "executed_tflops": executed, "executed_frac": executed / tc_peak,
            "encoding_ceiling": count_flops(n, d) / executed_count_flops(n, info["kpad"]),
            "encoding_note": f"2d = {2 * d} algorithmic FLOP per pair against 2K = "
                             f"{2 * info['kpad']} executed (K = {info['kpad']}: the d coordinates "
                             "plus the norm and threshold digits, padded to the MMA's K step)",
            "frac_vs_sustained": achieved / (sust * ratio) if sust else None,
            "kernel": f"count sweep on tensor cores (tcgen05 {DTYPE_NAMES[path]}, "
                      f"K={info['kpad']}, upper triangle)",
            "peak_source": src,
            "fp32_equivalent": {"achieved": achieved, "peak": fp32_peak,
                                "frac": achieved / fp32_peak,
                                "note": "the same algorithmic FLOP against the derived FP32 "
                                        "CUDA-core peak (" + fp32_source + ")"}}


# ---------------------------------------------------------------------------
def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return 0
    import oracle
    from all_pairs_distance_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    P = synth.generate(args.workload) if args.n is None else synth.scaled(args.workload, args.n)
    n = len(P)
    m = min(n, 20_000 if w.d <= 4 else 6_000)
    S = P[:m]
    for _ in range(args.warmup):
        oracle.dbscan(S, w.eps, w.min_pts)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.dbscan(S, w.eps, w.min_pts)
        times.append(time.perf_counter() - t)
    step = sum(times) / len(times)
    value = m * m / step
    name = w.name if args.n is None else f"{w.name} scaled to n={n}"
    sample = (f"first {m} of {n} points of {name} per step, full oracle DBSCAN "
              f"(count + BFS), single-threaded")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": name, "n": n, "d": w.d, "eps": w.eps,
                       "min_pts": w.min_pts, "sample_points": m},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args, dist: Dist):
    import torch
    from all_pairs_distance_gb300 import binding, synth
    from all_pairs_distance_gb300 import build as lib_build

    w = synth.WORKLOADS[args.workload]
    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    binding.load()
    if args.no_fused:
        binding.dbscan_set_options(fused=0)
    if args.force_path:
        binding.dbscan_set_options(paths=[args.force_path])
    P = synth.generate(args.workload) if args.n is None else synth.scaled(args.workload, args.n)
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x = torch.from_numpy(P).to(dev).to(dtype)
    n, d = x.shape
    ws = binding.workspace_for(x)
    labels = torch.empty(n, dtype=torch.int32, device=dev)
    is_core = torch.empty(n, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # a stream of our own: the library captures a repeated call (same stream,
    # workspace and buffers) into a CUDA graph in warm-up and replays it
    stream = torch.cuda.Stream(device=dev)

    def step():
        binding.dbscan_fit_ex(x, w.eps, w.min_pts, labels=labels, is_core=is_core,
                              workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            step()
    torch.cuda.synchronize()
    st = binding.dbscan_workspace_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {binding.dbscan_strerror(st)}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dist.local) if dist.rank == 0 else None
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop() if clocks else None
    # stage times and launch count: the same steps again with the library's
    # stage events (these calls launch directly: events are not captured)
    binding.dbscan_profile_begin()
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush.zero_()
            step()
    torch.cuda.synchronize()
    stage_ms, calls, launches = binding.dbscan_profile_end()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_ms = sum(step_ms) / len(step_ms)
    mean_ms = dist.max(mean_ms)
    value = dist.world * float(n) * float(n) / (mean_ms * 1e-3)
    st = binding.dbscan_workspace_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {binding.dbscan_strerror(st)}")

    # roofline of the dominant kernel (the count sweep) on the path the data took
    info = binding.dbscan_workspace_info(ws)
    count_ms = stage_ms["count"] / max(calls, 1)
    peaks = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = getattr(props, "multi_processor_count", SM_COUNT_FALLBACK)
    max_mhz = (peaks or {}).get("sm_max_mhz", SM_MAX_MHZ_FALLBACK)
    roofline = roofline_fields(info, n, d, count_ms, peaks, sms, max_mhz)
    roofline["traffic"] = recorded_traffic(w.name, info["path"])
    # the executed view: the tensor pipe's active share in the committed ncu
    # capture of this kernel and path (null once the kernel's code changed)
    tp_active = recorded_profile(w.name, info["path"], "tensor_pipe_active_pct")
    roofline["ncu_tensor_pipe_active"] = tp_active / 100.0 if tp_active is not None else None

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_NAMES[info["path"]],
            "data": "synthetic",
            "config": {"workload": w.name if args.n is None else f"{w.name} scaled to n={n}",
                       "n": n, "d": d, "eps": w.eps, "min_pts": w.min_pts,
                       "input_dtype": w.dtype, "l2": "flushed between steps (256 MiB write, untimed)",
                       "launch": "each step replays the call's CUDA graph (captured in warm-up) "
                                 "on a dedicated stream; stage times from a second, event-marked pass",
                       "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU"},
            "stages_ms": {k: v / max(calls, 1) for k, v in stage_ms.items()},
            "path": info["path"], "fused_pipeline": info["fused"],
            "n_core": info["n_core"], "n_cand": info["n_cand"],
            "exact": info["exact"],
            "count_pair_evals_per_s": float(n) * n / (count_ms * 1e-3),
            "roofline": roofline, "gpu_launches": launches, "clocks": clk}

    # Tile culling (dbscan_fit_culled), reported beside the headline: same
    # results, but pairs in tiles whose boxes are eps apart are never
    # evaluated, so its time is not an all-pairs figure.
    if not args.no_culled:
        def step_culled():
            binding.dbscan_fit_culled(x, w.eps, w.min_pts, labels=labels, is_core=is_core,
                                      workspace=ws, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush.zero_()
                step_culled()
        cs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ce = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        dist.barrier()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                flush.zero_()
                cs[k].record(stream)
                step_culled()
                ce[k].record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        binding.dbscan_profile_begin()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                flush.zero_()
                step_culled()
        torch.cuda.synchronize()
        c_stage_ms, c_calls, _ = binding.dbscan_profile_end()
        st = binding.dbscan_workspace_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {binding.dbscan_strerror(st)}")
        c_ms = dist.max(sum(a.elapsed_time(b) for a, b in zip(cs, ce)) / args.steps)
        line["culled"] = {"ms_per_step": c_ms, "speedup_vs_all_pairs": mean_ms / c_ms,
                          "stages_ms": {k: v / max(c_calls, 1) for k, v in c_stage_ms.items()},
                          "api": "dbscan_fit_culled",
                          "note": "tile pairs whose bounding boxes are eps apart are skipped "
                                  "(identical labels); not an all-pairs evaluation, so no "
                                  "pair-evals/s figure"}

    def timed_variant(paths, step_fn=step):
        """Mean ms of args.steps calls with only `paths` allowed (warm-up and
        L2 flushes as for the headline), the stage times of a second pass, and
        the path the call took."""
        with binding.options(paths=paths):
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    flush.zero_()
                    step_fn()
            torch.cuda.synchronize()
            vs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            ve = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            dist.barrier()
            with torch.cuda.stream(stream):
                for k in range(args.steps):
                    flush.zero_()
                    vs[k].record(stream)
                    step_fn()
                    ve[k].record(stream)
            torch.cuda.synchronize()
            dist.barrier()
            binding.dbscan_profile_begin()
            with torch.cuda.stream(stream):
                for k in range(args.steps):
                    flush.zero_()
                    step_fn()
            torch.cuda.synchronize()
            v_stage_ms, v_calls, _ = binding.dbscan_profile_end()
            v_info = binding.dbscan_workspace_info(ws)
        st = binding.dbscan_workspace_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {binding.dbscan_strerror(st)}")
        v_ms = dist.max(sum(a.elapsed_time(b) for a, b in zip(vs, ve)) / args.steps)
        return v_ms, {k: v / max(v_calls, 1) for k, v in v_stage_ms.items()}, v_info

    # The opt-in f16-accumulator variant of the f16 path (DBSCAN_PATH_F16_ACC16),
    # reported in a field of its own: it accumulates in f16, narrower than the
    # float32 the headline uses.
    if info["path"] == "f16" and not args.no_f16acc and not args.force_path:
        h_ms, h_stages, h_info = timed_variant(binding.PATHS_DEFAULT | binding.PATH_BITS["f16acc16"])
        if h_info["path"] == "f16acc16":   # the opt-in path needs rows of one K = 16 MMA
            h_count = h_stages["count"]
            line["f16_accumulator_optin"] = {
                "path": h_info["path"], "dtype": DTYPE_NAMES[h_info["path"]], "ms_per_step": h_ms,
                "value": dist.world * float(n) * n / (h_ms * 1e-3), "unit": UNIT,
                "count_ms": h_count,
                "count_frac_of_tensor_peak": count_flops(n, d) / (h_count * 1e-3) / 1e12 /
                                             roofline["peak"],
                "note": "opt-in DBSCAN_PATH_F16_ACC16: f16 operands and an f16 accumulator (one K "
                        "= 16 MMA per tile pair); identical results here, but narrower than the "
                        "float32 accumulation of the headline, whose exactness NVIDIA does not "
                        "document"}

    # The same call on CUDA cores only (fp32 FFMA in every sweep), the path the
    # library takes for data the exact operand encoding cannot hold: its own
    # time and its count sweep against the FP32 FMA roofline.
    if info["path"] != "fp32" and not args.no_ffma and not args.force_path:
        f_ms, f_stages, f_info = timed_variant(["fp32"])
        f_roof = roofline_fields(f_info, n, d, f_stages["count"], peaks, sms, max_mhz)
        line["ffma_path"] = {
            "path": f_info["path"], "dtype": DTYPE_NAMES[f_info["path"]], "ms_per_step": f_ms,
            "value": dist.world * float(n) * n / (f_ms * 1e-3), "unit": UNIT,
            "stages_ms": f_stages,
            "count_pair_evals_per_s": float(n) * n / (f_stages["count"] * 1e-3),
            "roofline": {k: f_roof[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                 "kernel", "peak_source")},
            "note": "every sweep on CUDA cores (fp32 FFMA, float32 throughout), selected with "
                    "dbscan_set_options(paths = 0); same results"}

    if not args.no_e2e:
        ph = torch.from_numpy(P).to(dtype).pin_memory()
        lh = torch.empty(n, dtype=torch.int32).pin_memory()
        ch = torch.empty(n, dtype=torch.uint8).pin_memory()
        binding.dbscan_fit_host(ph, w.eps, w.min_pts, labels=lh, is_core=ch, stream=stream)
        ts = []
        for _ in range(max(1, min(args.steps, 5))):
            flush.zero_()
            torch.cuda.synchronize()
            t = time.perf_counter()
            binding.dbscan_fit_host(ph, w.eps, w.min_pts, labels=lh, is_core=ch, stream=stream)
            ts.append(time.perf_counter() - t)
        e2e_s = dist.max(sum(ts) / len(ts))
        line["e2e"] = {"value": dist.world * float(n) * n / e2e_s, "unit": UNIT,
                       "ms": e2e_s * 1e3, "h2d_bytes_per_step": int(ph.numel() * ph.element_size()),
                       "d2h_bytes_per_step": int(n * 4 + n),
                       "api": "dbscan_fit_host (pinned host buffers, copies inside the timed call)"}
    if dist.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(P, w.eps, w.min_pts)
        line["cpu_baseline_parallel"] = cpu_baseline_parallel(P, w.eps, w.min_pts)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            return run_reference(args, dist)
        return run_gb300(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
