#!/usr/bin/env python3
"""Benchmark of the W4A16 matmul on one GB300.

One step = one pass of the workload's GEMMs (default: the Llama-2-7B-like
decode sweep, M in {1..128} x the four layer shapes, group 128), each reading
its own copy of the packed weights so the step streams more distinct bytes
than L2 holds. Steps are replayed from CUDA Graphs of several consecutive steps
with an event node at every change of M, so per-kernel durations come from CUDA
events on the launching stream. Prints one JSON line.

  python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

The GPU arm runs on one GPU only: with --gpus above 1, or under a launcher that
sets WORLD_SIZE above 1, it exits with an error before any CUDA work (the 2-CTA
cluster kernels load X by TMA multicast within one GPU's memory, and nothing here
is written for several GPUs). --impl reference times the CPU oracle (test
infrastructure) on the host cores on a bounded sample of the same workload; it
touches no GPU, and under a multi-process launcher rank 0 alone runs it.
"""
import argparse
import ctypes
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from weight_only_int4_02_gb300 import inputs  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_WORKLOAD = "llama2_7b_decode_sweep"


# --------------------------------------------------------------------------- accounting
def n_groups(K, G):
    return -(-K // G)


def weight_bytes(K, N, G):
    """Packed INT4 codes (K padded to a whole group) plus FP16 group scales."""
    ng = n_groups(K, G)
    return ng * G * N // 2 + ng * N * 2


def algorithmic_bytes(M, K, N, G):
    return weight_bytes(K, N, G) + 2 * M * K + 2 * M * N


def flops(M, K, N):
    return 2 * M * N * K


def fp16_over_int4_byte_ratio(G):
    """Bytes per weight, FP16 over INT4 with one FP16 scale per G weights."""
    return 2.0 / (0.5 + 2.0 / G)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def kernel_name(plan, N):
    """The kernel instance a plan (path, tile or rows, grid) of w4a16_plan launches for
    N output columns: the decode kernel by rows of X and columns per block (one CTA
    per block of 16 to 128 columns, read back from the grid), the others by rows of X."""
    path, tile, grid = plan
    if path == 3:
        cb = next(c for c in (16, 32, 48, 64, 80, 128) if grid == -(-N // c))
        return "w4a16_decode_kernel<%d,%d>" % (tile, cb)
    return ("w4a16_gemv_kernel<%d>" if path == 1 else "w4a16_tc_kernel<%d>") % tile


def kernel_roofline(name, k, peaks, workload):
    """Per-step time of one kernel instance in the sweep and its roofline fraction:
    algorithmic bytes (or flops, when the tensor pipe bounds it) over its mean launch,
    against the measured peak; the committed ncu traffic per launch when the sources
    match."""
    us = k["ms"] * 1e3
    hbm_s = k["bytes"] / (peaks["hbm_gbs"] * 1e9)
    tc_s = k["flops"] / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if hbm_s >= tc_s else "tensor"
    return {"launches_per_step": k["launches"], "us_per_step": us, "bound": bound,
            "roofline_frac": max(hbm_s, tc_s) / (us * 1e-6),
            "algorithmic_bytes_per_launch": k["bytes"] / k["launches"],
            "traffic": load_traffic(name, workload)}


def roofline_seconds(M, K, N, G, peaks):
    return max(algorithmic_bytes(M, K, N, G) / (peaks["hbm_gbs"] * 1e9),
               flops(M, K, N) / (peaks["bf16_tflops"] * 1e12))


# --------------------------------------------------------------------------- runtime helpers
class Cudart:
    """The few CUDA runtime calls torch does not expose (event nodes in graphs)."""

    def __init__(self):
        import torch
        self.lib = None
        cands = ["libcudart.so.13", "libcudart.so"]
        cands += glob.glob(os.path.join(os.path.dirname(torch.__file__), "..", "nvidia", "*", "lib", "libcudart.so*"))
        cands += ["/usr/local/cuda/lib64/libcudart.so"]
        for c in cands:
            try:
                self.lib = ctypes.CDLL(c)
                break
            except OSError:
                continue
        if self.lib is None:
            raise RuntimeError("libcudart not found")
        self.lib.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.lib.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.lib.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.lib.cudaEventDestroy.argtypes = [ctypes.c_void_p]

    def event(self):
        e = ctypes.c_void_p()
        rc = self.lib.cudaEventCreate(ctypes.byref(e))
        if rc != 0:
            raise RuntimeError("cudaEventCreate failed: %d" % rc)
        return e

    def record_external(self, ev, stream):
        rc = self.lib.cudaEventRecordWithFlags(ev, ctypes.c_void_p(stream.cuda_stream), 1)
        if rc != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed: %d" % rc)

    def elapsed_ms(self, a, b):
        ms = ctypes.c_float()
        rc = self.lib.cudaEventElapsedTime(ctypes.byref(ms), a, b)
        if rc != 0:
            raise RuntimeError("cudaEventElapsedTime failed: %d" % rc)
        return ms.value

    def destroy(self, ev):
        self.lib.cudaEventDestroy(ev)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, wall0, wall1):
        """Summary of the samples taken between wall-clock times wall0 and wall1."""
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside, near = [], []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sample = (float(r[2]), float(r[3]), [n for n, v in zip(names, r[6:10]) if v.strip() == "Active"])
            except ValueError:
                continue
            if wall0 <= ts <= wall1:
                inside.append(sample)
            elif wall0 - 0.2 <= ts <= wall1 + 0.2:
                near.append(sample)
        use = inside if inside else near
        reasons = sorted(set(r for s in use for r in s[2]))
        return {"sm_mhz": statistics.median(s[0] for s in use) if use else None,
                "sm_max_mhz": max(s[1] for s in use) if use else None,
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "within 0.2 s of the timed region"}


def strip_comments(src):
    """C/C++ source without its comments and with runs of whitespace folded, so that
    edits of comments alone leave the code's digest unchanged (string and character
    literals are kept as they are, whitespace included)."""
    parts, code, i, n = [], [], 0, len(src)

    def flush():
        if code:
            parts.append(" ".join("".join(code).split()))
            code.clear()

    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            flush()
            parts.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            code.append(" ")
        else:
            code.append(c)
            i += 1
    flush()
    return " ".join(p for p in parts if p)


def source_digest():
    """Digest of the CUDA sources' code (comments and layout left out): the key under
    which profiles/dram_traffic.txt records counters."""
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "weight_only_int4_02_gb300", "csrc", "*"))):
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest()
    with open(path) as f:
        for line in f:
            kv = dict(p.split("=", 1) for p in line.split() if "=" in p)
            if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("src") == digest:
                return float(kv["bytes_per_launch"])
    return None


# --------------------------------------------------------------------------- CPU baseline (oracle)
def oracle_sample_run(cases, G, scale_mult, outlier_frac, col_stride, threads, data_cache):
    """Time the oracle over every case, on every col_stride-th column. Returns (seconds, flops done)."""
    import oracle
    done = 0
    t = 0.0
    for (M, K, N) in cases:
        key = (K, N)
        if key not in data_cache:
            data_cache[key] = (inputs.codes(K, N, 0), inputs.scales(K, N, G, 0, "halfnormal", scale_mult))
        q, s = data_cache[key]
        x = data_cache.setdefault(("x", M, K), inputs.activations(M, K, 0, outlier_frac))
        cols = np.arange(0, N, col_stride, dtype=np.int32)
        rows = np.arange(M, dtype=np.int32)
        t0 = time.perf_counter()
        oracle.gemm_sample(x, q, s, G, rows, cols, threads=threads)
        t += time.perf_counter() - t0
        done += flops(M, K, len(cols))
    return t, done


def cpu_baseline(wl, budget_s=15.0):
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    cache = {}
    cases = wl["cases"]
    total = sum(flops(*c) for c in cases)
    # calibrate on a coarse sample, then size the timed sample to the budget
    stride = 512
    t, done = oracle_sample_run(cases, wl["group_size"], wl["scale_mult"], wl.get("outlier_frac", 0.0), stride,
                                threads, cache)
    rate = done / max(t, 1e-9)
    want = rate * budget_s
    stride = max(1, int(total / max(want, 1.0)))
    t, done = oracle_sample_run(cases, wl["group_size"], wl["scale_mult"], wl.get("outlier_frac", 0.0), stride,
                                threads, cache)
    if stride == 1:
        # the whole workload fits the budget: repeat it (up to 8 passes) for a steadier rate
        passes = 1
        while passes < 8 and t * (passes + 1) / passes <= budget_s:
            dt, dd = oracle_sample_run(cases, wl["group_size"], wl["scale_mult"], wl.get("outlier_frac", 0.0), 1,
                                       threads, cache)
            t, done, passes = t + dt, done + dd, passes + 1
        sample = "the whole workload (every case, all rows and columns), %d pass%s, %.1f s" % (
            passes, "" if passes == 1 else "es", t)
    else:
        sample = ("every case of the workload, all rows, every %d-th output column (%.3g of the "
                  "workload's flops), %.1f s" % (stride, done / total, t))
    return {"value": done / t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": sample, "seconds": t}


# --------------------------------------------------------------------------- our arm
def single_gpu_refusal(gpus, env):
    """The error text when the GPU arm is asked for more than one GPU, else None."""
    world = int(env.get("WORLD_SIZE", "1") or "1")
    if gpus > 1 or world > 1:
        return ("bench.py runs the W4A16 kernels on one GPU only (asked for --gpus %d, WORLD_SIZE %d); "
                "run it without a multi-process launcher and with --gpus 1" % (gpus, world))
    return None


def run_ours(args):
    import torch
    from weight_only_int4_02_gb300 import w4a16

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wl = inputs.WORKLOADS[args.workload]
    G = wl["group_size"]
    cases = wl["cases"]
    peaks = load_peaks()
    cud = Cudart()

    # ---- data: pack each layer once, then give every case its own copy
    layer_data = {}
    for (M, K, N) in cases:
        if (K, N) not in layer_data:
            q = inputs.codes(K, N, 0)
            s = inputs.scales(K, N, G, 0, "halfnormal", wl["scale_mult"])
            layer_data[(K, N)] = w4a16.pack(torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev), G)
            del q
    per_case = []
    for (M, K, N) in cases:
        packed, sp = layer_data[(K, N)]
        x = torch.from_numpy(inputs.activations(M, K, 0, wl.get("outlier_frac", 0.0))).to(dev)
        per_case.append(dict(M=M, K=K, N=N, packed=packed.clone(), sp=sp.clone(), x=x,
                             y=torch.empty((M, N), dtype=torch.float16, device=dev)))
    del layer_data
    distinct_bytes = sum(c["packed"].numel() * 4 + c["sp"].numel() * 2 for c in per_case)
    torch.cuda.synchronize()

    def launch_all():
        for c in per_case:
            w4a16.gemm(c["x"], c["packed"], c["sp"], c["N"], G, y=c["y"])

    launch_all()   # first call allocates the library's workspace (outside capture)
    torch.cuda.synchronize()
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("kernel wait timed out during warm-up")

    # ---- a pool of graphs of R consecutive steps each, with an event node at every
    # change of M. The event nodes hang off a side branch (forked after the group's last
    # launch, joined once at the end of the graph): every launch follows the previous one
    # directly, so launches overlap through programmatic dependent launch across the
    # changes of M and across the steps inside a graph (an event node between two
    # launches would serialise them). An event node records when every launch before it
    # has completed. Only the first step of a graph starts from an idle GPU; the
    # one-step-graph figure below measures what that start costs when every step pays it.
    bounds = [0] + [ci for ci in range(1, len(per_case)) if per_case[ci]["M"] != per_case[ci - 1]["M"]]
    bounds.append(len(per_case))
    cap = torch.cuda.Stream()
    side = torch.cuda.Stream()
    K = args.steps
    R = max(1, min(K, args.steps_per_graph))

    def capture(nsteps):
        """One graph of nsteps steps; returns (graph, per-step event lists), the first
        event of a step being the last of the step before it (the graph's start for the
        first step)."""
        step_evs = []
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            st = torch.cuda.current_stream()
            # the graph's start is recorded on the side branch too, so that no event node
            # precedes the first GEMM
            start = torch.cuda.Event()
            start.record(st)
            side.wait_event(start)
            prev = cud.event()
            cud.record_external(prev, side)
            for _ in range(nsteps):
                ev = [prev]
                for b in range(len(bounds) - 1):
                    for ci in range(bounds[b], bounds[b + 1]):
                        c = per_case[ci]
                        w4a16.gemm(c["x"], c["packed"], c["sp"], c["N"], G, y=c["y"], stream=st)
                    fork = torch.cuda.Event()
                    fork.record(st)
                    side.wait_event(fork)
                    e = cud.event()
                    cud.record_external(e, side)
                    ev.append(e)
                prev = ev[-1]
                step_evs.append(ev)
            join = torch.cuda.Event()
            join.record(side)
            st.wait_event(join)
        return g, step_evs

    pool = max(1, min(K, 64) // R)
    graphs = [capture(R) for _ in range(pool)]
    tail = {n: capture(n) for n in {K % R, args.warmup % R} if n}

    def run_steps(n):
        for i in range(n // R):
            graphs[i % pool][0].replay()
        if n % R:
            tail[n % R][0].replay()

    torch.cuda.synchronize()
    run_steps(args.warmup)
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record()
    run_steps(K)
    t1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)
    ms_step = t0.elapsed_time(t1) / K
    status = w4a16.check_device_status()
    if status != w4a16.OK:
        raise RuntimeError("a kernel wait timed out in the timed region")

    # ---- per-M durations from the event nodes of every step whose graph ran last in the
    # timed region (every pool graph runs there, and the tail graph of K % R steps)
    timed_evs = [ev for g in graphs for ev in g[1]] + (tail[K % R][1] if K % R else [])
    grp_ms = np.array([[cud.elapsed_ms(ev[b], ev[b + 1]) for b in range(len(bounds) - 1)] for ev in timed_evs])
    grp_mean = grp_ms.mean(axis=0)
    step_flops = sum(flops(c["M"], c["K"], c["N"]) for c in per_case)
    value = step_flops / (ms_step * 1e-3) / 1e12

    # ---- the same steps issued as one graph per step (each step then starts from an
    # idle GPU: no launch of it overlaps the step before), outside the timed region
    one = [capture(1) for _ in range(8)]
    n1 = max(3, min(K, 400))
    for i in range(3):
        one[i % 8][0].replay()
    torch.cuda.synchronize()
    t0.record()
    for i in range(n1):
        one[i % 8][0].replay()
    t1.record()
    torch.cuda.synchronize()
    ms_one = t0.elapsed_time(t1) / n1
    one_step_graphs = {"ms_per_step": ms_one, "value": step_flops / (ms_one * 1e-3) / 1e12, "steps": n1,
                       "note": "every step its own graph, so no launch of a step overlaps the step before"}
    del one

    # ---- diagnostic, outside the timed region: every launch between two event nodes
    diag = torch.cuda.CUDAGraph()
    diag_ev = [cud.event() for _ in range(len(per_case) + 1)]
    with torch.cuda.graph(diag, stream=cap):
        st = torch.cuda.current_stream()
        cud.record_external(diag_ev[0], st)
        for ci, c in enumerate(per_case):
            w4a16.gemm(c["x"], c["packed"], c["sp"], c["N"], G, y=c["y"], stream=st)
            cud.record_external(diag_ev[ci + 1], st)
    mean_ms = np.zeros(len(per_case))
    for r in range(8):
        diag.replay()
        torch.cuda.synchronize()
        if r >= 3:
            mean_ms += np.array([cud.elapsed_ms(diag_ev[ci], diag_ev[ci + 1]) for ci in range(len(per_case))]) / 5

    mean_ms_by_case = {id(c): mean_ms[ci] for ci, c in enumerate(per_case)}

    # ---- per kernel instance and per M
    kernels = {}
    per_m = {}
    for b in range(len(bounds) - 1):
        group = per_case[bounds[b]:bounds[b + 1]]
        M = group[0]["M"]
        # a group of one M may mix kernels (the CUDA-core one for its smallest layer):
        # its measured time is shared among them in proportion to their isolated times
        # (diagnostic run above), every launch counted under its own kernel
        grp_names = [kernel_name(w4a16.plan(c["M"], c["N"], c["K"], G), c["N"]) for c in group]
        iso = [float(mean_ms_by_case[id(c)]) for c in group]
        for c, name, t_iso in zip(group, grp_names, iso):
            k = kernels.setdefault(name, dict(ms=0.0, bytes=0, flops=0, launches=0))
            k["ms"] += grp_mean[b] * (t_iso / sum(iso))
            k["bytes"] += algorithmic_bytes(c["M"], c["K"], c["N"], G)
            k["flops"] += flops(c["M"], c["K"], c["N"])
            k["launches"] += 1
        d = per_m.setdefault(M, dict(ms=0.0, fl=0, wb=0, roof_s=0.0))
        d["ms"] += grp_mean[b]
        d["fl"] += sum(flops(c["M"], c["K"], c["N"]) for c in group)
        d["wb"] += sum(weight_bytes(c["K"], c["N"], G) for c in group)
        d["roof_s"] += sum(roofline_seconds(c["M"], c["K"], c["N"], G, peaks) for c in group)
    dom_name = max(kernels, key=lambda n: kernels[n]["ms"])
    dom = kernels[dom_name]
    hbm_s = dom["bytes"] / (peaks["hbm_gbs"] * 1e9)
    tc_s = dom["flops"] / (peaks["bf16_tflops"] * 1e12)
    if hbm_s >= tc_s:
        achieved = dom["bytes"] / (dom["ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    else:
        achieved = dom["flops"] / (dom["ms"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"]}
    roof["traffic"] = load_traffic(dom_name, args.workload)
    roof["kernel"] = dom_name
    roof["launches_per_step"] = dom["launches"]
    roof["algorithmic_bytes_per_launch"] = dom["bytes"] / dom["launches"]
    roof["avg_launch_us"] = dom["ms"] * 1e3 / dom["launches"]
    roof["peak_source"] = peaks["source"] + (" (HBM copy)" if roof["bound"] == "hbm" else " (bf16 burst)")

    # ---- FP16-weight GEMM of the same shapes (cuBLAS through torch.matmul), same protocol
    fp16 = fp16_baseline(per_case, dev, reps=max(3, min(K, 50)))

    per_m_out = []
    for M in sorted(per_m):
        d = per_m[M]
        entry = {"M": M, "tflops": d["fl"] / (d["ms"] * 1e-3) / 1e12,
                 "weight_gbs": d["wb"] / (d["ms"] * 1e-3) / 1e9,
                 "roofline_frac": d["roof_s"] / (d["ms"] * 1e-3),
                 "us": d["ms"] * 1e3}
        if fp16 is not None:
            entry["fp16_us"] = fp16[M] * 1e3
            entry["speedup_vs_fp16"] = fp16[M] / d["ms"]
        per_m_out.append(entry)

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(per_case, G, dev, K, args.warmup, R)

    out = {
        "metric": "W4A16 GEMM TFLOP/s and weight GB/s vs M; % of HBM/tensor roofline",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # the same step from the event nodes of the last steps (a check on the timed
        # region: well below ms_per_step means a stall somewhere inside it)
        "ms_per_step_events": float(grp_mean.sum()),
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": args.workload, "gemms_per_step": len(per_case),
                   "shapes": "M in %s x (K,N) in %s, group %d" % (
                       sorted(set(c["M"] for c in per_case)), sorted(set((c["K"], c["N"]) for c in per_case)), G),
                   "parallelism": "single-gpu",
                   "l2": "inputs larger than L2: every GEMM reads its own copy of the packed weights "
                         "(%.0f MB distinct per step vs 129 MB L2)" % (distinct_bytes / 1e6),
                   "timing": "CUDA Graphs of %d consecutive steps with an event node at every change of "
                             "M, on a side branch (every launch follows the previous one directly, across "
                             "steps too); per-kernel durations are the mean over the last %d steps of the "
                             "timed region; one_step_graphs times the same steps one graph each; "
                             "per_case_isolated has an event node after every launch (outside the timed "
                             "region), which removes the overlap of consecutive launches" % (R, len(timed_evs))},
        "roofline": roof,
        "gpu_launches": K * len(per_case),
        "clocks": clocks,
        "e2e": e2e,
        "per_M": per_m_out,
        "one_step_graphs": one_step_graphs,
        "per_case_isolated": [{"M": c["M"], "K": c["K"], "N": c["N"], "us": float(mean_ms[ci] * 1e3),
                      "kernel": kernel_name(w4a16.plan(c["M"], c["N"], c["K"], G), c["N"]),
                      "weight_gbs": weight_bytes(c["K"], c["N"], G) / (mean_ms[ci] * 1e-3) / 1e9,
                      "roofline_frac": roofline_seconds(c["M"], c["K"], c["N"], G, peaks) / (mean_ms[ci] * 1e-3)}
                     for ci, c in enumerate(per_case)],
        "kernels": {n: kernel_roofline(n, v, peaks, args.workload) for n, v in kernels.items()},
        "byte_ratio_fp16_over_w4g128": fp16_over_int4_byte_ratio(G),
    }
    if args.workload == DEFAULT_WORKLOAD and not args.no_probes:
        out["fp16_peak"] = fp16_peak_probe()
        out["workloads"] = workloads_probe(G, peaks)
        out["fused_epilogue"] = fused_epilogue_probe(G)
        out["layer_chain"] = layer_chain_probe(G)
        out["zero_points"] = zero_point_probe(G)
        out["w8a16"] = w8_probe(G)
        out["bf16_activations"] = bf16_probe(G)
        out["sparse_2to4"] = sparse_probe(G)
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl)
    return out


def graph_us_per_launch(body, copies, reps=40):
    """Mean microseconds of body(copy) launched `reps` times back to back from one
    CUDA Graph, cycling over `copies` (each its own packed weights)."""
    import torch
    for c in copies:
        body(c)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        for r in range(reps):
            body(copies[r % len(copies)])
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps


def zero_point_probe(G):
    """The per-group zero-point format beside the symmetric one on the same shapes:
    mean time per launch of w4a16_gemm and of w4a16_gemm_zp, launched back to back
    from a CUDA Graph over rotating copies of the packed weights (more bytes than
    L2), on the gate/up decode layer (M = 16, K = 4096, N = 22016) and a prefill
    layer (M = 1024, K = 5120, N = 15360). The zero-points add ceil(K/G) * N / 2
    bytes to the weight stream."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    rows = []
    for M, K, N in ((16, 4096, 22016), (1024, 5120, 15360)):
        q = torch.from_numpy(inputs.codes(K, N, 0)).cuda()
        s = torch.from_numpy(inputs.scales(K, N, G, 0)).cuda()
        z = torch.from_numpy(inputs.zeros(K, N, G, 0)).cuda()
        packed, sp = w4a16.pack(q, s, G)
        zp = w4a16.pack_zeros(z, K, G)
        del q, s, z
        n_copies = max(2, int(400e6 // (packed.numel() * 4)) + 1)
        copies = [(packed.clone(), sp.clone(), zp.clone()) for _ in range(n_copies)]
        del packed, sp, zp
        x = torch.from_numpy(inputs.activations(M, K, 0)).cuda()
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        us_sym = graph_us_per_launch(
            lambda c: w4a16.gemm(x, c[0], c[1], N, G, y=y, stream=torch.cuda.current_stream()), copies)
        us_zp = graph_us_per_launch(
            lambda c: w4a16.gemm_zp(x, c[0], c[1], c[2], N, G, y=y, stream=torch.cuda.current_stream()), copies)
        rows.append({"case": [M, K, N], "us_symmetric": us_sym, "us_zero_points": us_zp,
                     "tflops_zero_points": flops(M, K, N) / (us_zp * 1e-6) / 1e12,
                     "weight_gbs_zero_points": (weight_bytes(K, N, G) + n_groups(K, G) * N / 2) / (us_zp * 1e-6) / 1e9})
        del copies
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    return rows


def w8_probe(G):
    """The W8A16 format (8-bit codes, 128-value stages): mean time per launch of
    w4a16_w8_gemm, launched back to back from a CUDA Graph over rotating copies of
    the packed weights (more bytes than L2), on the gate/up decode layer
    (16 x 4096 x 22016) and the 18432 x 73728 layer at M = 16; weight bytes are
    the 8-bit codes plus the FP16 scales."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    rows = []
    for M, K, N in ((16, 4096, 22016), (16, 18432, 73728)):
        q = torch.randint(0, 256, (K, N), dtype=torch.uint8, device="cuda",
                          generator=torch.Generator(device="cuda").manual_seed(0))
        s = torch.from_numpy(inputs.scales(K, N, G, 0, mult=0.02 / 16)).cuda()
        packed, sp = w4a16.w8_pack(q, s, G)
        del q, s
        n_copies = max(2, int(400e6 // packed.numel()) + 1)
        copies = [(packed, sp)] + [(packed.clone(), sp.clone()) for _ in range(n_copies - 1)]
        del packed, sp
        x = torch.from_numpy(inputs.activations(M, K, 0)).cuda()
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        us = graph_us_per_launch(
            lambda c: w4a16.w8_gemm(x, c[0], c[1], N, G, y=y, stream=torch.cuda.current_stream()), copies,
            reps=40 if K * N < 10 ** 9 else 8)
        wb = n_groups(K, G) * G * N + n_groups(K, G) * N * 2
        rows.append({"case": [M, K, N], "us": us, "weight_gbs": wb / (us * 1e-6) / 1e9,
                     "tflops": flops(M, K, N) / (us * 1e-6) / 1e12})
        del copies
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    return rows


def bf16_probe(G):
    """BF16 activations beside FP16 on the same shapes: mean time per launch of
    w4a16_gemm (FP16) and w4a16_bf16_gemm (BF16 X, scales and Y), launched back to
    back from a CUDA Graph over rotating copies of the packed weights, on the
    gate/up decode layer (16 x 4096 x 22016) and a prefill layer (1024 x 5120 x 15360)."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    rows = []
    for M, K, N in ((16, 4096, 22016), (1024, 5120, 15360)):
        q = torch.from_numpy(inputs.codes(K, N, 0)).cuda()
        s16 = torch.from_numpy(inputs.scales(K, N, G, 0)).cuda()
        packed, sp16 = w4a16.pack(q, s16, G)
        sbf = torch.from_numpy(inputs.scales_bf16(K, N, G, 0).view(np.int16)).cuda().view(torch.bfloat16)
        _, spbf = w4a16.pack(q, sbf, G)
        del q, s16, sbf
        n_copies = max(2, int(400e6 // (packed.numel() * 4)) + 1)
        copies = [(packed.clone(), sp16.clone(), spbf.clone()) for _ in range(n_copies)]
        del packed, sp16, spbf
        x16 = torch.from_numpy(inputs.activations(M, K, 0)).cuda()
        xbf = torch.from_numpy(inputs.activations_bf16(M, K, 0).view(np.int16)).cuda().view(torch.bfloat16)
        y16 = torch.empty((M, N), dtype=torch.float16, device="cuda")
        ybf = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        us16 = graph_us_per_launch(
            lambda c: w4a16.gemm(x16, c[0], c[1], N, G, y=y16, stream=torch.cuda.current_stream()), copies)
        usbf = graph_us_per_launch(
            lambda c: w4a16.bf16_gemm(xbf, c[0], c[2], N, G, y=ybf, stream=torch.cuda.current_stream()), copies)
        rows.append({"case": [M, K, N], "us_fp16": us16, "us_bf16": usbf,
                     "tflops_bf16": flops(M, K, N) / (usbf * 1e-6) / 1e12})
        del copies
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    return rows


def sparse_probe(G):
    """2:4 sparse INT4 beside dense INT4 on the same 2:4 codes: mean time per launch of
    w4a16_gemm and w4a16_sp_gemm, launched back to back from a CUDA Graph over
    rotating copies of the packed weights (more bytes than L2), on the gate/up decode
    layer (16 x 4096 x 22016) and the 18432 x 73728 layer at M = 1, 16 and 128. The
    codes are drawn on the GPU: uniform on 0..15, two of every four k kept (one of
    the six position pairs, uniformly), the rest 8. Sparse weight bytes: stored
    codes (K*N/4) + position words (K*N/8) + FP16 scales."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    rows = []
    pairs = torch.tensor([[1, 1, 0, 0], [1, 0, 1, 0], [1, 0, 0, 1], [0, 1, 1, 0], [0, 1, 0, 1], [0, 0, 1, 1]],
                         dtype=torch.bool, device="cuda")
    for K, N, Ms in ((4096, 22016, (16,)), (18432, 73728, (1, 16, 128))):
        gen = torch.Generator(device="cuda").manual_seed(0)
        q = torch.randint(0, 16, (K, N), dtype=torch.uint8, device="cuda", generator=gen)
        choice = torch.randint(0, 6, (K // 4, N), dtype=torch.int64, device="cuda", generator=gen)
        keep = pairs[choice]                               # [K/4][N][4]
        del choice
        q = torch.where(keep.permute(0, 2, 1).reshape(K, N), q, torch.full_like(q, 8))
        del keep
        s = torch.from_numpy(inputs.scales(K, N, G, 0)).cuda()
        dense = w4a16.pack(q, s, G)
        viol = torch.zeros(1, dtype=torch.int64, device="cuda")
        sparse = w4a16.sp_pack(q, s, G, violations=viol)
        del q
        if int(viol.item()) != 0:
            raise RuntimeError("sparse probe codes are not 2:4")
        n_copies = max(2, int(400e6 // (dense[0].numel() * 4)) + 1)
        dcopies = [dense] + [(dense[0].clone(), dense[1].clone()) for _ in range(n_copies - 1)]
        scopies = [sparse] + [(sparse[0].clone(), sparse[1].clone()) for _ in range(n_copies - 1)]
        del dense, sparse
        for M in Ms:
            x = torch.from_numpy(inputs.activations(M, K, 0)).cuda()
            y = torch.empty((M, N), dtype=torch.float16, device="cuda")
            reps = 40 if K * N < 10 ** 9 else 8
            us_d = graph_us_per_launch(
                lambda c: w4a16.gemm(x, c[0], c[1], N, G, y=y, stream=torch.cuda.current_stream()), dcopies, reps)
            us_s = graph_us_per_launch(
                lambda c: w4a16.sp_gemm(x, c[0], c[1], N, G, y=y, stream=torch.cuda.current_stream()), scopies, reps)
            sb = K * N // 4 + K * N // 8 + n_groups(K, G) * N * 2
            rows.append({"case": [M, K, N], "us_dense": us_d, "us_sparse": us_s, "speedup": us_d / us_s,
                         "sparse_gbs": sb / (us_s * 1e-6) / 1e9,
                         "dense_gbs": weight_bytes(K, N, G) / (us_d * 1e-6) / 1e9,
                         "tflops_sparse": flops(M, K, N) / (us_s * 1e-6) / 1e12})
        del dcopies, scopies
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    return rows


def fused_epilogue_probe(G):
    """The fused epilogue on the gate/up layer (M = 16, K = 4096, N = 22016): mean time
    per launch of the plain GEMM, of w4a16_gemm_fused with bias + SiLU, and of the plain
    GEMM followed by torch's bias add and SiLU (two more kernels that re-read and
    re-write Y), each launched back to back from a CUDA Graph over rotating copies of
    the packed weights (more bytes than L2)."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    M, K, N = 16, 4096, 22016
    q = inputs.codes(K, N, 0)
    s = inputs.scales(K, N, G, 0)
    packed, sp = w4a16.pack(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), G)
    copies = [(packed.clone(), sp.clone()) for _ in range(max(2, int(400e6 // (packed.numel() * 4)) + 1))]
    x = torch.from_numpy(inputs.activations(M, K, 0)).cuda()
    bias = torch.from_numpy(np.random.default_rng(1).standard_normal(N).astype(np.float16)).cuda()
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tmp = torch.empty_like(y)
    def timed(body):
        return graph_us_per_launch(body, copies)

    def plain(c):
        w4a16.gemm(x, c[0], c[1], N, G, y=y, stream=torch.cuda.current_stream())

    def fused(c):
        w4a16.gemm_fused(x, c[0], c[1], N, G, bias=bias, activation="silu", y=y, stream=torch.cuda.current_stream())

    def unfused(c):
        w4a16.gemm(x, c[0], c[1], N, G, y=y, stream=torch.cuda.current_stream())
        torch.add(y, bias, out=tmp)
        torch.nn.functional.silu(tmp, inplace=True)

    us_plain, us_fused, us_unfused = timed(plain), timed(fused), timed(unfused)
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    return {"case": [M, K, N], "epilogue": "bias + SiLU", "us_gemm": us_plain, "us_fused": us_fused,
            "us_gemm_then_torch_bias_silu": us_unfused}


def layer_chain_probe(G):
    """A Llama-2-7B-like decode layer as a chain of dependent GEMMs (each X is the
    previous output, so every launch waits for its predecessor before reading X):
    QKV (4096 -> 12288), O (the first 4096 columns of QKV's output, read in place
    through the row stride -> 4096, plus the layer input as residual), gate/up
    (4096 -> 22016, SiLU fused), down (the first 11008 columns of gate/up's output ->
    4096, plus O's output as residual). Four launches, nothing between them (attention
    and the gate product, which are not W4A16 work, would sit where the column slices
    are read). Mean time per chain from a CUDA Graph of back-to-back chains over
    rotating copies of the packed weights, at M = 1 and 16."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    dims = [(4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096)]
    packs = []
    for i, (K, N) in enumerate(dims):
        q = inputs.codes(K, N, 50 + i)
        s = inputs.scales(K, N, G, 50 + i, "halfnormal", 0.01)
        pk = w4a16.pack(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), G)
        packs.append(pk)
    layer_bytes = sum(p[0].numel() * 4 + p[1].numel() * 2 for p in packs)
    rot = max(2, int(500e6 // layer_bytes) + 1)
    sets = [[(p[0].clone(), p[1].clone()) for p in packs] for _ in range(rot)]
    out = {"layers": "QKV 4096x12288, O 4096x4096 (+residual), gate/up 4096x22016 (SiLU), down 11008x4096 "
                     "(+residual); slices read in place",
           "weight_bytes_per_chain": layer_bytes}
    reps = 20
    for M in (1, 16):
        x = torch.from_numpy(inputs.activations(M, 4096, 7)).cuda()
        h_qkv = torch.empty((M, 12288), dtype=torch.float16, device="cuda")
        h_o = torch.empty((M, 4096), dtype=torch.float16, device="cuda")
        h_gu = torch.empty((M, 22016), dtype=torch.float16, device="cuda")
        h_out = torch.empty((M, 4096), dtype=torch.float16, device="cuda")

        def chain(ws):
            st = torch.cuda.current_stream()
            w4a16.gemm(x, ws[0][0], ws[0][1], 12288, G, y=h_qkv, stream=st)
            w4a16.gemm_strided(h_qkv[:, :4096], ws[1][0], ws[1][1], 4096, G, residual=x, y=h_o, stream=st)
            w4a16.gemm_strided(h_o, ws[2][0], ws[2][1], 22016, G, activation="silu", y=h_gu, stream=st)
            w4a16.gemm_strided(h_gu[:, :11008], ws[3][0], ws[3][1], 4096, G, residual=h_o, y=h_out, stream=st)

        for ws in sets:
            chain(ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream()):
            for r in range(reps):
                chain(sets[r % rot])
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        out["M=%d" % M] = {"us_per_chain": us, "weight_gbs": layer_bytes / (us * 1e3)}
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    return out


def _gpu_codes_scales(K, N, G, seed, mult):
    """Codes uniform on 0..15 and scales FP16(|N(0,1)| * mult), drawn on the GPU (the
    distributions of the workloads; the 18432 x 73728 layer would take long on the host)."""
    import torch
    gen = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randint(0, 16, (K, N), dtype=torch.uint8, device="cuda", generator=gen)
    s = (torch.randn((n_groups(K, G), N), device="cuda", generator=gen).abs() * mult).half()
    return q, s


def _gpu_activations(M, K, seed, outlier_frac):
    import torch
    gen = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((M, K), device="cuda", generator=gen)
    if outlier_frac > 0.0:
        x = torch.where(torch.rand((M, K), device="cuda", generator=gen) < outlier_frac, x * 20.0, x)
    return x.half()


def fp16_us_per_launch(x, weights, y, reps):
    """torch.matmul(x, w) with FP16 weights, back to back over the weight copies: from a
    CUDA Graph when cuBLAS can be captured, else launched eagerly between two events."""
    import torch
    try:
        return graph_us_per_launch(lambda wt: torch.matmul(x, wt, out=y), weights, reps)
    except RuntimeError:
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for r in range(reps):
            torch.matmul(x, weights[r % len(weights)], out=y)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / reps


def fp16_peak_probe(reps=10):
    """FP16 dense tensor throughput of torch.matmul (cuBLAS) on 8192^3, best of reps:
    the FP16 peak measured on this GPU in this run (the BF16 one is in MEASURED_PEAKS.json)."""
    import torch
    n = 8192
    a = torch.randn((n, n), dtype=torch.float16, device="cuda")
    b = torch.randn((n, n), dtype=torch.float16, device="cuda")
    c = torch.empty((n, n), dtype=torch.float16, device="cuda")
    for _ in range(3):
        torch.matmul(a, b, out=c)
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b, out=c)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del a, b, c
    return {"tflops": 2 * n ** 3 / (best * 1e-3) / 1e12, "shape": [n, n, n], "ms": best, "of": "best of %d" % reps}


def workloads_probe(G, peaks):
    """Every other workload's headline shapes, each timed as a CUDA Graph of launches
    back to back over rotating weight copies (more bytes than L2 unless one copy
    already is): the single 16 x 4096 x 4096 GEMM, the 18432 x 73728 layer at
    M = 1, 16, 128, and the four Llama-2-13B-like prefill layers at M = 1024 and 4096
    (X with 1% outliers x20). Each entry: microseconds per launch, TFLOP/s, weight
    GB/s, the roofline fraction (algorithmic bytes over the measured HBM copy rate,
    or flops over the measured BF16 burst peak, whichever binds), the kernel the
    dispatcher picked, and torch.matmul with FP16 weights of the same shape under
    the same protocol."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    groups = [("single_m16_4096x4096", 4096, 4096, 0.02, 0.0, (16,)),
              ("large_layer_18432x73728", 18432, 73728, 0.01, 0.0, (1, 16, 128))]
    groups += [("llama2_13b_prefill", k, n, 0.02, 0.01, (1024, 4096)) for (k, n) in inputs.LLAMA2_13B_LAYERS]
    rows = []
    for wi, (name, K, N, mult, outl, Ms) in enumerate(groups):
        q, s = _gpu_codes_scales(K, N, G, 100 + wi, mult)
        packed, sp = w4a16.pack(q, s, G)
        del q, s
        wb = packed.numel() * 4 + sp.numel() * 2
        n_copies = max(1, int(-(-400e6 // wb)))
        copies = [(packed, sp)] + [(packed.clone(), sp.clone()) for _ in range(n_copies - 1)]
        del packed, sp
        fb = K * N * 2
        f_copies = max(1, int(-(-400e6 // fb)))
        wf = [torch.randn((K, N), dtype=torch.float16, device="cuda") for _ in range(f_copies)]
        for M in Ms:
            x = _gpu_activations(M, K, 200 + M, outl)
            y = torch.empty((M, N), dtype=torch.float16, device="cuda")
            fl = flops(M, K, N)
            reps = max(2, min(40, int(2e12 // max(fl, 1)), int(4e9 // wb)))
            us = graph_us_per_launch(
                lambda c: w4a16.gemm(x, c[0], c[1], N, G, y=y, stream=torch.cuda.current_stream()), copies, reps)
            us16 = fp16_us_per_launch(x, wf, y, reps)
            path, tile, grid = w4a16.plan(M, N, K, G)
            roof_s = roofline_seconds(M, K, N, G, peaks)
            hbm_s = algorithmic_bytes(M, K, N, G) / (peaks["hbm_gbs"] * 1e9)
            rows.append({"workload": name, "M": M, "K": K, "N": N, "us": us, "tflops": fl / (us * 1e-6) / 1e12,
                         "weight_gbs": weight_bytes(K, N, G) / (us * 1e-6) / 1e9,
                         "roofline_frac": roof_s / (us * 1e-6), "bound": "hbm" if hbm_s >= roof_s else "tensor",
                         "kernel": kernel_name((path, tile, grid), N),
                         "fp16_us": us16, "speedup_vs_fp16": us16 / us, "launches_timed": reps})
            del x, y
        del copies, wf
        torch.cuda.empty_cache()
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    return rows


def fp16_baseline(per_case, dev, reps, inner=4):
    """Time per M of torch.matmul with FP16 weights of the same shapes (own copy per
    case): per M, one CUDA Graph of that M's matmuls repeated `inner` times, replayed
    `reps` times between two events, so that neither host launch costs nor a graph's
    start are counted. One M's FP16 weights (405 MB for the four decode layers) are
    more than L2 holds, so every matmul streams its weights from HBM."""
    import torch
    try:
        mats = []
        for c in per_case:
            wgt = torch.randn((c["K"], c["N"]), dtype=torch.float16, device=dev)
            mats.append((c["M"], c["x"], wgt, torch.empty((c["M"], c["N"]), dtype=torch.float16, device=dev)))
        for _, x, wgt, y in mats:
            torch.matmul(x, wgt, out=y)
        torch.cuda.synchronize()
        per_m = {}
        cap = torch.cuda.Stream()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for M in sorted(set(m[0] for m in mats)):
            grp = [m for m in mats if m[0] == M]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for _ in range(inner):
                    for _, x, wgt, y in grp:
                        torch.matmul(x, wgt, out=y)
            g.replay()
            torch.cuda.synchronize()
            t0.record()
            for _ in range(reps):
                g.replay()
            t1.record()
            torch.cuda.synchronize()
            per_m[M] = t0.elapsed_time(t1) / (reps * inner)
            del g
        del mats
        torch.cuda.empty_cache()
        return per_m
    except RuntimeError:
        return None


def run_e2e(per_case, G, dev, K, W, R=1):
    """Same metric through the public API with host buffers: per step, every GEMM's X
    from pinned host memory to the device, the GEMMs, and every Y back to pinned host
    memory, all inside the timed region. Steps go as CUDA Graphs of R consecutive steps
    (the device-only loop's grouping), with two sets of device X and Y buffers used in
    turn, so that a step's uploads run while the step before computes. The copies run on
    two side streams: the GEMMs go by groups of equal M, largest M first; in a graph's
    first step the first group's X is uploaded GEMM by GEMM and every later group's X in
    one copy, in the later steps all of X in one copy; each group's Y is downloaded in
    one copy once its GEMMs are done, while later groups compute. A step's uploads wait for the GEMMs that last read their buffer set (two
    steps back), and its first GEMM for the downloads that last read its Y buffers. What
    stays exposed, once per graph, is the first step's first X and the last step's
    last (smallest) Y."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    order = sorted(range(len(per_case)), key=lambda i: (-per_case[i]["M"], i))
    groups = []
    for i in order:
        if groups and per_case[groups[-1][0]]["M"] == per_case[i]["M"]:
            groups[-1].append(i)
        else:
            groups.append([i])
    x_sizes = {i: per_case[i]["M"] * per_case[i]["K"] for i in order}   # multiples of 8: 16-byte aligned views
    y_sizes = {i: per_case[i]["M"] * per_case[i]["N"] for i in order}
    NB = 2
    x_dev = [torch.empty(sum(x_sizes.values()), dtype=torch.float16, device="cuda") for _ in range(NB)]
    y_dev = [torch.empty(sum(y_sizes.values()), dtype=torch.float16, device="cuda") for _ in range(NB)]
    x_host = torch.empty(sum(x_sizes.values()), dtype=torch.float16).pin_memory()
    y_host = torch.empty(sum(y_sizes.values()), dtype=torch.float16).pin_memory()
    ys_h, x_rng, y_rng = {}, {}, {}
    ox = oy = 0
    for i in order:
        c, nx, ny = per_case[i], x_sizes[i], y_sizes[i]
        x_host[ox:ox + nx].copy_(c["x"].reshape(-1).cpu())
        ys_h[i] = y_host[oy:oy + ny].view(c["M"], c["N"])
        x_rng[i], y_rng[i] = (ox, ox + nx), (oy, oy + ny)
        ox += nx
        oy += ny
    h2d = x_host.numel() * 2
    d2h = y_host.numel() * 2
    # X copies: one per GEMM of the first group, one per later group; Y copies: one per group
    x_chunks = [[i] for i in groups[0]] + groups[1:]
    cap, up, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            main = torch.cuda.current_stream()
            up.wait_stream(main)
            down.wait_stream(main)
            gemms_done, dl_done = [], []
            for s in range(nsteps):
                xb, yb = x_dev[s % NB], y_dev[s % NB]
                ready = {}
                with torch.cuda.stream(up):
                    if s >= NB:
                        up.wait_event(gemms_done[s - NB])
                    # after the first step the uploads run under the previous step's
                    # GEMMs: one copy of all of X, one wait for the step's first GEMM
                    for ch in (x_chunks if s == 0 else [order]):
                        a, b = x_rng[ch[0]][0], x_rng[ch[-1]][1]
                        xb[a:b].copy_(x_host[a:b], non_blocking=True)
                        ev = torch.cuda.Event()
                        ev.record(up)
                        for i in ch:
                            ready[i] = ev
                if s >= NB:
                    main.wait_event(dl_done[s - NB])
                # Every launch follows the previous one directly (programmatic dependent
                # launch) except where it waits for an upload: the first group's GEMMs each
                # wait for their own X, and its last GEMM also for every later group's X,
                # so the later groups start without a wait.
                waited = set()
                for gi, grp in enumerate(groups):
                    for i in grp:
                        need = [ready[i]]
                        if gi == 0 and i == grp[-1]:
                            need += [ready[j] for g2 in groups[1:] for j in g2]
                        for ev in need:
                            if id(ev) not in waited:
                                main.wait_event(ev)
                                waited.add(id(ev))
                        c = per_case[i]
                        xi = xb[x_rng[i][0]:x_rng[i][1]].view(c["M"], c["K"])
                        yi = yb[y_rng[i][0]:y_rng[i][1]].view(c["M"], c["N"])
                        w4a16.gemm(xi, c["packed"], c["sp"], c["N"], G, y=yi, stream=main)
                    done = torch.cuda.Event()
                    done.record(main)
                    down.wait_event(done)
                    with torch.cuda.stream(down):
                        a, b = y_rng[grp[0]][0], y_rng[grp[-1]][1]
                        y_host[a:b].copy_(yb[a:b], non_blocking=True)
                gemms_done.append(done)
                ev = torch.cuda.Event()
                ev.record(down)
                dl_done.append(ev)
            main.wait_stream(up)
            main.wait_stream(down)
        return g

    R = max(1, min(K, R))
    graphs = {R: capture(R)}
    for n in {K % R, W % R}:
        if n:
            graphs[n] = capture(n)

    def run_steps(n):
        for _ in range(n // R):
            graphs[R].replay()
        if n % R:
            graphs[n % R].replay()

    run_steps(max(W, 1))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    run_steps(K)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    step_flops = sum(flops(c["M"], c["K"], c["N"]) for c in per_case)
    ok = all(torch.equal(ys_h[i], per_case[i]["y"].cpu()) for i in order)   # the device-timed run's Y
    return {"value": step_flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "outputs_match_device": ok,
            "steps_per_graph": R,
            "copies_per_step": {"h2d": (len(x_chunks) + R - 1) / R, "d2h": len(groups)}}


# --------------------------------------------------------------------------- reference arm (oracle)
def run_reference(args):
    """The oracle on the host cores. Each step is one case of the workload in turn (all
    rows, every s-th output column, s sized so that the whole run takes about 90 s of
    oracle time whatever --steps is), so that the driver's full step count still ends
    within a few minutes."""
    import oracle
    oracle.build()
    wl = inputs.WORKLOADS[args.workload]
    threads = os.cpu_count() or 1
    cache = {}
    cases = wl["cases"]
    G, mult, outl = wl["group_size"], wl["scale_mult"], wl.get("outlier_frac", 0.0)
    total = sum(flops(*c) for c in cases)
    t, done = oracle_sample_run(cases, G, mult, outl, 1024, threads, cache)   # calibration
    rate = done / max(t, 1e-9)
    budget = min(10.0, 90.0 / max(1, args.steps + args.warmup))             # oracle seconds per step
    strides = {c: max(1, int(flops(*c) / max(rate * budget, 1.0))) for c in cases}

    def step(i):
        c = cases[i % len(cases)]
        return oracle_sample_run([c], G, mult, outl, strides[c], threads, cache)

    for i in range(args.warmup):
        step(i)
    t_all, d_all = 0.0, 0
    for i in range(args.steps):
        t, d = step(args.warmup + i)
        t_all += t
        d_all += d
    v = d_all / t_all / 1e12
    sample = ("CPU oracle (FP64 C, %d threads): per step one of the workload's %d cases in turn, all rows, every "
              "s-th output column (s = %d .. %d; %.3g of the workload's flops over the run)"
              % (threads, len(cases), min(strides.values()), max(strides.values()), d_all / total))
    return {"impl": "reference", "metric": "W4A16 GEMM TFLOP/s and weight GB/s vs M; % of HBM/tensor roofline",
            "value": v, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_all / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_case(args):
    """One GEMM shape, launched back to back from a CUDA Graph over rotating copies
    of the packed weights (more bytes than L2); prints the mean time per launch.
    Used as the small, repeatable command for profiling single kernels."""
    import torch
    from weight_only_int4_02_gb300 import w4a16
    M, K, N = (int(v) for v in args.case.split(","))
    G = 128
    s = torch.from_numpy(inputs.scales(K, N, G, 0)).cuda()
    x = torch.from_numpy(inputs.activations(M, K, 0)).cuda()
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    if args.format == "w8":
        q = inputs.rng(0, inputs.CODE_STREAM).integers(0, 256, size=(K, N), dtype=np.uint8)
        weights = w4a16.w8_pack(torch.from_numpy(q).cuda(), s, G)

        def call(c, stream=None):
            w4a16.w8_gemm(x, c[0], c[1], N, G, y=y, stream=stream)
    elif args.format == "sparse":
        weights = w4a16.sp_pack(torch.from_numpy(inputs.codes_2to4(K, N, 0)).cuda(), s, G)

        def call(c, stream=None):
            w4a16.sp_gemm(x, c[0], c[1], N, G, y=y, stream=stream)
    else:
        weights = w4a16.pack(torch.from_numpy(inputs.codes(K, N, 0)).cuda(), s, G)

        def call(c, stream=None):
            w4a16.gemm(x, c[0], c[1], N, G, y=y, stream=stream)
    wbytes = weights[0].numel() * weights[0].element_size() + weights[1].numel() * 2
    copies = [(weights[0].clone(), weights[1].clone()) for _ in range(max(2, int(400e6 // wbytes) + 1))]
    for c in copies:
        call(c)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        for r in range(args.reps):
            call(copies[r % len(copies)], stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / args.reps
    if w4a16.check_device_status() != w4a16.OK:
        raise RuntimeError("a kernel wait timed out")
    print(json.dumps({"case": [M, K, N], "format": args.format, "us_per_launch": us, "weight_gbs": wbytes / us / 1e3,
                      "tflops": flops(M, K, N) / us / 1e6, "plan": w4a16.plan(M, N, K, G),
                      "launches_before_timed": len(copies) + args.reps}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--steps-per-graph", type=int, default=8,
                    help="consecutive steps captured in one CUDA Graph (decode sweep)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-probes", action="store_true",
                    help="leave out the other workloads and side probes (profiling aid: the launch list of "
                         "the decode sweep alone)")
    ap.add_argument("--case", default=None, help="M,K,N: time one GEMM shape (profiling aid)")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--format", default="int4", choices=["int4", "w8", "sparse"],
                    help="weight format of --case: 4-bit codes, 8-bit codes, or 2:4 sparse 4-bit codes")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3 steps (asked for %d)" % args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.case:
        refusal = single_gpu_refusal(args.gpus, os.environ)
        if refusal:
            print(refusal, file=sys.stderr, flush=True)
            sys.exit(2)
        run_case(args)
        return
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; the other ranks exit without work
        if rank == 0:
            line = run_reference(args)
            line["n_gpus"] = world
            print(json.dumps(line), flush=True)
        return

    refusal = single_gpu_refusal(args.gpus, os.environ)
    if refusal:
        print(refusal, file=sys.stderr, flush=True)
        sys.exit(2)
    out = run_ours(args)
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
